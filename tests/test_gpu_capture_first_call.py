"""Graph capture as the very first use: a fresh process whose first call of
each kernel (one-launch cluster layout, chunked layout, fused layout +
dispatch, FP8 dispatch, combine) happens inside torch.cuda.graph capture.
The launchers configure kernel attributes and query cluster occupancy on
first use; none of that may break or be refused during capture."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, torch
sys.path.insert(0, ROOT_DIR)
import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import workloads as W
dev = torch.device("cuda:0")

def graph(fn):
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        res = fn()
    g.replay()
    torch.cuda.synchronize()
    return res

for T in (300, 5000):  # a 16-block cluster, then the chunked kernels
    wl = W.WORKLOADS["decode_fp8"].scaled(T=T, capacity=T)
    idx = W.route(wl, device=dev)
    lay = graph(lambda: ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity))
    ref = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    assert torch.equal(lay.dst_row, ref.dst_row) and ep.status_read(lay.status) == 0
wl = W.WORKLOADS["decode_fp8"].scaled(T=100, capacity=100)
idx, x = W.route(wl, device=dev), W.hidden_states(wl, device=dev)
# zero-filled buffers: masked padding rows are never written
q, s, q2, s2 = (torch.zeros(wl.rows, wl.H, dtype=torch.uint8, device=dev),
                torch.zeros(wl.rows, wl.H // 128, device=dev),
                torch.zeros(wl.rows, wl.H, dtype=torch.uint8, device=dev),
                torch.zeros(wl.rows, wl.H // 128, device=dev))
lay = graph(lambda: ep.layout_dispatch(x, idx, wl.E, wl.R, wl.kind, wl.capacity, fp8=True,
                                       recv_q=q, recv_scale=s)[0])
assert ep.status_read(lay.status) == 0
graph(lambda: ep.dispatch_fp8(x, lay.dst_row, wl.rows, recv_q=q2, recv_scale=s2))
assert torch.equal(q, q2) and torch.equal(s, s2)
w = W.topk_weights(wl, device=dev)
y = torch.randn(wl.rows, wl.H, device=dev).to(torch.bfloat16)
out = graph(lambda: ep.combine(y, w, lay.dst_row))
assert torch.equal(out, ep.combine(y, w, lay.dst_row))
print("CAPTURE-FIRST OK")
'''


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def test_first_calls_inside_graph_capture():
    code = SCRIPT.replace("ROOT_DIR", repr(ROOT))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "CAPTURE-FIRST OK" in r.stdout
