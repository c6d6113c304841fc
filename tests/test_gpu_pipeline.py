"""Host-buffer executor (ep_roundtrip_host): one step from pinned host inputs
to a pinned host output gives exactly what the device-side calls give, and
matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import binding
from combine_ep_layout_02_gb300 import workloads as W

from gpu_helpers import DEV, check_combine

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("name,T,H,chunk", [("prefill", 3000, 7168, 512), ("masked", 2048, 2048, 2048),
                                            ("small", 128, 2048, 7), ("prefill", 5, 64, 1),
                                            ("masked", 2048, 1024, 100)])
def test_roundtrip_matches_device_calls(name, T, H, chunk):
    wl = W.WORKLOADS[name].scaled(T=T, H=H, capacity=min(W.WORKLOADS[name].capacity, T) or None)
    x, idx, w = W.hidden_states(wl), W.route(wl), W.topk_weights(wl)
    pipe = binding.Pipeline(wl.T, wl.H, wl.k, wl.E, wl.R, wl.kind, wl.capacity, chunk_tokens=chunk,
                            device=DEV)
    xh, ih, wh = x.pin_memory(), idx.pin_memory(), w.pin_memory()
    outs = []
    for _ in range(2):   # reused buffers, two steps in a row
        oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
        pipe.run(xh, ih, wh, oh)
        torch.cuda.synchronize()
        outs.append(oh.clone())
    assert ep.status_read(pipe.layout.status) == 0
    xd, idd, wd = x.to(DEV), idx.to(DEV), w.to(DEV)
    lay = ep.layout(idd, wl.E, wl.R, wl.kind, wl.capacity)
    recv = ep.dispatch(xd, lay.dst_row, wl.rows)
    ref = ep.combine(recv, wd, lay.dst_row).cpu()
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    # and the oracle (fp64 tolerance) on the identity-expert combine
    r = oracle.layout(idx.numpy(), wl.E, wl.R, oracle.LAYOUT_MASKED if wl.kind == "masked" else 0, wl.capacity)
    rrecv = oracle.dispatch_bf16(W.bf16_bits(x), r["dst_row"], wl.rows)
    _, refd, absum = oracle.combine_f64(rrecv, w.numpy(), r["dst_row"])
    check_combine(W.bf16_bits(outs[0]), refd, absum, name)
    pipe.close()


def test_roundtrip_with_expert_outputs_on_device():
    wl = W.WORKLOADS["decode_fp8"].scaled(T=700, H=1024, capacity=700)
    x, idx, w = W.hidden_states(wl), W.route(wl), W.topk_weights(wl)
    y = W.independent_expert_outputs(wl, device=DEV)
    pipe = binding.Pipeline(wl.T, wl.H, wl.k, wl.E, wl.R, wl.kind, wl.capacity, chunk_tokens=256,
                            device=DEV, y=y)
    oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
    pipe.run(x.pin_memory(), idx.pin_memory(), w.pin_memory(), oh)
    torch.cuda.synchronize()
    lay = ep.layout(idx.to(DEV), wl.E, wl.R, wl.kind, wl.capacity)
    ref = ep.combine(y, w.to(DEV), lay.dst_row).cpu()
    assert torch.equal(oh.view(torch.int16), ref.view(torch.int16))
    # the dispatch buffer was written too
    recv_ref = ep.dispatch(x.to(DEV), lay.dst_row, wl.rows)
    used = lay.dst_row.view(-1).long()
    assert torch.equal(pipe.recv[used].view(torch.int16), recv_ref[used].view(torch.int16))
    pipe.close()


def test_roundtrip_fp8_dispatch():
    wl = W.WORKLOADS["prefill_fp8"].scaled(T=1500, H=1024)
    x, idx, w = W.hidden_states(wl), W.route(wl), W.topk_weights(wl)
    y = W.independent_expert_outputs(wl, device=DEV)
    pipe = binding.Pipeline(wl.T, wl.H, wl.k, wl.E, wl.R, wl.kind, wl.capacity, chunk_tokens=400,
                            device=DEV, y=y, payload="fp8")
    oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
    pipe.run(x.pin_memory(), idx.pin_memory(), w.pin_memory(), oh)
    torch.cuda.synchronize()
    assert ep.status_read(pipe.layout.status) == 0
    lay = ep.layout(idx.to(DEV), wl.E, wl.R, wl.kind, wl.capacity)
    q, s = ep.dispatch_fp8(x.to(DEV), lay.dst_row, wl.rows)
    used = lay.dst_row.view(-1).long()
    assert torch.equal(pipe.recv_q[used], q[used]) and torch.equal(pipe.recv_scale[used], s[used])
    ref = ep.combine(y, w.to(DEV), lay.dst_row).cpu()
    assert torch.equal(oh.view(torch.int16), ref.view(torch.int16))
    pipe.close()
