"""No kernel writes outside the buffers it is given: every output is a window
into a larger sentinel-filled allocation, and the guard regions around it
must be unchanged after the call (including with bad rows and bad ids in the
inputs)."""
import numpy as np
import pytest
import torch

import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import workloads as W

from gpu_helpers import DEV

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of guard on each side


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


class Guarded:
    """A tensor of `shape`/`dtype` placed inside a sentinel-filled byte buffer."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), 0xA5, dtype=torch.uint8, device=DEV)
        self.n = n
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)

    def intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        return bool(torch.all(head == 0xA5)) and bool(torch.all(tail == 0xA5))


@pytest.mark.parametrize("T,kind", [(300, "contiguous"), (3000, "masked"), (200, "masked")])
def test_no_writes_outside_outputs(T, kind):
    wl = W.WORKLOADS["masked" if kind == "masked" else "prefill"].scaled(T=T, H=1024, capacity=max(8, T // 20))
    idx = W.route(wl, device=DEV).clone()
    idx[0, 0] = wl.E + 5          # a bad id
    idx[1, 1] = -1                # an unrouted pair
    x = W.hidden_states(wl, device=DEV)
    w = W.topk_weights(wl, device=DEV)
    E, R, k, H = wl.E, wl.R, wl.k, wl.H
    guards = []
    gl = [Guarded((E,), torch.int32), Guarded((E + 1,), torch.int32), Guarded((T, k), torch.int32),
          Guarded((R,), torch.int32), Guarded((1,), torch.int32)]
    lay = ep.LayoutOut(*(g.t for g in gl))
    ep.layout(idx, E, R, wl.kind, wl.capacity, out=lay)
    flags = ep.status_read(lay.status)
    assert flags & ep.EP_FLAG_BAD_EXPERT
    guards += gl
    rows = wl.rows
    d = lay.dst_row.clone()
    d[2, 2] = rows + 100          # an out-of-range row: must be skipped, not written
    grecv = Guarded((rows, H), torch.bfloat16)
    ep.dispatch(x, d, rows, recv=grecv.t, status=lay.status)
    gq, gs = Guarded((rows, H), torch.uint8), Guarded((rows, H // 128), torch.float32)
    ep.dispatch_fp8(x, d, rows, recv_q=gq.t, recv_scale=gs.t, status=lay.status)
    y = torch.randn(rows, H, device=DEV).to(torch.bfloat16)
    gout = Guarded((T, H), torch.bfloat16)
    ep.combine(y, w, d, out=gout.t, status=lay.status)
    y_q, y_s = W.fp8_expert_outputs(wl, device=DEV)
    gout8 = Guarded((T, H), torch.bfloat16)
    ep.combine_fp8(y_q, y_s, w, d, out=gout8.t, status=lay.status)
    assert ep.status_read(lay.status) & ep.EP_FLAG_BAD_ROW
    guards += [grecv, gq, gs, gout, gout8]
    # two-stage path
    cap = ep.rank_rows_bound(T, k, R)
    gr = [Guarded((R,), torch.int32), Guarded((R + 1,), torch.int32), Guarded((T, k), torch.int32),
          Guarded((T, k), torch.int32), Guarded((cap,), torch.int32), Guarded((1,), torch.int32)]
    rl = ep.RankLayoutOut(*(g.t for g in gr))
    ep.rank_layout(idx, E, R, out=rl)
    grb = Guarded((cap, H), torch.bfloat16)
    ep.dispatch(x, rl.rank_dst_row, cap, recv=grb.t)
    grecv2 = Guarded((rows, H), torch.bfloat16)
    ep.expand(grb.t, rl, d, rows, recv=grecv2.t)
    gpart = Guarded((cap, H), torch.bfloat16)
    ep.combine_partial(y, w, d, rl, cap, partial=gpart.t)
    gout2 = Guarded((T, H), torch.bfloat16)
    ep.combine_reduce(gpart.t, rl, T, out=gout2.t)
    torch.cuda.synchronize()
    guards += gr + [grb, grecv2, gpart, gout2]
    for i, g in enumerate(guards):
        assert g.intact(), "guard %d damaged" % i
