"""Full-size parity: every token of the largest workloads, through the C ABI,
against the CPU oracle (run on token chunks over the host's cores).  Combine:
bit-exact against the oracle's fp32 FMA chain and within 2^-7 of its fp64 sum;
FP8 dispatch: codes and scales bit-exact for every copy of every token."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import workloads as W

from gpu_helpers import DEV, check_combine, draw
from oracle_threads import map_token_chunks

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _combine_every_token(out, y, w, dst, what):
    """Compare out [T,H] (device bf16) with the oracle for all T tokens; y is
    the bf16 expert-output buffer on the device."""
    yb = W.bf16_bits(y)
    wb = w.cpu().numpy()
    db = dst.cpu().numpy()
    ob = W.bf16_bits(out)

    def chunk(t0, t1):
        seq = oracle.combine_fp32_seq(yb, wb[t0:t1], db[t0:t1])
        assert np.array_equal(seq, ob[t0:t1]), "%s: tokens %d..%d differ from the FMA chain" % (what, t0, t1)
        _, ref, absum = oracle.combine_f64(yb, wb[t0:t1], db[t0:t1])
        return check_combine(ob[t0:t1], ref, absum, what)

    worst = max(map_token_chunks(chunk, db.shape[0]))
    assert worst <= 2.0 ** -7


def test_combine_every_token_prefill():
    wl = W.WORKLOADS["prefill"]                      # identity experts: y = dispatched rows
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    recv = ep.dispatch(x, lay.dst_row, wl.rows, status=lay.status)
    out = ep.combine(recv, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    del x
    _combine_every_token(out, recv, w, lay.dst_row, "prefill")


def test_combine_every_token_prefill_fp8_workload():
    wl = W.WORKLOADS["prefill_fp8"]                  # independent bf16 expert outputs (15 GB)
    _, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    y = W.independent_expert_outputs(wl, device=DEV)
    out = ep.combine(y, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    _combine_every_token(out, y, w, lay.dst_row, "prefill_fp8")


def test_combine_every_token_decode_fp8_full_shape():
    wl = W.WORKLOADS["decode_fp8"]                   # T=2048, H=7168, masked, independent outputs
    _, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    y = W.independent_expert_outputs(wl, device=DEV)
    out = ep.combine(y, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    _combine_every_token(out, y, w, lay.dst_row, "decode_fp8")


def test_combine_fp8_every_token_prefill_fp8():
    wl = W.WORKLOADS["prefill_fp8"]
    _, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    y_q, y_s = W.fp8_expert_outputs(wl, device=DEV)
    out = ep.combine_fp8(y_q, y_s, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    qh, sh = y_q.cpu().numpy(), y_s.cpu().numpy()
    wb, db, ob = w.cpu().numpy(), lay.dst_row.cpu().numpy(), W.bf16_bits(out)

    def chunk(t0, t1):
        seq = oracle.combine_fp8_fp32_seq(qh, sh, wb[t0:t1], db[t0:t1])
        assert np.array_equal(seq, ob[t0:t1]), "tokens %d..%d differ from the FMA chain" % (t0, t1)
        _, ref, absum = oracle.combine_fp8_f64(qh, sh, wb[t0:t1], db[t0:t1])
        return check_combine(ob[t0:t1], ref, absum, "prefill_fp8 fp8 combine")

    assert max(map_token_chunks(chunk, wl.T)) <= 2.0 ** -7


@pytest.mark.parametrize("name", ["prefill_fp8", "decode_fp8"])
def test_dispatch_fp8_every_copy_of_every_token(name):
    wl = W.WORKLOADS[name]
    x, idx, _ = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    q, s = ep.dispatch_fp8(x, lay.dst_row, wl.rows, status=lay.status)
    assert ep.status_read(lay.status) == 0
    xb = W.bf16_bits(x)
    ident = np.arange(4096, dtype=np.int32).reshape(4096, 1)

    def chunk(t0, t1):   # the oracle's codes and scales of each token, once
        n = t1 - t0
        return oracle.dispatch_fp8(xb[t0:t1], ident[:n], n)

    refs = map_token_chunks(chunk, wl.T, chunk=4096)
    d = lay.dst_row.long()
    for i, (rq, rs) in enumerate(refs):
        t0 = i * 4096
        blk = d[t0:t0 + rq.shape[0]]
        rq_d = torch.from_numpy(rq).to(DEV)
        rs_d = torch.from_numpy(rs.view(np.int32)).to(DEV)
        for j in range(wl.k):                           # every copy of every token
            rows = blk[:, j]
            assert torch.equal(q[rows], rq_d), "codes differ, tokens from %d, j=%d" % (t0, j)
            assert torch.equal(s[rows].view(torch.int32), rs_d), "scales differ, tokens from %d" % t0
