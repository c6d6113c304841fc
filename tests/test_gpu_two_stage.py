"""Two-stage (rank, then expert) path on the GPU against the oracle: rank
layout bit-exact, dispatch-to-ranks + expansion equal to the single-stage
dispatch bit for bit, partial + final reduction bit-exact against the
oracle's two-stage definition and within tolerance of the fp64 sum."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import workloads as W

from gpu_helpers import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _bits(t):
    return W.bf16_bits(t)


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _check_rank_layout(idx_host, E, R, rl):
    ref = oracle.rank_layout(idx_host, E, R)
    assert np.array_equal(rl.rank_counts.cpu().numpy(), ref["rank_counts"])
    assert np.array_equal(rl.rank_offsets.cpu().numpy(), ref["rank_offsets"])
    assert np.array_equal(rl.rank_dst_row.cpu().numpy(), ref["rank_dst_row"])
    assert np.array_equal(rl.pair_rank_row.cpu().numpy(), ref["pair_rank_row"])
    n = int(ref["rank_offsets"][-1])
    assert np.array_equal(rl.rank_row_token.cpu().numpy()[:n], ref["rank_row_token"])
    assert ep.status_read(rl.status) == ref["flags"]
    return ref


@pytest.mark.parametrize("T,k,E,R", [(1, 1, 1, 1), (33, 8, 128, 4), (700, 8, 256, 16), (3000, 8, 64, 64),
                                     (2500, 4, 96, 96), (513, 32, 1024, 128), (4100, 6, 12, 3)])
def test_rank_layout_random(T, k, E, R):
    rng = np.random.default_rng(T + 5 * R)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    idx[0, 0] = E + 3 if T > 0 and E < 1000 else idx[0, 0]   # one bad id
    rl = ep.rank_layout(torch.from_numpy(idx).to(DEV), E, R)
    _check_rank_layout(idx, E, R, rl)


@pytest.mark.parametrize("name,T,H", [("small", 128, 2048), ("prefill", 3000, 1024),
                                      ("decode_fp8", 700, 512), ("masked", 2048, 256),
                                      ("prefill", 20, 1336), ("small", 3, 7168),
                                      ("prefill_grouped", 3000, 1024)])
def test_two_stage_path_matches_single_stage(name, T, H):
    wl = W.WORKLOADS[name].scaled(T=T, H=H, capacity=min(W.WORKLOADS[name].capacity, T) or None)
    x = W.hidden_states(wl, device=DEV)
    idx = W.route(wl, device=DEV)
    w = W.topk_weights(wl, device=DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    rl = ep.rank_layout(idx, wl.E, wl.R)
    ref = _check_rank_layout(idx.cpu().numpy(), wl.E, wl.R, rl)
    cap = ep.rank_rows_bound(wl.T, wl.k, wl.R)
    # dispatch to ranks, then expand into the experts
    rank_buf = ep.dispatch(x, rl.rank_dst_row, cap)
    recv2 = torch.zeros(wl.rows, wl.H, dtype=torch.bfloat16, device=DEV)
    ep.expand(rank_buf, rl, lay.dst_row, wl.rows, recv=recv2, status=lay.status)
    recv1 = ep.dispatch(x, lay.dst_row, wl.rows)
    used = lay.dst_row.view(-1).long()
    assert torch.equal(recv2[used].view(torch.int16), recv1[used].view(torch.int16))
    # partial + final reduction
    y = W.independent_expert_outputs(wl, device=DEV)
    part = ep.combine_partial(y, w, lay.dst_row, rl, cap, status=lay.status)
    out = ep.combine_reduce(part, rl, wl.T, status=lay.status)
    assert ep.status_read(lay.status) == 0
    dst = lay.dst_row.cpu().numpy()
    n = int(ref["rank_offsets"][-1])
    rpart = oracle.combine_partial(_bits(y), w.cpu().numpy(), dst, ref["pair_rank_row"], ref["rank_row_token"])
    assert np.array_equal(_bits(part[:n]), rpart)
    rout = oracle.combine_reduce(rpart, ref["rank_dst_row"], wl.H)
    assert np.array_equal(_bits(out), rout)
    _, r64, absum = oracle.combine_f64(_bits(y), w.cpu().numpy(), dst)
    assert np.all(np.abs(_f(_bits(out)) - r64) <= 2.0 ** -8 * np.abs(r64) + 2.0 ** -8 * absum + 1e-30)
    if wl.route == "grouped":             # at most groups_per_token rank copies per token
        assert n <= wl.T * wl.groups_per_token


def test_two_stage_full_size_prefill():
    wl = W.WORKLOADS["prefill"]
    x = W.hidden_states(wl, device=DEV)
    idx = W.route(wl, device=DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    rl = ep.rank_layout(idx, wl.E, wl.R)
    _check_rank_layout(idx.cpu().numpy(), wl.E, wl.R, rl)
    cap = ep.rank_rows_bound(wl.T, wl.k, wl.R)
    rank_buf = ep.dispatch(x, rl.rank_dst_row, cap)
    recv = ep.expand(rank_buf, rl, lay.dst_row, wl.rows, status=lay.status)
    assert ep.status_read(lay.status) == 0
    d = lay.dst_row.view(-1).long()
    tok = torch.arange(wl.T * wl.k, device=DEV) // wl.k
    xi, ri = x.view(torch.int16), recv.view(torch.int16)
    for c0 in range(0, d.numel(), 1 << 16):
        assert torch.equal(ri[d[c0:c0 + (1 << 16)]], xi[tok[c0:c0 + (1 << 16)]])
    # one copy per (token, rank) reached
    assert int(rl.rank_offsets[-1]) == int(lay.rank_token_counts.sum())


@pytest.mark.parametrize("name,T,H", [("decode_fp8", 2048, 7168), ("prefill_fp8", 1500, 384),
                                      ("decode_fp8", 40, 7168), ("prefill_fp8", 9, 1664)])
def test_two_stage_fp8_matches_direct_and_oracle(name, T, H):
    wl = W.WORKLOADS[name].scaled(T=T, H=H, capacity=min(W.WORKLOADS[name].capacity, T) or None)
    x = W.hidden_states(wl, device=DEV)
    idx = W.route(wl, device=DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    rl = ep.rank_layout(idx, wl.E, wl.R)
    cap = ep.rank_rows_bound(wl.T, wl.k, wl.R)
    rq, rs = ep.dispatch_fp8(x, rl.rank_dst_row, cap)          # one quantised copy per (token, rank)
    q2, s2 = ep.expand_fp8(rq, rs, rl, lay.dst_row, wl.rows, status=lay.status)
    q1, s1 = ep.dispatch_fp8(x, lay.dst_row, wl.rows, status=lay.status)
    assert ep.status_read(lay.status) == 0
    used = lay.dst_row.view(-1).long()
    assert torch.equal(q2[used], q1[used])
    assert torch.equal(s2[used].view(torch.int32), s1[used].view(torch.int32))
    dst = lay.dst_row.cpu().numpy()
    keep = dst.reshape(-1) >= 0
    compact = np.full(dst.size, -1, np.int32)
    compact[keep] = np.arange(int(keep.sum()), dtype=np.int32)
    oq, os_ = oracle.dispatch_fp8(_bits(x), compact.reshape(dst.shape), int(keep.sum()))
    rows_used = torch.from_numpy(dst.reshape(-1)[keep].astype(np.int64)).to(DEV)
    assert np.array_equal(q2[rows_used].cpu().numpy(), oq)
    assert np.array_equal(s2[rows_used].cpu().numpy().view(np.uint32), os_.view(np.uint32))
