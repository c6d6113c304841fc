"""Pins for the oracle's two-stage (rank, then expert) path: brute force of
the rank layout, the composition identity expand(dispatch-to-ranks(x)) ==
dispatch(x), and special cases of the two-stage combine (one rank = the
single-stage FMA chain; one expert per rank = per-pair bf16 products summed in
fp32) computed independently with numpy/torch."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_02_gb300 import workloads as W


def brute_rank_layout(idx, E, R):
    T, k = idx.shape
    per = E // R
    reach = [[False] * R for _ in range(T)]
    first = np.zeros((T, k), bool)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if 0 <= e < E and not reach[t][e // per]:
                reach[t][e // per] = True
                first[t, j] = True
    counts = [sum(reach[t][r] for t in range(T)) for r in range(R)]
    offs = [sum(counts[:r]) for r in range(R + 1)]
    rdst = np.full((T, k), -1, np.int64)
    prr = np.full((T, k), -1, np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if not (0 <= e < E):
                continue
            r = e // per
            row = offs[r] + sum(reach[t2][r] for t2 in range(t))
            prr[t, j] = row
            if first[t, j]:
                rdst[t, j] = row
    return counts, offs, rdst, prr


@pytest.mark.parametrize("T,k,E,R", [(1, 1, 1, 1), (9, 3, 6, 3), (40, 8, 16, 4), (64, 8, 64, 64), (33, 4, 8, 1)])
def test_rank_layout_matches_brute_force(T, k, E, R):
    rng = np.random.default_rng(T * 3 + E + R)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    got = oracle.rank_layout(idx, E, R)
    counts, offs, rdst, prr = brute_rank_layout(idx, E, R)
    assert got["rank_counts"].tolist() == counts
    assert got["rank_offsets"].tolist() == offs
    assert np.array_equal(got["rank_dst_row"], rdst)
    assert np.array_equal(got["pair_rank_row"], prr)
    # each rank row's token is the token that owns it
    for t in range(T):
        for j in range(k):
            if rdst[t, j] >= 0:
                assert got["rank_row_token"][rdst[t, j]] == t
    # per-rank counts equal the expert layout's tokens-per-rank
    assert np.array_equal(got["rank_counts"], oracle.layout(idx, E, R)["rank_token_counts"])


@pytest.mark.parametrize("name", ["small", "prefill", "decode_fp8"])
def test_expand_after_rank_dispatch_equals_dispatch(name):
    wl = W.WORKLOADS[name].scaled(T=200, H=256, capacity=200)
    x = W.bf16_bits(W.hidden_states(wl))
    idx = W.route(wl).numpy()
    kind = oracle.LAYOUT_MASKED if wl.kind == "masked" else oracle.LAYOUT_CONTIGUOUS
    lay = oracle.layout(idx, wl.E, wl.R, kind, wl.capacity)
    rl = oracle.rank_layout(idx, wl.E, wl.R)
    nrows = int(rl["rank_offsets"][-1])
    rank_buf = oracle.dispatch_bf16(x, rl["rank_dst_row"], nrows)
    two = oracle.expand(rank_buf, rl["pair_rank_row"], lay["dst_row"], wl.rows)
    one = oracle.dispatch_bf16(x, lay["dst_row"], wl.rows)
    assert np.array_equal(two, one)
    # one copy per (token, rank): fewer rank rows than pairs unless ranks = experts
    assert nrows == (rl["rank_dst_row"] >= 0).sum() <= (lay["dst_row"] >= 0).sum()


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _two_stage(y, w, dst, idx, E, R):
    rl = oracle.rank_layout(idx, E, R)
    part = oracle.combine_partial(y, w, dst, rl["pair_rank_row"], rl["rank_row_token"])
    return oracle.combine_reduce(part, rl["rank_dst_row"], y.shape[1]), rl


def test_two_stage_one_rank_is_the_single_stage_chain():
    wl = W.WORKLOADS["masked"].scaled(T=100, H=128, capacity=100)
    idx = W.route(wl).numpy()
    w = W.topk_weights(wl).numpy()
    lay = oracle.layout(idx, wl.E, 1, oracle.LAYOUT_MASKED, wl.capacity)
    y = W.bf16_bits(W.independent_expert_outputs(wl))
    out, _ = _two_stage(y, w, lay["dst_row"], idx, wl.E, 1)
    assert np.array_equal(out, oracle.combine_fp32_seq(y, w, lay["dst_row"]))


def test_two_stage_one_expert_per_rank_independent():
    # R = E: each partial is bf16(fp32(w*y)); the reduce sums them in fp32 in j order
    wl = W.WORKLOADS["small"].scaled(T=50, H=64)
    idx = W.route(wl).numpy()
    w = W.topk_weights(wl).numpy()
    lay = oracle.layout(idx, wl.E, wl.E)
    rng = np.random.default_rng(4)
    yt = torch.from_numpy(rng.standard_normal((wl.rows, wl.H)).astype(np.float32)).to(torch.bfloat16)
    y = W.bf16_bits(yt)
    out, _ = _two_stage(y, w, lay["dst_row"], idx, wl.E, wl.E)
    yf = yt.float()
    expect = torch.zeros(wl.T, wl.H, dtype=torch.float32)
    for j in range(wl.k):
        rows = torch.from_numpy(lay["dst_row"][:, j].astype(np.int64))
        prod = (torch.from_numpy(w[:, j]).view(-1, 1) * yf[rows]).to(torch.bfloat16).float()
        expect = expect + prod
    assert np.array_equal(out, W.bf16_bits(expect.to(torch.bfloat16)))


def test_two_stage_within_tolerance_of_fp64():
    wl = W.WORKLOADS["prefill"].scaled(T=300, H=256)
    idx = W.route(wl).numpy()
    w = W.topk_weights(wl).numpy()
    lay = oracle.layout(idx, wl.E, wl.R)
    y = W.bf16_bits(W.independent_expert_outputs(wl))
    out, _ = _two_stage(y, w, lay["dst_row"], idx, wl.E, wl.R)
    _, ref, absum = oracle.combine_f64(y, w, lay["dst_row"])
    err = np.abs(_f(out) - ref)
    # per-rank bf16 rounding (<= 2^-9 of each partial, sum <= 2^-9 S), fp32
    # sums, final bf16 rounding (<= 2^-9 |ref|)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -8 * absum + 1e-30)
