"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs.  Layout, BF16 dispatch and FP8 codes + scales must be
bit-exact; combine must be within 2^-7 of the oracle's fp64 sum (and is also
checked bit-exact against the oracle's fp32 fused-multiply-add sequence)."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import workloads as W

from gpu_helpers import DEV, bf16_to_f64, check_combine, draw, oracle_kind, rows_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _bits(t):
    return W.bf16_bits(t)


def _compare_layout(idx_host, E, R, kind, cap, lay, expect_flags=None):
    ref = oracle.layout(idx_host, E, R, oracle.LAYOUT_MASKED if kind == "masked" else 0, cap)
    assert np.array_equal(lay.expert_counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(lay.expert_offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(lay.dst_row.cpu().numpy(), ref["dst_row"])
    if lay.rank_token_counts is not None:
        assert np.array_equal(lay.rank_token_counts.cpu().numpy(), ref["rank_token_counts"])
    flags = ep.status_read(lay.status)
    assert flags == ref["flags"]
    if expect_flags is not None:
        assert flags == expect_flags
    return ref


# --------------------------------------------------------------------------- layout

LAYOUT_CASES = [
    (1, 1, 1, 1), (1, 8, 256, 16), (31, 2, 3, 3), (33, 8, 128, 4), (511, 8, 256, 16),
    (512, 8, 256, 16), (513, 8, 256, 16), (1500, 8, 128, 4), (1500, 32, 1024, 8),
    (1025, 1, 1024, 1024), (2000, 3, 7, 7), (4096, 8, 256, 32), (777, 16, 64, 2),
    # one-launch boundaries: a single block up to 64 tokens, an 8-block cluster
    # up to 256, a 16-block one up to 2048 (smaller blocks or the chunked path
    # when shared memory runs out); pieces of 32 // k tokens (k = 5, 6, 32),
    # E / R not a power of two, E > 32 * ranges
    (384, 32, 1024, 1024), (385, 8, 256, 16), (2048, 8, 256, 16), (2048, 32, 1024, 1024),
    (100, 5, 120, 5), (1999, 7, 600, 24), (2049, 8, 128, 4), (128, 8, 128, 4), (300, 1, 33, 11),
    (64, 8, 256, 16), (65, 8, 128, 4), (256, 8, 256, 16), (257, 8, 256, 16), (257, 6, 96, 3),
    (2048, 8, 128, 4), (1000, 6, 256, 16), (2048, 1, 1024, 1024), (1536, 4, 1024, 32),
]


@pytest.mark.parametrize("T,k,E,R", LAYOUT_CASES)
def test_layout_random_ids_with_duplicates(T, k, E, R):
    rng = np.random.default_rng(T * 7 + k * 131 + E)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    idx_d = torch.from_numpy(idx).to(DEV)
    lay = ep.layout(idx_d, E, R, "contiguous")
    _compare_layout(idx, E, R, "contiguous", 0, lay)
    cap = max(1, (T * k) // E // 2)    # forces overflow for most shapes
    lay = ep.layout(idx_d, E, R, "masked", cap)
    _compare_layout(idx, E, R, "masked", cap, lay)
    lay = ep.layout(idx_d, E, R, "masked", T * k)
    _compare_layout(idx, E, R, "masked", T * k, lay, expect_flags=0)


def test_layout_bad_ids_flagged():
    idx = np.array([[0, 9, -1, 3], [-7, 1, 2, 2], [3, 3, 3, 300]], np.int32)
    lay = ep.layout(torch.from_numpy(idx).to(DEV), 4, 2, "contiguous")
    ref = _compare_layout(idx, 4, 2, "contiguous", 0, lay, expect_flags=ep.EP_FLAG_BAD_EXPERT)
    assert ref["dst_row"][0, 1] == -1 and ref["dst_row"][1, 0] == -1


def test_layout_without_rank_counts_and_empty():
    idx = np.random.default_rng(1).integers(0, 64, size=(700, 4)).astype(np.int32)
    lay = ep.layout(torch.from_numpy(idx).to(DEV), 64, 4, "contiguous", with_rank_counts=False)
    assert lay.rank_token_counts is None
    _compare_layout(idx, 64, 4, "contiguous", 0, lay)
    empty = torch.empty(0, 8, dtype=torch.int32, device=DEV)
    lay = ep.layout(empty, 256, 16, "contiguous")
    assert int(lay.expert_counts.abs().sum()) == 0 and int(lay.expert_offsets.abs().sum()) == 0
    assert int(lay.rank_token_counts.abs().sum()) == 0
    assert ep.status_read(lay.status) == 0


def test_layout_balanced_route():
    idx = W.balanced_route(4096, 8, 256, seed=5)
    lay = ep.layout(idx.to(DEV), 256, 16, "contiguous")
    _compare_layout(idx.numpy(), 256, 16, "contiguous", 0, lay, expect_flags=0)
    assert torch.all(lay.expert_counts == 128)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_layout_full_size_workloads(name):
    wl = W.WORKLOADS[name]
    idx = W.route(wl, device=DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    _compare_layout(idx.cpu().numpy(), wl.E, wl.R, wl.kind, wl.capacity, lay, expect_flags=0)


# --------------------------------------------------------------------------- dispatch BF16

SENTINEL = -21555  # 0xABCD as int16


@pytest.mark.parametrize("name,T,H", [("small", 128, 2048), ("small", 1500, 2048),
                                      ("masked", 2048, 2048), ("prefill", 1500, 7168),
                                      ("prefill", 77, 7168 + 8), ("masked", 300, 8)])
def test_dispatch_bf16_bit_exact(name, T, H):
    wl = W.WORKLOADS[name].scaled(T=T, H=H)
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    recv = torch.full((wl.rows, wl.H), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    ep.dispatch(x, lay.dst_row, wl.rows, recv=recv, status=lay.status)
    dst = lay.dst_row.cpu().numpy()
    ref = oracle.dispatch_bf16(_bits(x), dst, wl.rows,
                               recv=np.full((wl.rows, wl.H), np.uint16(0xABCD), np.uint16))
    got = _bits(recv)
    assert np.array_equal(got, ref)          # used rows equal, untouched rows keep the sentinel
    assert ep.status_read(lay.status) == 0


@pytest.mark.parametrize("T,k,H,E", [(1, 8, 2048, 64), (3, 13, 1336, 32), (37, 8, 7168, 256),
                                     (5, 1, 1664, 8), (200, 8, 384, 16), (64, 32, 4096, 1024)])
def test_few_tokens_column_slices(T, k, H, E):
    # with few tokens the row kernels (BF16 and FP8 dispatch, combine) split
    # each row into column slices, one warp each; these shapes give single,
    # ragged and unsplit rows, k above the 8 rows held in registers, and
    # FP8 slices of 512-channel groups with a short last slice
    g = torch.Generator().manual_seed(T * 1000 + H)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    x = (torch.randn(T, H, generator=g) * 3).to(torch.bfloat16)
    w = torch.rand(T, k, generator=g) - 0.25
    y = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    lay = ep.layout(idx.to(DEV), E, 1)
    rows = T * k
    dst = lay.dst_row.cpu().numpy()
    recv = ep.dispatch(x.to(DEV), lay.dst_row, rows, status=lay.status)
    assert np.array_equal(_bits(recv), oracle.dispatch_bf16(_bits(x), dst, rows))
    out = ep.combine(y.to(DEV), w.to(DEV), lay.dst_row, status=lay.status)
    assert np.array_equal(_bits(out), oracle.combine_fp32_seq(_bits(y), w.numpy(), dst))
    if H % 128 == 0:
        q, s = ep.dispatch_fp8(x.to(DEV), lay.dst_row, rows, status=lay.status)
        rq, rs = oracle.dispatch_fp8(_bits(x), dst, rows)
        assert np.array_equal(q.cpu().numpy(), rq)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert ep.status_read(lay.status) == 0


def test_dispatch_bad_rows_are_skipped_and_flagged():
    x = torch.randn(4, 64, device=DEV).to(torch.bfloat16)
    dst = torch.tensor([[0, 9], [1, -1], [-3, 2], [3, 4]], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    recv = torch.zeros(5, 64, dtype=torch.bfloat16, device=DEV)
    ep.dispatch(x, dst, 5, recv=recv, status=status)     # row 9 and row -3 are out of range
    assert ep.status_read(status) == ep.EP_FLAG_BAD_ROW
    assert torch.equal(recv[0], x[0]) and torch.equal(recv[1], x[1]) and torch.equal(recv[2], x[2])
    assert torch.equal(recv[3], x[3]) and torch.equal(recv[4], x[3])


def test_dispatch_full_size_prefill():
    wl = W.WORKLOADS["prefill"]
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    recv = ep.dispatch(x, lay.dst_row, wl.rows, status=lay.status)
    assert ep.status_read(lay.status) == 0
    # property at full size: every routed pair's row is its token's row, bitwise
    d = lay.dst_row.view(-1).long()
    tok = torch.arange(wl.T * wl.k, device=DEV) // wl.k
    xi, ri = x.view(torch.int16), recv.view(torch.int16)
    for c0 in range(0, d.numel(), 1 << 16):
        assert torch.equal(ri[d[c0:c0 + (1 << 16)]], xi[tok[c0:c0 + (1 << 16)]])
    # contiguous layout: every row below expert_offsets[E] is written exactly once
    assert int(lay.expert_offsets[-1]) == wl.T * wl.k
    assert torch.equal(torch.sort(d).values, torch.arange(wl.T * wl.k, device=DEV))
    # sampled tokens against the oracle
    rng = np.random.default_rng(0)
    ts = np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 254, replace=False)])
    dst = lay.dst_row.cpu().numpy()[ts]
    compact = np.arange(len(ts) * wl.k, dtype=np.int32).reshape(len(ts), wl.k)
    ref = oracle.dispatch_bf16(_bits(x[torch.from_numpy(ts).to(DEV)]), compact, compact.size)
    got = _bits(recv[torch.from_numpy(dst.reshape(-1)).long().to(DEV)])
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------- dispatch FP8

def _fp8_compare(x, lay, wl, q, s, ts=None):
    dst = lay.dst_row.cpu().numpy()
    if ts is not None:
        dst = dst[ts]
        xb = _bits(x[torch.from_numpy(ts).to(DEV)])
    else:
        xb = _bits(x)
    used = dst.reshape(-1)
    keep = used >= 0
    compact = np.full(used.shape, -1, np.int32)
    compact[keep] = np.arange(int(keep.sum()), dtype=np.int32)
    rq, rs = oracle.dispatch_fp8(xb, compact.reshape(dst.shape), int(keep.sum()))
    rows = torch.from_numpy(used[keep].astype(np.int64)).to(DEV)
    assert np.array_equal(q[rows].cpu().numpy(), rq), "FP8 codes differ"
    assert np.array_equal(s[rows].cpu().numpy().view(np.uint32), rs.view(np.uint32)), "scales differ"


@pytest.mark.parametrize("name,T,H", [("decode_fp8", 2048, 7168), ("prefill_fp8", 1500, 7168),
                                      ("decode_fp8", 130, 128), ("prefill_fp8", 33, 384)])
def test_dispatch_fp8_bit_exact(name, T, H):
    wl = W.WORKLOADS[name].scaled(T=T, H=H, capacity=min(W.WORKLOADS[name].capacity, T) or None)
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    q = torch.full((wl.rows, wl.H), 0x5A, dtype=torch.uint8, device=DEV)
    s = torch.full((wl.rows, wl.H // 128), -1.0, dtype=torch.float32, device=DEV)
    ep.dispatch_fp8(x, lay.dst_row, wl.rows, recv_q=q, recv_scale=s, status=lay.status)
    assert ep.status_read(lay.status) == 0
    _fp8_compare(x, lay, wl, q, s)
    # rows no pair maps to are untouched
    mask = torch.ones(wl.rows, dtype=torch.bool, device=DEV)
    mask[lay.dst_row.view(-1).long()] = False
    assert torch.all(q[mask] == 0x5A) and torch.all(s[mask] == -1.0)


def test_dispatch_fp8_every_bf16_pattern():
    # all 65536 bf16 bit patterns (non-finite ones replaced by 0), 512 blocks
    # of 128 consecutive patterns, so the per-block scale and the conversion
    # are exercised across every exponent, both signs and subnormals
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = (bits & 0x7F80) != 0x7F80
    bits = np.where(finite, bits, 0).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16).reshape(64, 1024)).view(torch.bfloat16).to(DEV)
    # also a permuted copy so blocks mix magnitudes
    perm = np.random.default_rng(11).permutation(65536)
    x2 = torch.from_numpy(bits[perm].view(np.int16).reshape(64, 1024)).view(torch.bfloat16).to(DEV)
    for xx in (x, x2):
        dst = torch.arange(64, dtype=torch.int32, device=DEV).view(64, 1)
        q, s = ep.dispatch_fp8(xx, dst, 64)
        rq, rs = oracle.dispatch_fp8(_bits(xx), dst.cpu().numpy(), 64)
        assert np.array_equal(q.cpu().numpy(), rq)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_dispatch_fp8_full_size_sampled():
    wl = W.WORKLOADS["prefill_fp8"]
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    q, s = ep.dispatch_fp8(x, lay.dst_row, wl.rows, status=lay.status)
    assert ep.status_read(lay.status) == 0
    rng = np.random.default_rng(1)
    ts = np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 126, replace=False)])
    _fp8_compare(x, lay, wl, q, s, ts=ts)
    # property at full size: all k copies of a token are identical
    d = lay.dst_row.long()
    for c0 in range(0, wl.T, 8192):
        blk = d[c0:c0 + 8192]
        q0 = q[blk[:, 0]]
        for j in range(1, wl.k):
            assert torch.equal(q[blk[:, j]], q0)
            assert torch.equal(s[blk[:, j]], s[blk[:, 0]])


# --------------------------------------------------------------------------- combine

def _expert_outputs(wl, x, idx, lay, recv):
    if wl.expert_out == "recv":
        return recv
    if wl.expert_out == "scaled_recv":
        row_expert = torch.full((wl.rows,), -1, dtype=torch.int64, device=DEV)
        row_expert[lay.dst_row.view(-1).long()] = idx.view(-1).long()
        return W.scale_rows(recv, row_expert, W.expert_scales(wl, device=DEV))
    return W.independent_expert_outputs(wl, device=DEV)


@pytest.mark.parametrize("name,T,H", [("small", 128, 2048), ("masked", 2048, 2048),
                                      ("decode_fp8", 600, 7168), ("prefill", 1500, 7168),
                                      ("prefill_fp8", 1100, 1024), ("masked", 45, 8)])
def test_combine_within_tolerance_and_fma_exact(name, T, H):
    wl = W.WORKLOADS[name].scaled(T=T, H=H, capacity=min(W.WORKLOADS[name].capacity, T) or None)
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    recv = ep.dispatch(x, lay.dst_row, wl.rows, status=lay.status)
    y = _expert_outputs(wl, x, idx, lay, recv)
    out = ep.combine(y, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    dst = lay.dst_row.cpu().numpy()
    yb, wb = _bits(y), w.cpu().numpy()
    ob, ref, absum = oracle.combine_f64(yb, wb, dst)
    check_combine(_bits(out), ref, absum, name)
    assert np.array_equal(_bits(out), oracle.combine_fp32_seq(yb, wb, dst))
    if wl.expert_out == "recv":           # identity experts, weights summing to ~1
        xf = bf16_to_f64(_bits(x))
        assert np.all(np.abs(bf16_to_f64(_bits(out)) - xf * wb.astype(np.float64).sum(1)[:, None])
                      <= 2.0 ** -7 * np.abs(xf) + 1e-30)


def test_combine_dropped_pairs_and_unit_weight():
    rows, H = 40, 256
    y = torch.randn(rows, H, device=DEV).to(torch.bfloat16)
    dst = torch.tensor([[3, -1, 7], [-1, -1, -1], [39, 0, -1], [5, 5, 5]], dtype=torch.int32, device=DEV)
    w = torch.tensor([[0.5, 9.0, 0.25], [1, 1, 1], [1.0, 0.0, 3.0], [1, -1, 0.5]], device=DEV)
    out = ep.combine(y, w, dst)
    ref = oracle.combine_fp32_seq(_bits(y), w.cpu().numpy(), dst.cpu().numpy())
    assert np.array_equal(_bits(out), ref)
    assert torch.all(out[1].view(torch.int16) == 0)         # no valid pair -> +0
    one = torch.ones(4, 1, device=DEV)
    d1 = torch.tensor([[2], [17], [0], [39]], dtype=torch.int32, device=DEV)
    assert torch.equal(ep.combine(y, one, d1).view(torch.int16), y[d1.view(-1).long()].view(torch.int16))


def test_combine_bad_rows_flagged():
    y = torch.randn(8, 64, device=DEV).to(torch.bfloat16)
    dst = torch.tensor([[1, 8], [2, -2]], dtype=torch.int32, device=DEV)
    w = torch.ones(2, 2, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = ep.combine(y, w, dst, status=status)
    assert ep.status_read(status) == ep.EP_FLAG_BAD_ROW
    assert torch.equal(out.view(torch.int16), y[[1, 2]].view(torch.int16))


def test_combine_full_size_prefill_sampled():
    wl = W.WORKLOADS["prefill"]
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    recv = ep.dispatch(x, lay.dst_row, wl.rows, status=lay.status)
    out = ep.combine(recv, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    # property at full size: identity experts give x * sum_j w_j within 2^-7
    xs = x.float() * w.sum(1, keepdim=True)
    assert torch.all((out.float() - xs).abs() <= 2.0 ** -7 * xs.abs() + 1e-30)
    rng = np.random.default_rng(2)
    ts = np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 254, replace=False)])
    dst = lay.dst_row.cpu().numpy()[ts]
    compact = np.arange(dst.size, dtype=np.int32).reshape(dst.shape)
    yb = _bits(recv[torch.from_numpy(dst.reshape(-1)).long().to(DEV)])
    wb = w.cpu().numpy()[ts]
    ob, ref, absum = oracle.combine_f64(yb, wb, compact)
    got = _bits(out[torch.from_numpy(ts).to(DEV)])
    check_combine(got, ref, absum, "prefill full")
    assert np.array_equal(got, oracle.combine_fp32_seq(yb, wb, compact))


def test_combine_full_size_fp8_workload_sampled():
    wl = W.WORKLOADS["prefill_fp8"]
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    y = W.independent_expert_outputs(wl, device=DEV)
    out = ep.combine(y, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    rng = np.random.default_rng(3)
    ts = np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 126, replace=False)])
    dst = lay.dst_row.cpu().numpy()[ts]
    compact = np.arange(dst.size, dtype=np.int32).reshape(dst.shape)
    yb = _bits(y[torch.from_numpy(dst.reshape(-1)).long().to(DEV)])
    wb = w.cpu().numpy()[ts]
    ob, ref, absum = oracle.combine_f64(yb, wb, compact)
    got = _bits(out[torch.from_numpy(ts).to(DEV)])
    check_combine(got, ref, absum, "prefill_fp8 full")
    assert np.array_equal(got, oracle.combine_fp32_seq(yb, wb, compact))


# --------------------------------------------------------------------------- expert alignment, reuse

@pytest.mark.parametrize("T,k,E,R,alignment", [(1, 1, 1, 1, 4), (700, 8, 256, 16, 128), (3000, 8, 64, 4, 8),
                                               (2048, 4, 128, 4, 16), (129, 3, 7, 7, 2)])
def test_aligned_layout_and_path(T, k, E, R, alignment):
    rng = np.random.default_rng(T + alignment)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    lay = ep.layout(torch.from_numpy(idx).to(DEV), E, R, "contiguous", alignment=alignment)
    ref = oracle.layout_aligned(idx, E, R, alignment)
    assert np.array_equal(lay.expert_counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(lay.expert_offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(lay.dst_row.cpu().numpy(), ref["dst_row"])
    assert np.array_equal(lay.rank_token_counts.cpu().numpy(), ref["rank_token_counts"])
    assert ep.status_read(lay.status) == ref["flags"]
    rows = ep.binding.aligned_rows_bound(T, k, E, alignment)
    assert int(lay.expert_offsets[-1]) <= rows
    H = 256
    x = torch.randn(T, H, device=DEV).to(torch.bfloat16)
    recv = torch.full((rows, H), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    ep.dispatch(x, lay.dst_row, rows, recv=recv)
    rrecv = oracle.dispatch_bf16(_bits(x), ref["dst_row"], rows,
                                 recv=np.full((rows, H), np.uint16(0xABCD), np.uint16))
    assert np.array_equal(_bits(recv), rrecv)          # padding rows keep the sentinel
    w = torch.rand(T, k, device=DEV)
    out = ep.combine(recv, w, lay.dst_row)
    assert np.array_equal(_bits(out), oracle.combine_fp32_seq(rrecv, w.cpu().numpy(), ref["dst_row"]))


def test_layout_reused_across_calls():
    # the route is fixed: one layout serves several dispatch / combine calls
    wl = W.WORKLOADS["masked"].scaled(T=900, H=512, capacity=900)
    idx = W.route(wl, device=DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    ref = oracle.layout(idx.cpu().numpy(), wl.E, wl.R, oracle.LAYOUT_MASKED, wl.capacity)
    for seed in range(3):
        g = torch.Generator(device=DEV).manual_seed(seed)
        x = torch.randn(wl.T, wl.H, generator=g, device=DEV).to(torch.bfloat16)
        w = torch.rand(wl.T, wl.k, generator=g, device=DEV)
        recv = ep.dispatch(x, lay.dst_row, wl.rows)
        out = ep.combine(recv, w, lay.dst_row)
        rrecv = oracle.dispatch_bf16(_bits(x), ref["dst_row"], wl.rows)
        used = rows_of(ref["dst_row"])
        assert np.array_equal(_bits(recv)[used], rrecv[used])
        assert np.array_equal(_bits(out), oracle.combine_fp32_seq(rrecv, w.cpu().numpy(), ref["dst_row"]))


# --------------------------------------------------------------------------- large top-k (k > 8)

@pytest.mark.parametrize("k,E,H", [(9, 64, 1024), (16, 256, 7168), (32, 1024, 512)])
def test_large_topk_paths(k, E, H):
    # k > 8 takes the generic paths (row pointers in passes of 8, combine
    # batches of 8 rows inside each column group)
    T = 300
    rng = np.random.default_rng(k * 7 + E)
    keys = rng.random((T, E))
    idx = np.argsort(-keys, axis=1)[:, :k].astype(np.int32)   # k distinct experts per token
    idx[5, 3] = -1                                              # one unrouted pair
    idx_d = torch.from_numpy(idx).to(DEV)
    lay = ep.layout(idx_d, E, 4, "contiguous")
    ref = _compare_layout(idx, E, 4, "contiguous", 0, lay, expect_flags=0)
    rows = T * k
    x = torch.randn(T, H, device=DEV).to(torch.bfloat16)
    recv = ep.dispatch(x, lay.dst_row, rows, status=lay.status)
    rrecv = oracle.dispatch_bf16(_bits(x), ref["dst_row"], rows)
    used = rows_of(ref["dst_row"])
    assert np.array_equal(_bits(recv)[used], rrecv[used])
    if H % 128 == 0:
        q, s = ep.dispatch_fp8(x, lay.dst_row, rows, status=lay.status)
        rq, rs = oracle.dispatch_fp8(_bits(x), ref["dst_row"], rows)
        assert np.array_equal(q.cpu().numpy()[used], rq[used])
        assert np.array_equal(s.cpu().numpy()[used].view(np.uint32), rs[used].view(np.uint32))
    w = torch.rand(T, k, device=DEV)
    y = torch.randn(rows, H, device=DEV).to(torch.bfloat16)
    out = ep.combine(y, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    yb = _bits(y)
    assert np.array_equal(_bits(out), oracle.combine_fp32_seq(yb, w.cpu().numpy(), ref["dst_row"]))
    _, r64, absum = oracle.combine_f64(yb, w.cpu().numpy(), ref["dst_row"])
    check_combine(_bits(out), r64, absum, "k=%d" % k)


# --------------------------------------------------------------------------- 32-byte combine path

@pytest.mark.parametrize("T,k,H,offset", [(17000, 8, 528, 0), (20000, 16, 1024, 0), (16384, 8, 256, 16)])
def test_combine_large_batch_paths(T, k, H, offset):
    # T >= 16384 with H % 16 == 0 and 32-byte-aligned buffers takes the
    # 32-byte-access kernel (k > 8: its batched path); a 16-byte offset on the
    # output falls back to the 16-byte kernel.  Results are the same FMA chain.
    E = 64
    rng = np.random.default_rng(T + k)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[7, 1] = -1
    lay = ep.layout(torch.from_numpy(idx).to(DEV), E, 4, "contiguous")
    rows = T * k
    y = torch.randn(rows, H, device=DEV).to(torch.bfloat16)
    w = torch.rand(T, k, device=DEV)
    raw = torch.empty(T * H + offset // 2 + 16, dtype=torch.bfloat16, device=DEV)
    out = raw[offset // 2: offset // 2 + T * H].view(T, H)
    ep.combine(y, w, lay.dst_row, out=out, status=lay.status)
    assert ep.status_read(lay.status) == 0
    rng2 = np.random.default_rng(0)
    ts = np.concatenate([[0, 7, T - 1], rng2.choice(T, 200, replace=False)])
    dst = lay.dst_row.cpu().numpy()[ts]
    keep = dst >= 0
    compact = np.where(keep, np.arange(dst.size, dtype=np.int32).reshape(dst.shape), -1).astype(np.int32)
    gather = torch.from_numpy(np.where(keep, dst, 0).reshape(-1).astype(np.int64)).to(DEV)
    yb = _bits(y[gather])
    wb = w.cpu().numpy()[ts]
    got = _bits(out[torch.from_numpy(ts).to(DEV)])
    assert np.array_equal(got, oracle.combine_fp32_seq(yb, wb, compact))
    _, r64, absum = oracle.combine_f64(yb, wb, compact)
    check_combine(got, r64, absum, "T=%d k=%d" % (T, k))


def test_dispatch_fp8_every_pattern_at_fixed_scales():
    # blocks of 128 channels: slot 0 holds A (the block amax, which fixes
    # inv = 448 / max(A, 1e-4)); slots 1..127 hold every finite bf16 pattern of
    # magnitude <= A, so the conversion of v * inv is checked for all patterns
    # at each of these scales
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).float().numpy()
    finite = np.isfinite(vals)
    rows = []
    for A in (1e-4, 0.01, 1.0, 3.14159, 448.0, 1e4, 6e4):
        a_bits = W.bf16_bits(torch.tensor([A], dtype=torch.float32).to(torch.bfloat16))[0]
        a_val = float(torch.tensor([A]).to(torch.bfloat16).float())
        sel = pats[finite & (np.abs(vals) <= a_val)]
        nblk = -(-len(sel) // 127)
        blk = np.zeros((nblk, 128), np.uint16)
        blk[:, 0] = a_bits
        flat = np.zeros(nblk * 127, np.uint16)
        flat[:len(sel)] = sel
        blk[:, 1:] = flat.reshape(nblk, 127)
        rows.append(blk.reshape(-1))
    allv = np.concatenate(rows)
    H = 1024
    allv = np.concatenate([allv, np.zeros((-len(allv)) % H, np.uint16)]).reshape(-1, H)
    T = allv.shape[0]
    x = torch.from_numpy(allv.view(np.int16)).view(torch.bfloat16).to(DEV)
    dst = torch.arange(T, dtype=torch.int32, device=DEV).view(T, 1)
    q, s = ep.dispatch_fp8(x, dst, T)
    rq, rs = oracle.dispatch_fp8(allv, dst.cpu().numpy(), T)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


# --------------------------------------------------------------------------- layout + dispatch in one call

@pytest.mark.parametrize("T,k,E,R,kind,cap,H,fp8,rows_cut,bad", [
    (128, 8, 128, 4, "contiguous", 0, 2048, False, 0, False),      # the small workload's shape
    (1, 8, 64, 4, "contiguous", 0, 7168, False, 0, False),
    (1, 8, 64, 4, "contiguous", 0, 7168, True, 0, False),
    (37, 13, 32, 4, "contiguous", 0, 1336, False, 0, False),       # k > 8, ragged slices
    (200, 8, 64, 8, "masked", 10, 256, False, 0, False),           # capacity overflow
    (128, 8, 256, 16, "contiguous", 0, 7168, True, 0, False),      # largest fused batch
    (120, 8, 256, 16, "masked", 128, 1024, False, 0, True),        # bad expert ids
    (256, 8, 256, 16, "masked", 256, 1024, False, 0, True),        # bad ids, two launches
    (100, 8, 64, 4, "contiguous", 0, 512, False, 7, False),        # rows too few: BAD_ROW
    (257, 8, 256, 16, "contiguous", 0, 1024, True, 0, False),      # above the fused range
    (300, 8, 64, 4, "contiguous", 0, 512, True, 7, False),         # two launches, rows too few
    (1000, 8, 64, 4, "masked", 200, 512, False, 3000, False),      # masked rows past the buffer
    (129, 6, 96, 3, "masked", 40, 2048, False, 0, True),           # overflow, bad ids, 30-lane pieces
    (3000, 8, 256, 16, "masked", 3000, 512, False, 0, False),
    # two launches, the dispatch reading x before the layout ends: the
    # decode-like FP8 shape, the masked BF16 shape, and the large-batch
    # instance (one block per SM) from 16,384 tokens
    (2048, 8, 256, 16, "masked", 2048, 7168, True, 0, False),
    (2048, 8, 128, 4, "masked", 2048, 2048, False, 0, True),
    (17000, 8, 256, 16, "contiguous", 0, 512, False, 0, False),
    (17000, 8, 256, 16, "contiguous", 0, 512, True, 0, False),
])
def test_layout_dispatch_matches_oracle(T, k, E, R, kind, cap, H, fp8, rows_cut, bad):
    rng = np.random.default_rng(T * 31 + H + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if bad:
        idx[3, 2] = E + 3
        idx[5, 0] = -7
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32) * 2).to(torch.bfloat16)
    okind = oracle.LAYOUT_MASKED if kind == "masked" else oracle.LAYOUT_CONTIGUOUS
    ref = oracle.layout(idx, E, R, okind, cap)
    rows = (T * k if kind == "contiguous" else E * cap) - rows_cut
    xd, idd = x.to(DEV), torch.from_numpy(idx).to(DEV)
    if fp8:
        q0 = torch.full((rows, H), 0x5A, dtype=torch.uint8, device=DEV)
        s0 = torch.full((rows, H // 128), -1.0, dtype=torch.float32, device=DEV)
        lay, q, sc = ep.layout_dispatch(xd, idd, E, R, kind, cap, rows, fp8=True, recv_q=q0,
                                        recv_scale=s0)
    else:
        r0 = torch.full((rows, H), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        lay, recv = ep.layout_dispatch(xd, idd, E, R, kind, cap, rows, recv=r0)
    assert np.array_equal(lay.expert_counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(lay.expert_offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(lay.dst_row.cpu().numpy(), ref["dst_row"])
    assert np.array_equal(lay.rank_token_counts.cpu().numpy(), ref["rank_token_counts"])
    expect_flags = ref["flags"] | (ep.EP_FLAG_BAD_ROW if (ref["dst_row"] >= rows).any() else 0)
    assert ep.status_read(lay.status) == expect_flags
    dst = np.where(ref["dst_row"] < rows, ref["dst_row"], -1)       # rows past the buffer are skipped
    if fp8:
        rq, rs = oracle.dispatch_fp8(_bits(x), dst, rows, recv_q=np.full((rows, H), 0x5A, np.uint8),
                                     recv_scale=np.full((rows, H // 128), -1.0, np.float32))
        assert np.array_equal(q.cpu().numpy(), rq)
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    else:
        rr = oracle.dispatch_bf16(_bits(x), dst, rows, recv=np.full((rows, H), np.uint16(0xABCD), np.uint16))
        assert np.array_equal(_bits(recv), rr)


def test_layout_dispatch_empty_batch():
    idx = torch.zeros(0, 8, dtype=torch.int32, device=DEV)
    x = torch.zeros(0, 256, dtype=torch.bfloat16, device=DEV)
    lay, recv = ep.layout_dispatch(x, idx, 64, 4)
    assert int(lay.expert_counts.abs().sum()) == 0 and int(lay.expert_offsets.abs().sum()) == 0
    assert ep.status_read(lay.status) == 0 and recv.shape == (0, 256)
