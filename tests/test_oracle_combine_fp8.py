"""Pins for the oracle's combine of FP8 expert outputs (codes + one float32
scale per 128 channels, value = decode(code) * scale): special cases, an
independent torch/numpy computation of the same sums, the round trip through
the dispatch's quantisation, and fp32 cases that are exact -- never the
oracle checked against itself."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_02_gb300 import workloads as W


def _decode_torch(q):
    """e4m3 codes -> float64 through torch's float8_e4m3fn (independent of the
    oracle's decoder)."""
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double().numpy()


def _bf16_torch(v32):
    """float32 values -> bf16 bits, one rounding (torch)."""
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _case(T=48, H=384, k=8, rows=200, seed=3, drop=0.1):
    rng = np.random.default_rng(seed)
    wl = W.WORKLOADS["prefill_fp8"].scaled(T=rows // k, H=H, seed=seed)
    q, sc = W.fp8_expert_outputs(wl.scaled(T=rows, k=1))
    q, sc = q.numpy(), sc.numpy()
    dst = rng.integers(0, rows, size=(T, k)).astype(np.int32)
    dst[rng.random((T, k)) < drop] = -1
    w = rng.standard_normal((T, k)).astype(np.float32)
    return q, sc, w, dst


def test_k1_unit_weight_equals_dequantised_row():
    # scales with at most 20 significant bits: decode(q) * scale (<= 24 bits)
    # is exact in fp32, so torch's float32 product and its one bf16 rounding
    # give the exact result to compare with
    rng = np.random.default_rng(11)
    rows, H = 64, 256
    q = rng.integers(0, 254, size=(rows, H)).astype(np.uint8)
    q[q >= 127] += 1
    mant = rng.integers(1 << 19, 1 << 20, size=(rows, H // 128)).astype(np.float64)
    sc = (mant * 2.0 ** rng.integers(-30, -14, size=mant.shape)).astype(np.float32)
    assert np.array_equal(sc.astype(np.float64), mant * 2.0 ** np.log2(sc.astype(np.float64) / mant))
    dst = np.arange(rows, dtype=np.int32).reshape(rows, 1)
    w = np.ones((rows, 1), np.float32)
    out, ref, _ = oracle.combine_fp8_f64(q, sc, w, dst)
    # the sum starts from +0, so a code of -0 (0x80) contributes +0
    val = _decode_torch(q) * np.repeat(sc.astype(np.float64), 128, axis=1) + 0.0
    assert np.array_equal(ref, val) and not np.signbit(ref[q == 0x80]).any()
    assert np.array_equal(val.astype(np.float32).astype(np.float64), val)   # exact in fp32
    assert np.array_equal(out, _bf16_torch(val.astype(np.float32)))
    assert np.array_equal(oracle.combine_fp8_fp32_seq(q, sc, w, dst), out)


def test_f64_sum_matches_independent_numpy():
    q, sc, w, dst = _case()
    out, ref, absum = oracle.combine_fp8_f64(q, sc, w, dst)
    dec = _decode_torch(q)
    scale = np.repeat(sc.astype(np.float64), 128, axis=1)
    T, k = dst.shape
    H = q.shape[1]
    s = np.zeros((T, H))
    sa = np.zeros((T, H))
    for j in range(k):                      # the same j order: identical double sums
        r = dst[:, j]
        ok = (r >= 0)[:, None]
        p = w[:, j].astype(np.float64)[:, None] * (dec[np.maximum(r, 0)] * scale[np.maximum(r, 0)])
        s = s + np.where(ok, p, 0.0)
        sa = sa + np.where(ok, np.abs(p), 0.0)
    assert np.array_equal(ref, s)
    assert np.array_equal(absum, sa)
    # the bf16 rounding of the sum: within half a bf16 ulp (2^-8 relative at
    # most); its exactness is pinned where the sum is exact in fp32 (k = 1)
    got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref))


def test_dropped_pairs_and_empty_tokens():
    q, sc, w, dst = _case(T=6, k=4, rows=40, drop=0.0)
    dst[0, :] = -1                          # no valid pair: +0
    dst[1, 1] = -1
    out, ref, _ = oracle.combine_fp8_f64(q, sc, w, dst)
    assert np.all(out[0] == 0) and np.all(ref[0] == 0.0)
    assert np.all(oracle.combine_fp8_fp32_seq(q, sc, w, dst)[0] == 0)
    keep = dst.copy()
    keep[1, 1] = dst[1, 0]                  # same sum as dropping pair 1 and doubling weight 0
    w2 = w.copy()
    w2[1, 1] = 0.0
    _, ref2, _ = oracle.combine_fp8_f64(q, sc, w2, keep)
    assert np.array_equal(ref[1], ref2[1])


def test_nan_code_propagates():
    q = np.zeros((1, 128), np.uint8)
    q[0, 5] = 0x7F
    sc = np.ones((1, 1), np.float32)
    dst = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1), np.float32)
    out, ref, _ = oracle.combine_fp8_f64(q, sc, w, dst)
    assert np.isnan(ref[0, 5]) and out[0, 5] & 0x7FFF > 0x7F80
    assert np.all(out[0, :5] == 0) and np.all(out[0, 6:] == 0)


@pytest.mark.parametrize("name", ["prefill_fp8", "decode_fp8"])
def test_round_trip_through_the_dispatch_quantisation(name):
    # identity experts: every pair's row is the token's own FP8-quantised
    # row, weights sum to 1 -> out ~= x within the e4m3 error
    # (2^-4 |x| in the normal range, 2^-10 * scale below it) plus one bf16
    # rounding and the fp32 weight rounding
    wl = W.WORKLOADS[name].scaled(T=40, H=512, capacity=64)
    xb = W.bf16_bits(W.hidden_states(wl))
    T, k = wl.T, wl.k
    q = np.zeros((T, wl.H), np.uint8)
    sc = np.zeros((T, wl.H // 128), np.float32)
    for t in range(T):
        qq, ss = oracle.quantize_row_fp8(xb[t])
        q[t], sc[t] = qq, ss
    dst = np.repeat(np.arange(T, dtype=np.int32)[:, None], k, axis=1)
    lw = np.random.default_rng(5).standard_normal((T, k))
    w64 = np.exp(lw) / np.exp(lw).sum(axis=1, keepdims=True)
    w = w64.astype(np.float32)
    out, ref, _ = oracle.combine_fp8_f64(q, sc, w, dst)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).double().numpy()
    wsum = w.astype(np.float64).sum(axis=1, keepdims=True)
    s_el = np.repeat(sc.astype(np.float64), 128, axis=1)
    bound = (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s_el) * wsum + np.abs(x) * np.abs(wsum - 1)
    assert np.all(np.abs(ref - x) <= bound)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref))


def test_fp32_sequence_within_its_bound():
    q, sc, w, dst = _case(T=64, H=256, rows=300)
    _, ref, absum = oracle.combine_fp8_f64(q, sc, w, dst)
    seq = oracle.combine_fp8_fp32_seq(q, sc, w, dst)
    got = torch.from_numpy(seq.view(np.int16)).view(torch.bfloat16).double().numpy()
    k = dst.shape[1]
    acc_err = (k + 1) * 2.0 ** -24 * absum
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * (np.abs(ref) + acc_err) + acc_err)


def test_fp32_sequence_k1_matches_torch():
    # k = 1: bf16(fl32(fl32(w * s) * decode(q))), each step computed by torch
    rng = np.random.default_rng(17)
    q, sc, _, _ = _case(rows=50)
    dst = rng.integers(0, 50, size=(80, 1)).astype(np.int32)
    w = rng.standard_normal((80, 1)).astype(np.float32)
    seq = oracle.combine_fp8_fp32_seq(q, sc, w, dst)
    c = torch.from_numpy(w) * torch.from_numpy(sc)[torch.from_numpy(dst[:, 0]).long()]   # fp32, [80, H/128]
    c = c.repeat_interleave(128, dim=1).double()
    prod = (c * torch.from_numpy(_decode_torch(q)[dst[:, 0]])).float()  # exact in double, one fp32 rounding
    prod = prod + 0.0                       # the chain starts from +0: -0 products give +0
    assert np.array_equal(seq, _bf16_torch(prod.numpy()))


def test_fp32_sequence_exact_on_dyadic_data():
    # weights k/8, scales 2^-2..2^0 and codes of magnitude 0.5..15: every
    # coefficient, product and partial sum is exact in fp32, so the fp32
    # chain and the fp64 sum agree bit for bit (a misplaced scale block, row
    # or weight in either would break this)
    rng = np.random.default_rng(23)
    rows, H, T, k = 96, 384, 40, 8
    e = rng.integers(6, 11, size=(rows, H))          # exponent field: 2^-1 .. 2^3
    m = rng.integers(0, 8, size=(rows, H))
    sgn = rng.integers(0, 2, size=(rows, H))
    q = ((sgn << 7) | (e << 3) | m).astype(np.uint8)
    sc = (2.0 ** rng.integers(-2, 1, size=(rows, H // 128))).astype(np.float32)
    w = (rng.integers(1, 9, size=(T, k)) / 8.0).astype(np.float32)
    dst = rng.integers(0, rows, size=(T, k)).astype(np.int32)
    out, ref, _ = oracle.combine_fp8_f64(q, sc, w, dst)
    assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)
    assert np.array_equal(oracle.combine_fp8_fp32_seq(q, sc, w, dst), out)
    # and a transposed scale (block index from the row, not the channel) is caught
    sc_bad = sc.copy()
    sc_bad[:, [0, 1]] = sc_bad[:, [1, 0]]
    assert not np.array_equal(oracle.combine_fp8_f64(q, sc_bad, w, dst)[1], ref)
