"""Pins for the oracle's dispatch (BF16, FP8) and combine: closed forms,
invariants, error bounds and special cases, plus independent numpy / torch
computations -- never the oracle checked against itself."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_02_gb300 import workloads as W


def _inputs(name, T, H=None, seed_shift=0):
    wl = W.WORKLOADS[name].scaled(T=T, H=H)
    x = W.hidden_states(wl)
    idx = W.route(wl)
    w = W.topk_weights(wl)
    kind = oracle.LAYOUT_MASKED if wl.kind == "masked" else oracle.LAYOUT_CONTIGUOUS
    cap = min(wl.capacity, wl.T) if wl.kind == "masked" else 0
    wl = wl.scaled(capacity=cap)
    lay = oracle.layout(idx.numpy(), wl.E, wl.R, kind, cap)
    return wl, W.bf16_bits(x), idx.numpy(), w.numpy(), lay


def _f(bits):
    """bf16 bits -> float64 via torch (independent of the oracle)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


# ------------------------------------------------------------------ BF16 dispatch

@pytest.mark.parametrize("name", ["small", "masked", "prefill"])
def test_dispatch_bf16_closed_form(name):
    wl, x, idx, w, lay = _inputs(name, T=96, H=256)
    sentinel = np.uint16(0xDEAD)
    recv = np.full((wl.rows, wl.H), sentinel, np.uint16)
    oracle.dispatch_bf16(x, lay["dst_row"], wl.rows, recv)
    dst = lay["dst_row"]
    written = np.zeros(wl.rows, bool)
    for t in range(wl.T):
        for j in range(wl.k):
            r = dst[t, j]
            assert r >= 0
            assert np.array_equal(recv[r], x[t])
            written[r] = True
    # rows no pair maps to keep their sentinel (masked padding)
    assert np.all(recv[~written] == sentinel)
    # per-expert checksum: sum of row sums equals the routed tokens' sums
    tok_sum = x.astype(np.int64).sum(axis=1)
    row_sum = recv.astype(np.int64).sum(axis=1)
    assert row_sum[written].sum() == sum(tok_sum[t] for t in range(wl.T) for j in range(wl.k))


def test_dispatch_skips_dropped_pairs():
    x = np.arange(2 * 16, dtype=np.uint16).reshape(2, 16)
    dst = np.array([[1, -1], [-1, 0]], np.int32)
    recv = np.full((3, 16), 7, np.uint16)
    oracle.dispatch_bf16(x, dst, 3, recv)
    assert np.array_equal(recv[1], x[0]) and np.array_equal(recv[0], x[1])
    assert np.all(recv[2] == 7)


# ------------------------------------------------------------------ FP8 dispatch

def _dequant(q, s):
    H = q.shape[-1]
    vals = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double().numpy()
    return vals * np.repeat(s.astype(np.float64), 128, axis=-1).reshape(vals.shape)


@pytest.mark.parametrize("name", ["decode_fp8", "prefill_fp8"])
def test_fp8_quantisation_properties(name):
    wl, x, idx, w, lay = _inputs(name, T=64, H=1024)
    xf = _f(x)
    for t in range(wl.T):
        q, s = oracle.quantize_row_fp8(x[t])
        assert q.dtype == np.uint8 and s.shape == (wl.H // 128,)
        deq = _dequant(q, s)
        for b in range(wl.H // 128):
            blk = xf[t, b * 128:(b + 1) * 128]
            amax = np.abs(blk).max()
            qb = q[b * 128:(b + 1) * 128]
            sb = float(s[b])
            # the scale is amax / 448 up to one fp32 rounding
            assert abs(sb * 448.0 - max(amax, 1e-4)) <= 2.0 ** -23 * max(amax, 1e-4)
            if amax >= 1e-4:
                # the block maximum lands on the largest finite code
                assert np.any((qb & 0x7F) == 0x7E)
            # no code is NaN, signs follow x
            assert not np.any((qb & 0x7F) == 0x7F)
            nz = blk != 0
            assert np.all((qb[nz] >> 7) == (blk[nz] < 0))
            # e4m3 error bound: half an ulp relative in the normal range,
            # half a subnormal step (2^-10 * sf) below 2^-6 * sf
            err = np.abs(deq[b * 128:(b + 1) * 128] - blk)
            bound = np.maximum(2.0 ** -4 * np.abs(blk) * (1 + 2.0 ** -20), 2.0 ** -10 * sb * (1 + 2.0 ** -20))
            assert np.all(err <= bound + 1e-30)


def test_fp8_codes_match_torch_encoder():
    wl, x, idx, w, lay = _inputs("prefill_fp8", T=32, H=7168)
    xf32 = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    for t in range(wl.T):
        q, s = oracle.quantize_row_fp8(x[t])
        blocks = xf32[t].view(-1, 128)
        amax = blocks.abs().amax(dim=1).clamp_min(1e-4)
        inv = torch.tensor(448.0, dtype=torch.float32) / amax        # fp32 IEEE division
        qt = (blocks * inv.view(-1, 1)).to(torch.float8_e4m3fn).view(torch.uint8).reshape(-1).numpy()
        assert np.array_equal(q, qt)
        assert np.array_equal(s, (amax / torch.tensor(448.0)).numpy())


def test_fp8_zero_and_tiny_blocks():
    x = np.zeros((1, 256), np.uint16)
    x[0, 128:] = W.bf16_bits(torch.full((128,), 3e-5, dtype=torch.bfloat16))
    q, s = oracle.quantize_row_fp8(x[0])
    assert np.all(q[:128] == 0)
    assert 0 < s[0] < 1e-6 and s[0] == s[1]        # both blocks sit on the amax floor
    assert np.all(q[128:] < 0x7E)                   # below the floor the block max is not 448
    deq = _dequant(q, s)
    assert np.allclose(deq[128:], 3e-5, rtol=2.0 ** -4)


def test_fp8_dispatch_copies_codes_and_scales():
    wl, x, idx, w, lay = _inputs("decode_fp8", T=40, H=512)
    rq, rs = oracle.dispatch_fp8(x, lay["dst_row"], wl.rows)
    for t in range(wl.T):
        q, s = oracle.quantize_row_fp8(x[t])
        for j in range(wl.k):
            r = lay["dst_row"][t, j]
            assert np.array_equal(rq[r], q) and np.array_equal(rs[r], s)


# ------------------------------------------------------------------ combine

def test_combine_k1_unit_weight_is_exact():
    rng = np.random.default_rng(3)
    y = W.bf16_bits(torch.from_numpy(rng.standard_normal((10, 64)).astype(np.float32)).to(torch.bfloat16))
    dst = rng.permutation(10)[:6].reshape(6, 1).astype(np.int32)
    w = np.ones((6, 1), np.float32)
    out, ref, _ = oracle.combine_f64(y, w, dst)
    assert np.array_equal(out, y[dst[:, 0]])
    assert np.array_equal(oracle.combine_fp32_seq(y, w, dst), y[dst[:, 0]])


def test_combine_matches_numpy_f64_and_bf16_rounding():
    wl, x, idx, w, lay = _inputs("masked", T=64, H=256)
    rng = np.random.default_rng(5)
    y = W.bf16_bits(torch.from_numpy(rng.standard_normal((wl.rows, wl.H)).astype(np.float32)).to(torch.bfloat16))
    dst = lay["dst_row"].copy()
    dst[3, 2] = -1          # a dropped pair contributes nothing
    dst[5, :] = -1          # a token with no valid pair gives +0
    out, ref, absum = oracle.combine_f64(y, w, dst)
    yf = _f(y)
    valid = dst >= 0
    np_ref = np.einsum("tj,tjh->th", np.where(valid, w.astype(np.float64), 0.0), yf[np.where(valid, dst, 0)])
    np_abs = np.einsum("tj,tjh->th", np.where(valid, np.abs(w.astype(np.float64)), 0.0), np.abs(yf[np.where(valid, dst, 0)]))
    assert np.allclose(ref, np_ref, rtol=0, atol=1e-12 * np_abs.max())
    assert np.allclose(absum, np_abs, rtol=1e-12, atol=0)
    outf = _f(out)
    # one RNE rounding to bf16: within half an ulp (2^-8 relative to the
    # value's binade, i.e. at most 2^-8 |ref|)
    assert np.all(np.abs(outf - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-40)
    assert np.all(out[5] == 0)
    # torch's float32 -> bf16 rounding agrees wherever ref is exactly a float32
    r32 = ref.astype(np.float32)
    exact = r32.astype(np.float64) == ref
    tb = torch.from_numpy(r32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out[exact], tb[exact])


def test_combine_identity_experts_return_input():
    # y = dispatched rows, weights summing to one (renormalised in fp64)
    wl, x, idx, w, lay = _inputs("small", T=64, H=256)
    recv = oracle.dispatch_bf16(x, lay["dst_row"], wl.rows)
    w64 = w.astype(np.float64)
    w1 = (w64 / w64.sum(axis=1, keepdims=True)).astype(np.float32)
    out, ref, _ = oracle.combine_f64(recv, w1, lay["dst_row"])
    xf = _f(x)
    assert np.all(np.abs(_f(out) - xf) <= 2.0 ** -7 * np.abs(xf))
    assert np.mean(out == x) > 0.99


def test_combine_scaled_experts_closed_form():
    # y[row] = bf16(recv[row] * s_e)  =>  out ~= x * sum_j w_j s_{e_j}
    wl, x, idx, w, lay = _inputs("small", T=64, H=256)
    recv = oracle.dispatch_bf16(x, lay["dst_row"], wl.rows)
    s = W.expert_scales(wl)
    row_expert = torch.full((wl.rows,), -1, dtype=torch.int64)
    row_expert[torch.from_numpy(lay["dst_row"].reshape(-1)).long()] = torch.from_numpy(idx.reshape(-1)).long()
    recv_t = torch.from_numpy(recv.view(np.int16)).view(torch.bfloat16)
    y = W.bf16_bits(W.scale_rows(recv_t, row_expert, s))
    out, ref, _ = oracle.combine_f64(y, w, lay["dst_row"])
    factor = (w.astype(np.float64) * s.numpy().astype(np.float64)[idx]).sum(axis=1)
    expect = _f(x) * factor[:, None]
    # y rounding (2^-8 relative) plus the final bf16 rounding
    assert np.all(np.abs(_f(out) - expect) <= (2.0 ** -8 + 2.0 ** -8 + 2.0 ** -14) * np.abs(expect) + 1e-40)


def test_combine_fp32_sequence_within_fp32_bound():
    wl, x, idx, w, lay = _inputs("masked", T=64, H=256)
    rng = np.random.default_rng(9)
    y = W.bf16_bits(torch.from_numpy(rng.standard_normal((wl.rows, wl.H)).astype(np.float32)).to(torch.bfloat16))
    out, ref, absum = oracle.combine_f64(y, w, lay["dst_row"])
    seq = oracle.combine_fp32_seq(y, w, lay["dst_row"])
    err = np.abs(_f(seq) - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + wl.k * 2.0 ** -24 * absum * 1.01 + 1e-40)
