"""Pins for the oracle's number formats (bf16, OCP E4M3), checked against
the format definitions, hand-derived special cases and PyTorch's independent
CPU conversions -- never against the oracle itself."""
import math

import numpy as np
import pytest
import torch

import oracle


def _torch_e4m3_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy()


def test_e4m3_decode_matches_torch_all_codes():
    ref = _torch_e4m3_decode_all()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), (c, got, ref[c])


def test_e4m3_decode_landmarks():
    # OCP E4M3: bias 7, 3 mantissa bits, max finite 1.75 * 2^8, S.1111.111 = NaN
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9      # smallest subnormal
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    assert math.copysign(1, oracle.e4m3_decode(0x80)) == -1.0


def test_e4m3_roundtrip_all_codes():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_e4m3_encode_matches_torch_random():
    rng = np.random.default_rng(1234)
    mag = np.exp2(rng.uniform(-14, np.log2(448.0), size=20000)).astype(np.float32)
    sign = np.where(rng.random(20000) < 0.5, -1, 1).astype(np.float32)
    v = mag * sign
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(x) for x in v], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_midpoints_go_to_even():
    dec = _torch_e4m3_decode_all()
    n_checked = 0
    for c in range(0, 0x7E):              # positive finite codes c, c+1
        lo, hi = float(dec[c]), float(dec[c + 1])
        mid = np.float32((lo + hi) / 2)     # exact in fp32
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == even, (hex(c), mid)
        assert oracle.e4m3_encode(-float(mid)) == 0x80 | even
        # torch agrees on the ties as well
        assert torch.tensor([mid]).to(torch.float8_e4m3fn).view(torch.uint8).item() == even
        # just off the midpoint goes to the nearer code
        assert oracle.e4m3_encode(float(np.nextafter(mid, np.float32(0)))) == c
        assert oracle.e4m3_encode(float(np.nextafter(mid, np.float32(1e9)))) == c + 1
        n_checked += 1
    assert n_checked == 126


def test_e4m3_subnormal_ties():
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00      # 0 vs 2^-9: even is 0
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02  # m=1 vs m=2: even is 2
    assert oracle.e4m3_encode(15 * 2.0 ** -10) == 0x08  # 7*2^-9 vs 2^-6: even is 0x08
    assert oracle.e4m3_encode(2.0 ** -20) == 0x00
    assert oracle.e4m3_encode(-(2.0 ** -20)) == 0x80


@pytest.mark.parametrize("v", [448.0, 448.5, 463.9, 464.0, 464.1, 479.0, 480.0, 1e6, 3.0e38, math.inf])
def test_e4m3_saturates(v):
    assert oracle.e4m3_encode(v) == 0x7E
    assert oracle.e4m3_encode(-v) == 0xFE


def test_e4m3_nan():
    assert oracle.e4m3_encode(math.nan) == 0x7F


def test_bf16_to_float_matches_torch_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    sample = list(range(0, 65536, 7)) + [0x0000, 0x8000, 0x0001, 0x7F7F, 0xFF7F, 0x7F80]
    for b in sample:
        got = oracle.bf16_to_float(b)
        if math.isnan(ref[b]):
            assert math.isnan(got)
        else:
            assert got == ref[b], hex(b)


def test_bf16_from_double_matches_torch_on_fp32_inputs():
    # For inputs that are already fp32 a single RNE rounding is what torch does.
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # fp32 subnormals
        np.array([0.0, -0.0, 1.0, 3.0e38, -3.0e38], np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(x)) for x in v], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_from_double_is_one_rounding():
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7 (bf16 has 7 stored bits).
    assert oracle.bf16_from_double(1 + 2.0 ** -8) == 0x3F80            # tie -> even
    assert oracle.bf16_from_double(1 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81  # above the tie
    assert oracle.bf16_from_double(1 + 2.0 ** -8 - 2.0 ** -30) == 0x3F80
    assert oracle.bf16_from_double(1 + 3 * 2.0 ** -8) == 0x3F82        # tie -> even (up)
    assert oracle.bf16_from_double(-(1 + 2.0 ** -8 + 2.0 ** -30)) == 0xBF81
    assert oracle.bf16_from_double(0.0) == 0x0000
    assert oracle.bf16_from_double(-0.0) == 0x8000
    # largest finite bf16 and overflow
    assert oracle.bf16_from_double((2 - 2.0 ** -7) * 2.0 ** 127) == 0x7F7F
    assert oracle.bf16_from_double((2 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80  # tie -> even = inf
    assert oracle.bf16_from_double(2.0 ** 129) == 0x7F80
    # bf16 subnormals: spacing 2^-133
    assert oracle.bf16_from_double(2.0 ** -133) == 0x0001
    assert oracle.bf16_from_double(2.0 ** -134) == 0x0000                # tie -> even (0)
    assert oracle.bf16_from_double(3 * 2.0 ** -134) == 0x0002
