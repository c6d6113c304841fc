"""Property-based pins for the oracle (hypothesis; skipped where it is not
installed): the layout against an independent brute force on arbitrary tiny
routes, bad ids and capacities; the e4m3 encoder against torch's on arbitrary
in-range fp32 values; the fp64 combine against numpy's float64 arithmetic."""
import numpy as np
import pytest
import torch

import oracle

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies
from hypothesis import given, settings  # noqa: E402

from test_oracle_layout import brute_force_layout  # noqa: E402


@st.composite
def routes(draw):
    R = draw(st.integers(1, 4))
    E = R * draw(st.integers(1, 4))
    T = draw(st.integers(1, 12))
    k = draw(st.integers(1, 5))
    ids = draw(st.lists(st.integers(-3, E + 2), min_size=T * k, max_size=T * k))
    kind = draw(st.sampled_from([oracle.LAYOUT_CONTIGUOUS, oracle.LAYOUT_MASKED]))
    cap = draw(st.integers(0, T * k)) if kind == oracle.LAYOUT_MASKED else 0
    return np.array(ids, np.int32).reshape(T, k), E, R, kind, cap


@settings(max_examples=300, deadline=None)
@given(routes())
def test_layout_equals_brute_force_on_arbitrary_routes(case):
    idx, E, R, kind, cap = case
    got = oracle.layout(idx, E, R, kind, cap)
    c, o, d, r, f = brute_force_layout(idx, E, R, kind, cap)
    assert np.array_equal(got["counts"], c)
    assert np.array_equal(got["offsets"], o)
    assert np.array_equal(got["dst_row"], d)
    assert np.array_equal(got["rank_token_counts"], r)
    assert got["flags"] == f


@settings(max_examples=2000, deadline=None)
@given(st.floats(min_value=-448.0, max_value=448.0, allow_nan=False, width=32))
def test_e4m3_encoder_equals_torch_in_range(v):
    code = oracle.e4m3_encode(np.float32(v))
    ref = torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item()
    assert code == ref


@settings(max_examples=200, deadline=None)
@given(st.integers(1, 6), st.integers(1, 4), st.integers(0, 2 ** 31 - 1))
def test_combine_f64_equals_numpy(T, k, seed):
    rng = np.random.default_rng(seed)
    rows, H = T * k + 2, 8
    y = torch.from_numpy(rng.standard_normal((rows, H)).astype(np.float32)).to(torch.bfloat16)
    yb = y.view(torch.int16).numpy().view(np.uint16)
    w = rng.standard_normal((T, k)).astype(np.float32)
    dst = rng.integers(-1, rows, size=(T, k)).astype(np.int32)
    _, ref, absum = oracle.combine_f64(yb, w, dst)
    yf = y.double().numpy()
    expect = np.zeros((T, H))
    expect_abs = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            if dst[t, j] >= 0:
                expect[t] += np.float64(w[t, j]) * yf[dst[t, j]]
                expect_abs[t] += np.abs(np.float64(w[t, j]) * yf[dst[t, j]])
    # the products are exact in float64 (8 x 24 significant bits); the sum is
    # the same float64 sequence in j order
    assert np.array_equal(ref, expect)
    assert np.array_equal(absum, expect_abs)
