"""The seeded input recipe: shapes, dtypes, determinism, and the
distributions the workloads are defined with."""
import numpy as np
import pytest
import torch

from combine_ep_layout_02_gb300 import workloads as W


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_shapes_dtypes_and_determinism(name):
    wl = W.WORKLOADS[name].scaled(T=min(W.WORKLOADS[name].T, 300), H=256)
    x1, x2 = W.hidden_states(wl), W.hidden_states(wl)
    assert x1.dtype == torch.bfloat16 and x1.shape == (wl.T, wl.H)
    assert torch.equal(x1.view(torch.int16), x2.view(torch.int16))
    idx = W.route(wl)
    assert idx.dtype == torch.int32 and idx.shape == (wl.T, wl.k)
    assert torch.equal(idx, W.route(wl))
    assert int(idx.min()) >= 0 and int(idx.max()) < wl.E
    assert all(len(set(r)) == wl.k for r in idx.tolist())          # k distinct experts
    w = W.topk_weights(wl)
    assert w.dtype == torch.float32 and w.shape == (wl.T, wl.k)
    assert torch.all(w > 0) and torch.allclose(w.double().sum(1), torch.ones(wl.T, dtype=torch.float64), atol=1e-6)
    # different workloads draw different streams
    other = W.WORKLOADS["small" if name != "small" else "masked"].scaled(T=wl.T, H=wl.H)
    assert not torch.equal(W.hidden_states(other).view(torch.int16), x1.view(torch.int16))


def test_hidden_states_are_standard_normal():
    wl = W.WORKLOADS["prefill"].scaled(T=512, H=2048)
    x = W.hidden_states(wl).float()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01


def test_outlier_channels():
    wl = W.WORKLOADS["prefill_fp8"].scaled(T=2000)
    x = W.hidden_states(wl).float()
    col_std = x.std(dim=0)
    big = col_std > 10
    assert int(big.sum()) == round(0.01 * wl.H) == 72                # 1 % of 7168 channels
    assert float(col_std[big].mean()) == pytest.approx(100.0, rel=0.05)
    assert float(col_std[~big].mean()) == pytest.approx(1.0, rel=0.05)


def test_zipf_popularity_follows_rank():
    wl = W.WORKLOADS["prefill_fp8"].scaled(T=20000)   # s = 1.2
    cnt = np.bincount(W.route(wl).numpy().reshape(-1), minlength=wl.E)
    assert cnt[0] > cnt[1] > cnt[3] > cnt[15] > cnt[255]
    # sampling without replacement caps every expert at one pair per token
    assert cnt.max() <= wl.T
    uni = W.WORKLOADS["decode_fp8"].scaled(T=20000)
    cu = np.bincount(W.route(uni).numpy().reshape(-1), minlength=uni.E)
    assert cu.max() / cu.min() < 1.3                                  # uniform: flat


def test_expert_scales_and_independent_outputs():
    wl = W.WORKLOADS["small"]
    s = W.expert_scales(wl)
    assert s.shape == (wl.E,) and float(s.min()) >= 0.5 and float(s.max()) < 1.5
    wl2 = W.WORKLOADS["masked"].scaled(T=64, H=64, capacity=64)
    y = W.independent_expert_outputs(wl2)
    assert y.shape == (wl2.rows, wl2.H) and y.dtype == torch.bfloat16


def test_logical_bytes_formula():
    wl = W.WORKLOADS["prefill"]
    d, c = wl.logical_bytes()
    assert d == c == wl.T * wl.k * wl.H * 2
    f = W.WORKLOADS["prefill_fp8"]
    d, c = f.logical_bytes()
    assert d == f.T * f.k * (f.H + 4 * f.H // 128) and c == f.T * f.k * f.H * 2


def test_grouped_route_spans_few_ranks():
    wl = W.WORKLOADS["prefill_grouped"].scaled(T=4000)
    idx = W.route(wl).numpy()
    per = wl.E // wl.R
    ranks = idx // per
    spans = np.array([len(set(r)) for r in ranks.tolist()])
    assert spans.max() <= wl.groups_per_token                     # at most 4 of the 8 ranks
    assert spans.min() >= -(-wl.k // per)                          # k experts need this many ranks
    assert all(len(set(r)) == wl.k for r in idx.tolist())          # distinct experts
    # every rank and expert is used, roughly evenly (uniform within the chosen ranks)
    cnt = np.bincount(idx.reshape(-1), minlength=wl.E)
    assert cnt.min() > 0 and cnt.max() / cnt.min() < 1.6
    rc = np.bincount(ranks.reshape(-1), minlength=wl.R)
    assert rc.max() / rc.min() < 1.2
