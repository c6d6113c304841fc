"""Pins for the oracle's routing layout: brute force on tiny inputs, the
invariants of a stable slot assignment, and the balanced route's closed form."""
import json
import os
from collections import Counter

import numpy as np
import pytest

import oracle
from combine_ep_layout_02_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_force_layout(idx, E, R, kind, cap):
    """O(n^2) direct count, written independently of the oracle."""
    T, k = idx.shape
    flat = [int(v) for v in idx.reshape(-1)]
    valid = [0 <= e < E for e in flat]
    flags = 0
    if any(e < -1 or e >= E for e in flat):
        flags |= oracle.FLAG_BAD_EXPERT
    counts = [sum(1 for p in range(len(flat)) if valid[p] and flat[p] == e) for e in range(E)]
    offsets = [sum(counts[:e]) for e in range(E + 1)]
    dst = []
    for p, e in enumerate(flat):
        if not valid[p]:
            dst.append(-1)
            continue
        slot = sum(1 for q in range(p) if valid[q] and flat[q] == e)
        if kind == oracle.LAYOUT_CONTIGUOUS:
            dst.append(offsets[e] + slot)
        elif slot < cap:
            dst.append(e * cap + slot)
        else:
            dst.append(-1)
            flags |= oracle.FLAG_OVERFLOW
    per = E // R
    rtc = [sum(1 for t in range(T) if any(0 <= flat[t * k + j] < E and flat[t * k + j] // per == r
                                            for j in range(k))) for r in range(R)]
    return (np.array(counts), np.array(offsets), np.array(dst).reshape(T, k), np.array(rtc), flags)


@pytest.mark.parametrize("E,R", [(1, 1), (2, 1), (3, 3), (8, 2), (128, 4)])
@pytest.mark.parametrize("k", [1, 2, 8])
@pytest.mark.parametrize("T", [1, 5, 33, 64])
def test_layout_matches_brute_force(T, k, E, R):
    rng = np.random.default_rng(T * 1000 + k * 10 + E)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)   # duplicates and -1 allowed
    for kind, cap in [(oracle.LAYOUT_CONTIGUOUS, 0), (oracle.LAYOUT_MASKED, max(1, T * k // max(E, 1) // 2)),
                      (oracle.LAYOUT_MASKED, T * k)]:
        got = oracle.layout(idx, E, R, kind, cap)
        c, o, d, r, f = brute_force_layout(idx, E, R, kind, cap)
        assert np.array_equal(got["counts"], c)
        assert np.array_equal(got["offsets"], o)
        assert np.array_equal(got["dst_row"], d)
        assert np.array_equal(got["rank_token_counts"], r)
        assert got["flags"] == f


def test_layout_bad_expert_flag_and_skip():
    idx = np.array([[0, 5, -1], [7, 1, -3]], np.int32)
    got = oracle.layout(idx, E=4, R=2)
    assert got["flags"] == oracle.FLAG_BAD_EXPERT
    assert got["dst_row"].tolist() == [[0, -1, -1], [-1, 1, -1]]
    assert got["counts"].tolist() == [1, 1, 0, 0]
    assert got["rank_token_counts"].tolist() == [2, 0]


def test_layout_rejects_bad_sizes():
    idx = np.zeros((4, 2), np.int32)
    with pytest.raises(ValueError):
        oracle.layout(idx, E=6, R=4)      # E % R != 0


def _check_invariants(idx, E, kind, cap, got):
    T, k = idx.shape
    dst = got["dst_row"].reshape(-1)
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    cnt = Counter(flat[valid].tolist())
    assert got["counts"].sum() == valid.sum()
    for e in range(E):
        assert got["counts"][e] == cnt.get(e, 0)
    kept = dst[dst >= 0]
    assert len(np.unique(kept)) == len(kept)                 # injective
    if kind == oracle.LAYOUT_CONTIGUOUS:
        assert np.array_equal(np.sort(kept), np.arange(got["offsets"][E]))
        assert (dst >= 0).sum() == valid.sum()
    else:
        expect = sorted(e * cap + s for e in range(E) for s in range(min(cnt.get(e, 0), cap)))
        assert np.sort(kept).tolist() == expect
    # stable: within an expert the rows increase with the pair index
    for e in range(E):
        rows = dst[(flat == e) & (dst >= 0)]
        assert np.all(np.diff(rows) > 0)
    # row -> expert consistency
    rows_e = flat[dst >= 0]
    if kind == oracle.LAYOUT_CONTIGUOUS:
        lo = got["offsets"][rows_e]
        hi = got["offsets"][rows_e + 1]
        assert np.all((kept >= lo) & (kept < hi))
    else:
        assert np.array_equal(kept // cap, rows_e)


@pytest.mark.parametrize("name", ["small", "masked", "decode_fp8"])
def test_layout_invariants_on_workloads(name):
    wl = W.WORKLOADS[name]
    wl = wl.scaled(T=min(wl.T, 1024))
    idx = W.route(wl).numpy()
    kind = oracle.LAYOUT_MASKED if wl.kind == "masked" else oracle.LAYOUT_CONTIGUOUS
    got = oracle.layout(idx, wl.E, wl.R, kind, wl.capacity)
    assert got["flags"] == 0
    _check_invariants(idx, wl.E, kind, wl.capacity, got)


def test_layout_invariants_zipf_and_overflow():
    wl = W.WORKLOADS["prefill"].scaled(T=2048)
    idx = W.route(wl).numpy()
    got = oracle.layout(idx, wl.E, wl.R)
    _check_invariants(idx, wl.E, oracle.LAYOUT_CONTIGUOUS, 0, got)
    cap = 40   # hot experts overflow
    got = oracle.layout(idx, wl.E, wl.R, oracle.LAYOUT_MASKED, cap)
    assert got["flags"] == oracle.FLAG_OVERFLOW
    _check_invariants(idx, wl.E, oracle.LAYOUT_MASKED, cap, got)
    assert got["counts"].max() > cap     # true counts are still reported


def test_zipf_route_is_skewed_and_distinct():
    wl = W.WORKLOADS["prefill"].scaled(T=4096)
    idx = W.route(wl).numpy()
    assert all(len(set(r)) == wl.k for r in idx.tolist())
    cnt = np.bincount(idx.reshape(-1), minlength=wl.E)
    assert cnt[0] > 3 * cnt[wl.E // 2] and cnt[0] <= wl.T


def test_balanced_route_closed_form():
    with open(os.path.join(GOLDEN, "balanced_route.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        idx = W.balanced_route(case["T"], case["k"], case["E"], case["seed"]).numpy()
        assert all(len(set(r)) == case["k"] for r in idx.tolist())
        got = oracle.layout(idx, case["E"], 16)
        assert np.all(got["counts"] == case["expected_count_per_expert"])
        assert got["offsets"][-1] == case["T"] * case["k"]
        _check_invariants(idx, case["E"], oracle.LAYOUT_CONTIGUOUS, 0, got)


def test_logical_bytes_match_published_payload():
    with open(os.path.join(GOLDEN, "logical_bytes.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        wl = W.WORKLOADS["decode_fp8"].scaled(T=case["T"], H=case["H"], payload=case["payload"])
        disp, comb = wl.logical_bytes()
        # the printed per-rank payload is one dispatch plus one combine
        assert round((disp + comb) / 1e6, 2) == case["MB_per_rank"]
        assert disp + comb == case["bytes"]


@pytest.mark.parametrize("alignment", [1, 2, 8, 128])
@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (40, 8, 16), (300, 4, 7)])
def test_aligned_layout_matches_brute_force(T, k, E, alignment):
    rng = np.random.default_rng(T + k * 17 + E * 101 + alignment)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    got = oracle.layout_aligned(idx, E, 1, alignment)
    counts, _, _, _, flags = brute_force_layout(idx, E, 1, oracle.LAYOUT_CONTIGUOUS, 0)
    # segment starts: running sum of counts rounded up to the alignment
    starts = [0]
    for e in range(E):
        starts.append(starts[-1] + -(-int(counts[e]) // alignment) * alignment)
    assert got["offsets"].tolist() == starts
    assert all(o % alignment == 0 for o in starts)
    flat = idx.reshape(-1)
    dst = got["dst_row"].reshape(-1)
    for p, e in enumerate(flat):
        if 0 <= e < E:
            slot = sum(1 for q in range(p) if flat[q] == e)
            assert dst[p] == starts[e] + slot
        else:
            assert dst[p] == -1
    assert got["flags"] == flags
    assert np.array_equal(got["counts"], counts)
