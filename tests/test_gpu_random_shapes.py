"""Randomised shapes through the whole path (layout, BF16 and FP8 dispatch,
combine) against the oracle, plus the path captured in a CUDA graph on a
non-default stream and replayed."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import workloads as W

from gpu_helpers import DEV, check_combine

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _bits(t):
    return W.bf16_bits(t)


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    T = int(rng.choice([1, 2, 7, 31, 64, 127, 128, 129, 500, 513, 1000, 2049, 5000]))
    k = int(rng.choice([1, 2, 3, 5, 8, 11, 16]))
    R = int(rng.choice([1, 2, 3, 4, 8]))
    E = R * int(rng.integers(max(1, -(-k // R)), 48))
    H = int(rng.choice([8, 64, 128, 384, 520, 1024, 2048, 2176]))
    kind = "masked" if rng.random() < 0.4 else "contiguous"
    cap = int(rng.integers(1, max(2, T))) if kind == "masked" else 0
    dup = rng.random() < 0.3
    if dup:   # repeated experts within a token, and some -1
        idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    else:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    return T, k, E, R, H, kind, cap, idx


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes_end_to_end(seed):
    T, k, E, R, H, kind, cap, idx = _random_case(seed)
    okind = oracle.LAYOUT_MASKED if kind == "masked" else oracle.LAYOUT_CONTIGUOUS
    ref = oracle.layout(idx, E, R, okind, cap)
    lay = ep.layout(torch.from_numpy(idx).to(DEV), E, R, kind, cap)
    assert np.array_equal(lay.dst_row.cpu().numpy(), ref["dst_row"])
    assert np.array_equal(lay.expert_counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(lay.expert_offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(lay.rank_token_counts.cpu().numpy(), ref["rank_token_counts"])
    assert ep.status_read(lay.status) == ref["flags"]
    rows = T * k if kind == "contiguous" else E * cap
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = (torch.randn(T, H, generator=g, device=DEV) * 3).to(torch.bfloat16)
    used = ref["dst_row"].reshape(-1)
    used = used[used >= 0]
    if rows > 0:
        recv = ep.dispatch(x, lay.dst_row, rows)
        rrecv = oracle.dispatch_bf16(_bits(x), ref["dst_row"], rows)
        assert np.array_equal(_bits(recv)[used], rrecv[used])
        if H % 128 == 0:
            q, s = ep.dispatch_fp8(x, lay.dst_row, rows)
            rq, rs = oracle.dispatch_fp8(_bits(x), ref["dst_row"], rows)
            assert np.array_equal(q.cpu().numpy()[used], rq[used])
            assert np.array_equal(s.cpu().numpy()[used].view(np.uint32), rs[used].view(np.uint32))
    y = torch.randn(max(rows, 1), H, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.rand(T, k, generator=g, device=DEV) - 0.25        # some negative weights
    out = ep.combine(y, w, lay.dst_row)
    yb, wb = _bits(y), w.cpu().numpy()
    assert np.array_equal(_bits(out), oracle.combine_fp32_seq(yb, wb, ref["dst_row"]))
    _, r64, absum = oracle.combine_f64(yb, wb, ref["dst_row"])
    check_combine(_bits(out), r64, absum, "seed %d" % seed)


def test_whole_path_in_cuda_graph_on_side_stream():
    wl = W.WORKLOADS["prefill"].scaled(T=4000, H=1024)
    x, idx, w = W.hidden_states(wl, device=DEV), W.route(wl, device=DEV), W.topk_weights(wl, device=DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    ws = torch.empty(ep.layout_workspace_bytes(wl.T, wl.k, wl.E, wl.R), dtype=torch.uint8, device=DEV)
    recv = torch.empty(wl.rows, wl.H, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):       # warm-up on the side stream
        ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity, out=lay, workspace=ws)
        ep.dispatch(x, lay.dst_row, wl.rows, recv=recv, status=lay.status)
        ep.combine(recv, w, lay.dst_row, out=out, status=lay.status)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity, out=lay, workspace=ws)
        ep.dispatch(x, lay.dst_row, wl.rows, recv=recv, status=lay.status)
        ep.combine(recv, w, lay.dst_row, out=out, status=lay.status)
    for trial in range(3):
        out.zero_()
        lay.dst_row.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert ep.status_read(lay.status) == 0
        ref = oracle.layout(idx.cpu().numpy(), wl.E, wl.R)
        assert np.array_equal(lay.dst_row.cpu().numpy(), ref["dst_row"])
        rrecv = oracle.dispatch_bf16(_bits(x), ref["dst_row"], wl.rows)
        assert np.array_equal(_bits(out), oracle.combine_fp32_seq(rrecv, w.cpu().numpy(), ref["dst_row"]))
