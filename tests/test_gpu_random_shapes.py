"""Randomised shapes through the whole path (layout, BF16 and FP8 dispatch,
BF16 and FP8 combine) against the oracle, plus the path captured in a CUDA graph on a
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
    if H % 128 == 0:
        # FP8 expert outputs: finite e4m3 codes (no 0x7F / 0xFF) and positive block scales
        codes = torch.randint(0, 254, (max(rows, 1), H), generator=g, device=DEV)
        codes = torch.where(codes >= 0x7F, codes + 1, codes).to(torch.uint8)
        scales = torch.rand(max(rows, 1), H // 128, generator=g, device=DEV) * 4 + 2.0 ** -6
        out8 = ep.combine_fp8(codes, scales, w, lay.dst_row)
        qh, sh = codes.cpu().numpy(), scales.cpu().numpy()
        assert np.array_equal(_bits(out8), oracle.combine_fp8_fp32_seq(qh, sh, wb, ref["dst_row"]))
        _, r64, absum = oracle.combine_fp8_f64(qh, sh, wb, ref["dst_row"])
        check_combine(_bits(out8), r64, absum, "fp8 seed %d" % seed)


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


def _fuzz_shape(rng):
    T = int(rng.choice([rng.integers(1, 70), rng.integers(60, 300), rng.integers(250, 2100),
                        rng.integers(2000, 5000)]))
    k = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 8, 8, 9, 13, 16, 32]))
    E = int(rng.choice([1, 3, 8, 32, 64, 96, 128, 128, 256, 256, 257, 512, 1000, 1024]))
    R = int(rng.choice([r for r in range(1, E + 1) if E % r == 0]))
    return T, k, E, R


@pytest.mark.parametrize("block", range(3))
def test_layout_fuzz_against_oracle(block):
    """Fifty random layouts per block across every launch shape (single
    block, 8- and 16-block clusters, chunked kernels): ids with -1 and
    occasional bad ids, contiguous / masked / aligned, with and without rank
    counts; every output and the status word equal the oracle's."""
    rng = np.random.default_rng(7000 + block)
    for it in range(50):
        T, k, E, R = _fuzz_shape(rng)
        kind = "masked" if rng.random() < 0.4 else "contiguous"
        cap = int(rng.integers(0, max(2, T * k // E * 2))) if kind == "masked" else 0
        align = int(rng.choice([1, 1, 1, 4, 128])) if kind == "contiguous" else 1
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
        idx[rng.random((T, k)) < 0.05] = -1
        if rng.random() < 0.2:
            for _ in range(int(rng.integers(1, 4))):
                idx[rng.integers(0, T), rng.integers(0, k)] = int(rng.choice([-5, E, E + 7, 1 << 20]))
        ranks = bool(rng.random() < 0.8)
        if align > 1:
            ref = oracle.layout_aligned(idx, E, R, align)
        else:
            ref = oracle.layout(idx, E, R, oracle.LAYOUT_MASKED if kind == "masked" else 0, cap)
        lay = ep.layout(torch.from_numpy(idx).to(DEV), E, R, kind, cap, with_rank_counts=ranks,
                        alignment=align)
        what = "case %d: T=%d k=%d E=%d R=%d %s cap=%d align=%d" % (it, T, k, E, R, kind, cap, align)
        assert np.array_equal(lay.expert_counts.cpu().numpy(), ref["counts"]), what
        assert np.array_equal(lay.expert_offsets.cpu().numpy(), ref["offsets"]), what
        assert np.array_equal(lay.dst_row.cpu().numpy(), ref["dst_row"]), what
        if ranks:
            assert np.array_equal(lay.rank_token_counts.cpu().numpy(), ref["rank_token_counts"]), what
        assert ep.status_read(lay.status) == ref["flags"], what


def test_layout_dispatch_fuzz_against_oracle():
    """Forty random ep_layout_dispatch calls (one launch up to 128 tokens,
    two above), BF16 and FP8, some with a dispatch buffer too small for every
    row: layout, rows and status equal the oracle's."""
    rng = np.random.default_rng(7100)
    for it in range(40):
        T = int(rng.choice([rng.integers(1, 130), rng.integers(120, 400)]))
        k = int(rng.choice([1, 2, 4, 6, 8, 8, 13]))
        E = int(rng.choice([16, 32, 64, 96, 128, 256]))
        R = int(rng.choice([r for r in range(1, E + 1) if E % r == 0]))
        kind = "masked" if rng.random() < 0.4 else "contiguous"
        cap = int(rng.integers(1, max(2, T * k // E * 2))) if kind == "masked" else 0
        H = int(rng.choice([128, 256, 1024, 2048]))
        fp8 = bool(rng.random() < 0.5)
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        if rng.random() < 0.2:
            idx[rng.integers(0, T), rng.integers(0, k)] = E + 3
        full = T * k if kind == "contiguous" else E * cap
        rows = full - (int(rng.integers(0, max(1, full // 4))) if rng.random() < 0.3 else 0)
        x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
        ref = oracle.layout(idx, E, R, oracle.LAYOUT_MASKED if kind == "masked" else 0, cap)
        dst = np.where(ref["dst_row"] < rows, ref["dst_row"], -1)
        xd, idd = x.to(DEV), torch.from_numpy(idx).to(DEV)
        what = "case %d: T=%d k=%d E=%d %s cap=%d H=%d fp8=%s rows=%d" % (it, T, k, E, kind, cap, H,
                                                                       fp8, rows)
        if fp8:
            q0 = torch.full((rows, H), 0x5A, dtype=torch.uint8, device=DEV)
            s0 = torch.full((rows, H // 128), -1.0, dtype=torch.float32, device=DEV)
            lay, q, sc = ep.layout_dispatch(xd, idd, E, R, kind, cap, rows, fp8=True, recv_q=q0,
                                            recv_scale=s0)
            rq, rs = oracle.dispatch_fp8(_bits(x), dst, rows,
                                         recv_q=np.full((rows, H), 0x5A, np.uint8),
                                         recv_scale=np.full((rows, H // 128), -1.0, np.float32))
            assert np.array_equal(q.cpu().numpy(), rq), what
            assert np.array_equal(sc.cpu().numpy().view(np.uint32), rs.view(np.uint32)), what
        else:
            r0 = torch.full((rows, H), -21555, dtype=torch.int16, device=DEV).view(torch.bfloat16)
            lay, recv = ep.layout_dispatch(xd, idd, E, R, kind, cap, rows, recv=r0)
            rr = oracle.dispatch_bf16(_bits(x), dst, rows,
                                      recv=np.full((rows, H), np.uint16(0xABCD), np.uint16))
            assert np.array_equal(_bits(recv), rr), what
        assert np.array_equal(lay.dst_row.cpu().numpy(), ref["dst_row"]), what
        assert np.array_equal(lay.expert_offsets.cpu().numpy(), ref["offsets"]), what
        expect = ref["flags"] | (ep.EP_FLAG_BAD_ROW if (ref["dst_row"] >= rows).any() else 0)
        assert ep.status_read(lay.status) == expect, what
