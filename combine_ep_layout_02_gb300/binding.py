"""Thin ctypes binding over the C ABI in ``include/ep.h``.

Argument marshalling only: every step of layout, dispatch and combine runs in
the CUDA kernels of ``libep_gb300.so``.  Torch tensors supply device memory
and the current CUDA stream.  If the library is missing this module raises;
there is no fallback of any kind.
"""
import ctypes
import os
from collections import namedtuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_ALIGNMENT = 2
EP_ERR_WORKSPACE = 3
EP_ERR_CUDA = 4

EP_FLAG_BAD_EXPERT = 1
EP_FLAG_OVERFLOW = 2
EP_FLAG_BAD_ROW = 4
EP_FLAG_TIMEOUT = 8

LAYOUT_KINDS = {"contiguous": 0, "masked": 1}

_lib = None


class EpError(RuntimeError):
    def __init__(self, fn, code):
        lib = load()
        msg = lib.ep_status_string(code).decode()
        if code == EP_ERR_CUDA:
            msg += " (cudaError %d)" % lib.ep_last_cuda_error()
        super().__init__("%s failed: %s" % (fn, msg))
        self.code = code


def load():
    """Load libep_gb300.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("CUDA library %s is not built; run __graft_entry__.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sig = {
        "ep_version": ([], i32),
        "ep_status_string": ([i32], ctypes.c_char_p),
        "ep_last_cuda_error": ([], i32),
        "ep_layout_workspace_bytes": ([i64, i32, i32, i32, i32], sz),
        "ep_layout": ([P, i64, i32, i32, i32, i32, i32, P, P, P, P, P, P, sz, P], i32),
        "ep_layout_aligned": ([P, i64, i32, i32, i32, i32, P, P, P, P, P, P, sz, P], i32),
        "ep_layout_static_ws": ([P, i64, i32, i32, i32, i32, i32, P, P, P, P, P, P], i32),
        "ep_dispatch": ([P, i64, i64, i32, P, P, i64, P, P], i32),
        "ep_rank_layout_workspace_bytes": ([i64, i32, i32, i32], sz),
        "ep_rank_layout": ([P, i64, i32, i32, i32, P, P, P, P, P, i64, P, P, sz, P], i32),
        "ep_expand": ([P, P, i32, i64, P, P, P, i64, i64, i32, P, i64, P, P], i32),
        "ep_expand_fp8": ([P, P, P, i32, i64, P, P, P, i64, i64, i32, P, P, i64, P, P], i32),
        "ep_combine_partial": ([P, i64, P, P, P, P, P, i32, i64, i64, i64, i32, P, P, P], i32),
        "ep_combine_reduce": ([P, i64, P, i64, i64, i32, P, P, P], i32),
        "ep_dispatch_fp8": ([P, i64, i64, i32, P, P, P, i64, P, P], i32),
        "ep_layout_dispatch": ([P, i64, i32, i32, i32, i32, i32, P, i64, P, P, P, P, P, i64, P, P,
                                sz, P], i32),
        "ep_layout_dispatch_fp8": ([P, i64, i32, i32, i32, i32, i32, P, i64, P, P, P, P, P, P,
                                    i64, P, P, sz, P], i32),
        "ep_combine": ([P, P, P, i64, i64, i32, i64, P, P, P], i32),
        "ep_combine_fp8": ([P, P, P, P, i64, i64, i32, i64, P, P, P], i32),
        "ep_status_read": ([P, P, P], i32),
        "ep_pipeline_create": ([i32, ctypes.POINTER(ctypes.c_void_p)], i32),
        "ep_pipeline_destroy": ([P], i32),
        "ep_roundtrip_host": ([P, P, P, P, P, P, i64, i64, i32, i32, i32, i32, i32, i64, P, P, P,
                               P, P, P, i64, P, P, P, P, P, P, P, P, sz], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_dev(name, t, dtype, device=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def _on(device):
    """Run the enclosed C call with `device` current (the C ABI launches on the
    current device)."""
    return torch.cuda.device(device)


def _rc(fn, code):
    if code != EP_OK:
        raise EpError(fn, code)


LayoutOut = namedtuple("LayoutOut", "expert_counts expert_offsets dst_row rank_token_counts status")


def layout_workspace_bytes(T, k, E, R, with_rank_counts=True):
    return int(load().ep_layout_workspace_bytes(T, k, E, R, 1 if with_rank_counts else 0))


def aligned_rows_bound(T, k, E, alignment):
    """Rows a dispatch buffer needs for any route under ``ep_layout_aligned``."""
    return T * k + E * (alignment - 1)


def layout(topk_idx, E, R=1, kind="contiguous", capacity=0, *, out=None, workspace=None,
           with_rank_counts=True, alignment=1):
    """Routing layout of ``topk_idx`` [T, k] int32 (see ``ep_layout``; with
    ``alignment`` > 1, ``ep_layout_aligned``, contiguous only)."""
    _check_dev("topk_idx", topk_idx, torch.int32)
    T, k = topk_idx.shape
    dev = topk_idx.device
    if out is None:
        out = LayoutOut(
            torch.empty(E, dtype=torch.int32, device=dev),
            torch.empty(E + 1, dtype=torch.int32, device=dev),
            torch.empty(T, k, dtype=torch.int32, device=dev),
            torch.empty(R, dtype=torch.int32, device=dev) if with_rank_counts else None,
            torch.empty(1, dtype=torch.int32, device=dev),
        )
    need = layout_workspace_bytes(T, k, E, R, out.rank_token_counts is not None)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if alignment != 1:
        if kind != "contiguous":
            raise ValueError("expert alignment applies to the contiguous layout only")
        with _on(dev):
            code = load().ep_layout_aligned(_ptr(topk_idx), T, k, E, R, alignment,
                                            _ptr(out.expert_counts), _ptr(out.expert_offsets),
                                            _ptr(out.dst_row), _ptr(out.rank_token_counts),
                                            _ptr(out.status), _ptr(workspace), wbytes, _stream(dev))
        _rc("ep_layout_aligned", code)
        return out
    with _on(dev):
        code = load().ep_layout(_ptr(topk_idx), T, k, E, R, LAYOUT_KINDS[kind], capacity,
                                _ptr(out.expert_counts), _ptr(out.expert_offsets), _ptr(out.dst_row),
                                _ptr(out.rank_token_counts), _ptr(out.status), _ptr(workspace), wbytes,
                                _stream(dev))
    _rc("ep_layout", code)
    return out


def layout_static_ws(topk_idx, E, R=1, kind="contiguous", capacity=0, *, out=None,
                     with_rank_counts=True):
    """Routing layout through ``ep_layout_static_ws``: the same result as
    ``layout`` without any workspace, for callers that cannot allocate device
    memory.  The outputs must still be passed in (``out``) by such callers;
    when ``out`` is None they are allocated here for convenience."""
    _check_dev("topk_idx", topk_idx, torch.int32)
    T, k = topk_idx.shape
    dev = topk_idx.device
    if out is None:
        out = LayoutOut(
            torch.empty(E, dtype=torch.int32, device=dev),
            torch.empty(E + 1, dtype=torch.int32, device=dev),
            torch.empty(T, k, dtype=torch.int32, device=dev),
            torch.empty(R, dtype=torch.int32, device=dev) if with_rank_counts else None,
            torch.empty(1, dtype=torch.int32, device=dev),
        )
    with _on(dev):
        code = load().ep_layout_static_ws(_ptr(topk_idx), T, k, E, R, LAYOUT_KINDS[kind], capacity,
                                          _ptr(out.expert_counts), _ptr(out.expert_offsets),
                                          _ptr(out.dst_row), _ptr(out.rank_token_counts),
                                          _ptr(out.status), _stream(dev))
    _rc("ep_layout_static_ws", code)
    return out


def dispatch(x, dst_row, rows, recv=None, status=None):
    """BF16 dispatch of ``x`` [T, H] into ``recv`` [rows, H] (see ``ep_dispatch``)."""
    _check_dev("x", x, torch.bfloat16)
    _check_dev("dst_row", dst_row, torch.int32, x.device)
    T, H = x.shape
    k = dst_row.shape[1]
    if recv is None:
        recv = torch.empty(rows, H, dtype=torch.bfloat16, device=x.device)
    _check_dev("recv", recv, torch.bfloat16, x.device)
    with _on(x.device):
        code = load().ep_dispatch(_ptr(x), T, H, k, _ptr(dst_row), _ptr(recv), rows, _ptr(status),
                                  _stream(x.device))
    _rc("ep_dispatch", code)
    return recv


def _new_layout(T, k, E, R, with_rank_counts, dev):
    return LayoutOut(torch.empty(E, dtype=torch.int32, device=dev),
                     torch.empty(E + 1, dtype=torch.int32, device=dev),
                     torch.empty(T, k, dtype=torch.int32, device=dev),
                     torch.empty(R, dtype=torch.int32, device=dev) if with_rank_counts else None,
                     torch.empty(1, dtype=torch.int32, device=dev))


def layout_dispatch(x, topk_idx, E, R=1, kind="contiguous", capacity=0, rows=None, *, out=None,
                    recv=None, workspace=None, with_rank_counts=True, fp8=False, recv_q=None,
                    recv_scale=None):
    """``ep_layout`` then ``ep_dispatch`` (``fp8``: ``ep_dispatch_fp8``) in one
    call (see ``ep_layout_dispatch``): one kernel launch for up to 128 tokens.
    Returns (LayoutOut, recv), or (LayoutOut, recv_q, recv_scale) with ``fp8``."""
    _check_dev("x", x, torch.bfloat16)
    _check_dev("topk_idx", topk_idx, torch.int32, x.device)
    T, H = x.shape
    k = topk_idx.shape[1]
    dev = x.device
    if rows is None:
        rows = T * k if kind == "contiguous" else E * capacity
    if out is None:
        out = _new_layout(T, k, E, R, with_rank_counts, dev)
    need = layout_workspace_bytes(T, k, E, R, out.rank_token_counts is not None)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if fp8:
        if recv_q is None:
            recv_q = torch.empty(rows, H, dtype=torch.uint8, device=dev)
        if recv_scale is None:
            recv_scale = torch.empty(rows, H // 128, dtype=torch.float32, device=dev)
        _check_dev("recv_q", recv_q, torch.uint8, dev)
        _check_dev("recv_scale", recv_scale, torch.float32, dev)
        with _on(dev):
            code = load().ep_layout_dispatch_fp8(
                _ptr(topk_idx), T, k, E, R, LAYOUT_KINDS[kind], capacity, _ptr(x), H,
                _ptr(out.expert_counts), _ptr(out.expert_offsets), _ptr(out.dst_row),
                _ptr(out.rank_token_counts), _ptr(recv_q), _ptr(recv_scale), rows, _ptr(out.status),
                _ptr(workspace), wbytes, _stream(dev))
        _rc("ep_layout_dispatch_fp8", code)
        return out, recv_q, recv_scale
    if recv is None:
        recv = torch.empty(rows, H, dtype=torch.bfloat16, device=dev)
    _check_dev("recv", recv, torch.bfloat16, dev)
    with _on(dev):
        code = load().ep_layout_dispatch(
            _ptr(topk_idx), T, k, E, R, LAYOUT_KINDS[kind], capacity, _ptr(x), H,
            _ptr(out.expert_counts), _ptr(out.expert_offsets), _ptr(out.dst_row),
            _ptr(out.rank_token_counts), _ptr(recv), rows, _ptr(out.status), _ptr(workspace),
            wbytes, _stream(dev))
    _rc("ep_layout_dispatch", code)
    return out, recv


def dispatch_fp8(x, dst_row, rows, recv_q=None, recv_scale=None, status=None):
    """FP8 e4m3 dispatch with fused per-128-channel scaling (see ``ep_dispatch_fp8``).
    Returns (recv_q uint8 [rows, H], recv_scale float32 [rows, H/128])."""
    _check_dev("x", x, torch.bfloat16)
    _check_dev("dst_row", dst_row, torch.int32, x.device)
    T, H = x.shape
    k = dst_row.shape[1]
    if recv_q is None:
        recv_q = torch.empty(rows, H, dtype=torch.uint8, device=x.device)
    if recv_scale is None:
        recv_scale = torch.empty(rows, H // 128, dtype=torch.float32, device=x.device)
    _check_dev("recv_q", recv_q, torch.uint8, x.device)
    _check_dev("recv_scale", recv_scale, torch.float32, x.device)
    with _on(x.device):
        code = load().ep_dispatch_fp8(_ptr(x), T, H, k, _ptr(dst_row), _ptr(recv_q), _ptr(recv_scale),
                                      rows, _ptr(status), _stream(x.device))
    _rc("ep_dispatch_fp8", code)
    return recv_q, recv_scale


def combine(y, topk_w, dst_row, out=None, status=None):
    """Weighted top-k combine of ``y`` [rows, H] into ``out`` [T, H] (see ``ep_combine``)."""
    _check_dev("y", y, torch.bfloat16)
    _check_dev("topk_w", topk_w, torch.float32, y.device)
    _check_dev("dst_row", dst_row, torch.int32, y.device)
    rows, H = y.shape
    T, k = dst_row.shape
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    _check_dev("out", out, torch.bfloat16, y.device)
    with _on(y.device):
        code = load().ep_combine(_ptr(y), _ptr(topk_w), _ptr(dst_row), T, H, k, rows, _ptr(out),
                                 _ptr(status), _stream(y.device))
    _rc("ep_combine", code)
    return out


def combine_fp8(y_q, y_scale, topk_w, dst_row, out=None, status=None):
    """Weighted top-k combine of FP8 expert outputs (codes ``y_q`` [rows, H]
    uint8, scales ``y_scale`` [rows, H/128] float32) into ``out`` [T, H] bf16
    (see ``ep_combine_fp8``)."""
    _check_dev("y_q", y_q, torch.uint8)
    _check_dev("y_scale", y_scale, torch.float32, y_q.device)
    _check_dev("topk_w", topk_w, torch.float32, y_q.device)
    _check_dev("dst_row", dst_row, torch.int32, y_q.device)
    rows, H = y_q.shape
    T, k = dst_row.shape
    if tuple(y_scale.shape) != (rows, H // 128):
        raise ValueError("y_scale must be [rows, H/128]")
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=y_q.device)
    _check_dev("out", out, torch.bfloat16, y_q.device)
    with _on(y_q.device):
        code = load().ep_combine_fp8(_ptr(y_q), _ptr(y_scale), _ptr(topk_w), _ptr(dst_row), T, H,
                                     k, rows, _ptr(out), _ptr(status), _stream(y_q.device))
    _rc("ep_combine_fp8", code)
    return out


RankLayoutOut = namedtuple("RankLayoutOut",
                           "rank_counts rank_offsets rank_dst_row pair_rank_row rank_row_token status")


def rank_rows_bound(T, k, R):
    """Rows a rank buffer needs for any route: one per (token, rank) reached."""
    return T * min(k, R)


def rank_layout(topk_idx, E, R, *, out=None, workspace=None):
    """Two-stage layout (see ``ep_rank_layout``)."""
    _check_dev("topk_idx", topk_idx, torch.int32)
    T, k = topk_idx.shape
    dev = topk_idx.device
    cap = rank_rows_bound(T, k, R)
    if out is None:
        out = RankLayoutOut(torch.empty(R, dtype=torch.int32, device=dev),
                            torch.empty(R + 1, dtype=torch.int32, device=dev),
                            torch.empty(T, k, dtype=torch.int32, device=dev),
                            torch.empty(T, k, dtype=torch.int32, device=dev),
                            torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                            torch.empty(1, dtype=torch.int32, device=dev))
    need = int(load().ep_rank_layout_workspace_bytes(T, k, E, R))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() if workspace is not None else 0
    with _on(dev):
        code = load().ep_rank_layout(_ptr(topk_idx), T, k, E, R, _ptr(out.rank_counts),
                                     _ptr(out.rank_offsets), _ptr(out.rank_dst_row),
                                     _ptr(out.pair_rank_row), _ptr(out.rank_row_token),
                                     out.rank_row_token.numel(), _ptr(out.status), _ptr(workspace),
                                     wbytes, _stream(dev))
    _rc("ep_rank_layout", code)
    return out


def expand(rank_buf, rl, dst_row, rows, recv=None, status=None):
    """Expansion of rank rows into the expert rows (see ``ep_expand``)."""
    _check_dev("rank_buf", rank_buf, torch.bfloat16)
    T, k = dst_row.shape
    H = rank_buf.shape[1]
    R = rl.rank_counts.numel()
    if recv is None:
        recv = torch.empty(rows, H, dtype=torch.bfloat16, device=rank_buf.device)
    with _on(rank_buf.device):
        code = load().ep_expand(_ptr(rank_buf), _ptr(rl.rank_offsets), R, rank_buf.shape[0],
                                _ptr(rl.rank_row_token), _ptr(rl.pair_rank_row), _ptr(dst_row), T, H,
                                k, _ptr(recv), rows, _ptr(status), _stream(rank_buf.device))
    _rc("ep_expand", code)
    return recv


def expand_fp8(rank_q, rank_scale, rl, dst_row, rows, recv_q=None, recv_scale=None, status=None):
    """Expansion of FP8 rank rows (codes and scales) into the expert rows (see ``ep_expand_fp8``)."""
    _check_dev("rank_q", rank_q, torch.uint8)
    _check_dev("rank_scale", rank_scale, torch.float32)
    T, k = dst_row.shape
    H = rank_q.shape[1]
    R = rl.rank_counts.numel()
    if recv_q is None:
        recv_q = torch.empty(rows, H, dtype=torch.uint8, device=rank_q.device)
    if recv_scale is None:
        recv_scale = torch.empty(rows, H // 128, dtype=torch.float32, device=rank_q.device)
    with _on(rank_q.device):
        code = load().ep_expand_fp8(_ptr(rank_q), _ptr(rank_scale), _ptr(rl.rank_offsets), R,
                                    rank_q.shape[0], _ptr(rl.rank_row_token), _ptr(rl.pair_rank_row),
                                    _ptr(dst_row), T, H, k, _ptr(recv_q), _ptr(recv_scale), rows,
                                    _ptr(status), _stream(rank_q.device))
    _rc("ep_expand_fp8", code)
    return recv_q, recv_scale


def combine_partial(y, topk_w, dst_row, rl, rank_rows, partial=None, status=None):
    """Rank-local partial reduction (see ``ep_combine_partial``)."""
    _check_dev("y", y, torch.bfloat16)
    T, k = dst_row.shape
    H = y.shape[1]
    R = rl.rank_counts.numel()
    if partial is None:
        partial = torch.empty(max(rank_rows, 1), H, dtype=torch.bfloat16, device=y.device)
    with _on(y.device):
        code = load().ep_combine_partial(_ptr(y), y.shape[0], _ptr(topk_w), _ptr(dst_row),
                                         _ptr(rl.pair_rank_row), _ptr(rl.rank_row_token),
                                         _ptr(rl.rank_offsets), R, rank_rows, T, H, k, _ptr(partial),
                                         _ptr(status), _stream(y.device))
    _rc("ep_combine_partial", code)
    return partial


def combine_reduce(partial, rl, T, out=None, status=None):
    """Final reduction over each token's rank rows (see ``ep_combine_reduce``)."""
    _check_dev("partial", partial, torch.bfloat16)
    H = partial.shape[1]
    k = rl.rank_dst_row.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=partial.device)
    with _on(partial.device):
        code = load().ep_combine_reduce(_ptr(partial), partial.shape[0], _ptr(rl.rank_dst_row), T, H,
                                        k, _ptr(out), _ptr(status), _stream(partial.device))
    _rc("ep_combine_reduce", code)
    return out


def status_read(status):
    """Synchronise the current stream and return the device status word."""
    flags = ctypes.c_uint32(0)
    with _on(status.device):
        code = load().ep_status_read(_ptr(status), _stream(status.device), ctypes.byref(flags))
    _rc("ep_status_read", code)
    return int(flags.value)


class Pipeline:
    """Host-buffer executor (``ep_pipeline_create`` / ``ep_roundtrip_host``):
    one layout + dispatch + combine step from pinned host inputs to a pinned
    host output, with the copies overlapped with the kernels in token chunks.
    Device staging buffers are allocated once here, for one workload shape."""

    def __init__(self, T, H, k, E, R=1, kind="contiguous", capacity=0, chunk_tokens=2048,
                 device=None, y=None, payload="bf16"):
        self.T, self.H, self.k, self.E, self.R = T, H, k, E, R
        self.kind, self.capacity, self.chunk = kind, capacity, chunk_tokens
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.rows = T * k if kind == "contiguous" else E * capacity
        nch = max(1, (T + chunk_tokens - 1) // chunk_tokens)
        h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            _rc("ep_pipeline_create", load().ep_pipeline_create(nch, ctypes.byref(h)))
        self._h = h
        self.x_dev = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.idx_dev = torch.empty(T, k, dtype=torch.int32, device=dev)
        self.w_dev = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.out_dev = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.payload = payload
        if payload == "fp8":
            if y is None:
                raise ValueError("FP8 dispatch needs the expert outputs y to combine")
            self.recv = None
            self.recv_q = torch.empty(self.rows, H, dtype=torch.uint8, device=dev)
            self.recv_scale = torch.empty(self.rows, H // 128, dtype=torch.float32, device=dev)
        else:
            self.recv = torch.empty(self.rows, H, dtype=torch.bfloat16, device=dev)
            self.recv_q = self.recv_scale = None
        self.y = y
        self.layout = LayoutOut(torch.empty(E, dtype=torch.int32, device=dev),
                                torch.empty(E + 1, dtype=torch.int32, device=dev),
                                torch.empty(T, k, dtype=torch.int32, device=dev),
                                torch.empty(R, dtype=torch.int32, device=dev),
                                torch.zeros(1, dtype=torch.int32, device=dev))
        self.ws = torch.empty(max(16, layout_workspace_bytes(T, k, E, R)), dtype=torch.uint8, device=dev)

    def run(self, x_host, idx_host, w_host, out_host):
        """Enqueue one step on the current stream; host tensors must be pinned."""
        for name, t, dt in (("x_host", x_host, torch.bfloat16), ("idx_host", idx_host, torch.int32),
                            ("w_host", w_host, torch.float32), ("out_host", out_host, torch.bfloat16)):
            if t.is_cuda or not t.is_pinned() or t.dtype != dt or not t.is_contiguous():
                raise ValueError("%s must be a pinned contiguous host tensor of %s" % (name, dt))
        lay = self.layout
        with _on(self.device):
            code = load().ep_roundtrip_host(
                self._h, _stream(self.device), _ptr(x_host), _ptr(idx_host), _ptr(w_host),
                _ptr(out_host), self.T, self.H, self.k, self.E, self.R, LAYOUT_KINDS[self.kind],
                self.capacity, self.chunk, _ptr(self.x_dev), _ptr(self.idx_dev), _ptr(self.w_dev),
                _ptr(self.recv), _ptr(self.recv_q), _ptr(self.recv_scale), self.rows, _ptr(self.y),
                _ptr(self.out_dev), _ptr(lay.expert_counts), _ptr(lay.expert_offsets),
                _ptr(lay.dst_row), _ptr(lay.rank_token_counts), _ptr(lay.status), _ptr(self.ws),
                self.ws.numel())
        _rc("ep_roundtrip_host", code)
        return out_host

    def close(self):
        if getattr(self, "_h", None):
            with _on(self.device):
                load().ep_pipeline_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# The C ABI's names, for callers who prefer them (same functions as above).
ep_layout = layout
ep_layout_aligned = layout  # alignment= selects ep_layout_aligned
ep_layout_static_ws = layout_static_ws
ep_dispatch = dispatch
ep_dispatch_fp8 = dispatch_fp8
ep_combine = combine
ep_rank_layout = rank_layout
ep_expand = expand
ep_expand_fp8 = expand_fp8
ep_combine_partial = combine_partial
ep_combine_reduce = combine_reduce
ep_status_read = status_read
ep_layout_workspace_bytes = layout_workspace_bytes
