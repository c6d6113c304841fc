"""CPU oracle for MoE routing layout, dispatch and combine.

TEST INFRASTRUCTURE ONLY.  This package may be imported by the test-suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` -- nothing else.  The product path (the CUDA library and its
Python binding) never imports it, and it never imports the product path.

The arithmetic lives in plain single-threaded C (``ep_oracle.c``); this module
only marshals numpy arrays through ctypes.  Each C function cites the passage
it follows.  Parity pins (tests under ``tests/``) check it against brute force,
closed forms, invariants and independent library conversions.
"""
import ctypes

import numpy as np

from . import build as _build

LAYOUT_CONTIGUOUS = 0
LAYOUT_MASKED = 1
FLAG_BAD_EXPERT = 1
FLAG_OVERFLOW = 2

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_float.restype = ctypes.c_float
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_float
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_layout.argtypes = [P, i64, i32, i32, i32, i32, i32, P, P, P, P]
        lib.oracle_layout.restype = ctypes.c_uint32
        lib.oracle_layout_aligned.argtypes = [P, i64, i32, i32, i32, i32, P, P, P, P]
        lib.oracle_layout_aligned.restype = ctypes.c_uint32
        lib.oracle_rank_layout.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P]
        lib.oracle_rank_layout.restype = ctypes.c_uint32
        lib.oracle_expand.argtypes = [P, P, P, i64, i64, i32, P]
        lib.oracle_expand.restype = None
        lib.oracle_combine_partial.argtypes = [P, P, P, P, P, i64, i64, i32, P]
        lib.oracle_combine_partial.restype = None
        lib.oracle_combine_reduce.argtypes = [P, P, i64, i64, i32, P]
        lib.oracle_combine_reduce.restype = None
        lib.oracle_dispatch_bf16.argtypes = [P, i64, i64, i32, P, P]
        lib.oracle_dispatch_bf16.restype = None
        lib.oracle_quantize_row_fp8.argtypes = [P, i64, P, P]
        lib.oracle_quantize_row_fp8.restype = None
        lib.oracle_dispatch_fp8.argtypes = [P, i64, i64, i32, P, P, P]
        lib.oracle_dispatch_fp8.restype = None
        lib.oracle_combine_fp8_f64.argtypes = [P, P, P, P, i64, i64, i32, P, P, P]
        lib.oracle_combine_fp8_f64.restype = None
        lib.oracle_combine_fp8_fp32_seq.argtypes = [P, P, P, P, i64, i64, i32, P]
        lib.oracle_combine_fp8_fp32_seq.restype = None
        lib.oracle_combine_f64.argtypes = [P, P, P, i64, i64, i32, P, P, P]
        lib.oracle_combine_f64.restype = None
        lib.oracle_combine_fp32_seq.argtypes = [P, P, P, i64, i64, i32, P]
        lib.oracle_combine_fp32_seq.restype = None
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


# --- scalar formats -------------------------------------------------------

def bf16_to_float(b):
    return _load().oracle_bf16_to_float(int(b) & 0xFFFF)


def bf16_from_double(v):
    return _load().oracle_bf16_from_double(float(v))


def e4m3_decode(code):
    return _load().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(v):
    return _load().oracle_e4m3_encode(float(v))


# --- layout ---------------------------------------------------------------

def layout(topk_idx, E, R=1, kind=LAYOUT_CONTIGUOUS, capacity=0):
    """Return dict(counts, offsets, dst_row, rank_token_counts, flags)."""
    idx = _c(topk_idx, np.int32)
    if idx.ndim != 2:
        raise ValueError("topk_idx must be [T, k]")
    T, k = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    dst = np.zeros((T, k), np.int32)
    rtc = np.zeros(R, np.int32)
    flags = _load().oracle_layout(_p(idx), T, k, E, R, kind, capacity,
                                  _p(counts), _p(offsets), _p(dst), _p(rtc))
    if flags == 0xFFFFFFFF:
        raise ValueError("oracle_layout: invalid sizes")
    return dict(counts=counts, offsets=offsets, dst_row=dst,
                rank_token_counts=rtc, flags=int(flags))


def layout_aligned(topk_idx, E, R=1, alignment=1):
    """Contiguous layout with expert segments padded to multiples of `alignment`."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    dst = np.zeros((T, k), np.int32)
    rtc = np.zeros(R, np.int32)
    flags = _load().oracle_layout_aligned(_p(idx), T, k, E, R, alignment, _p(counts), _p(offsets),
                                          _p(dst), _p(rtc))
    if flags == 0xFFFFFFFF:
        raise ValueError("oracle_layout_aligned: invalid sizes")
    return dict(counts=counts, offsets=offsets, dst_row=dst, rank_token_counts=rtc,
                flags=int(flags))


# --- dispatch -------------------------------------------------------------

def dispatch_bf16(x, dst_row, rows, recv=None):
    """x: uint16 [T,H] bf16 bits.  Returns recv uint16 [rows,H]."""
    x = _c(x, np.uint16)
    dst = _c(dst_row, np.int32)
    T, H = x.shape
    k = dst.shape[1]
    if recv is None:
        recv = np.zeros((rows, H), np.uint16)
    assert recv.flags.c_contiguous and recv.dtype == np.uint16 and recv.shape == (rows, H)
    _load().oracle_dispatch_bf16(_p(x), T, H, k, _p(dst), _p(recv))
    return recv


def quantize_row_fp8(x_row):
    x_row = _c(x_row, np.uint16)
    H = x_row.shape[0]
    q = np.zeros(H, np.uint8)
    s = np.zeros(H // 128, np.float32)
    _load().oracle_quantize_row_fp8(_p(x_row), H, _p(q), _p(s))
    return q, s


def dispatch_fp8(x, dst_row, rows, recv_q=None, recv_scale=None):
    """Returns (recv_q uint8 [rows,H], recv_scale float32 [rows,H/128])."""
    x = _c(x, np.uint16)
    dst = _c(dst_row, np.int32)
    T, H = x.shape
    k = dst.shape[1]
    if H % 128:
        raise ValueError("FP8 dispatch needs H % 128 == 0")
    if recv_q is None:
        recv_q = np.zeros((rows, H), np.uint8)
    if recv_scale is None:
        recv_scale = np.zeros((rows, H // 128), np.float32)
    _load().oracle_dispatch_fp8(_p(x), T, H, k, _p(dst), _p(recv_q), _p(recv_scale))
    return recv_q, recv_scale


# --- combine --------------------------------------------------------------

def combine_f64(y, topk_w, dst_row):
    """Returns (out uint16 [T,H], ref float64 [T,H], absum float64 [T,H])."""
    y = _c(y, np.uint16)
    w = _c(topk_w, np.float32)
    dst = _c(dst_row, np.int32)
    T, k = dst.shape
    H = y.shape[1]
    out = np.zeros((T, H), np.uint16)
    ref = np.zeros((T, H), np.float64)
    absum = np.zeros((T, H), np.float64)
    _load().oracle_combine_f64(_p(y), _p(w), _p(dst), T, H, k, _p(out), _p(ref), _p(absum))
    return out, ref, absum


def combine_fp32_seq(y, topk_w, dst_row):
    y = _c(y, np.uint16)
    w = _c(topk_w, np.float32)
    dst = _c(dst_row, np.int32)
    T, k = dst.shape
    H = y.shape[1]
    out = np.zeros((T, H), np.uint16)
    _load().oracle_combine_fp32_seq(_p(y), _p(w), _p(dst), T, H, k, _p(out))
    return out


# --- two-stage (rank, then expert) path ------------------------------------

def combine_fp8_f64(y_q, y_scale, topk_w, dst_row):
    """Combine of FP8 expert outputs (codes [rows,H], scales [rows,H/128]).
    Returns (out uint16 [T,H], ref float64 [T,H], absum float64 [T,H])."""
    q = _c(y_q, np.uint8)
    sc = _c(y_scale, np.float32)
    w = _c(topk_w, np.float32)
    dst = _c(dst_row, np.int32)
    T, k = dst.shape
    H = q.shape[1]
    out = np.zeros((T, H), np.uint16)
    ref = np.zeros((T, H), np.float64)
    absum = np.zeros((T, H), np.float64)
    _load().oracle_combine_fp8_f64(_p(q), _p(sc), _p(w), _p(dst), T, H, k, _p(out), _p(ref),
                                   _p(absum))
    return out, ref, absum


def combine_fp8_fp32_seq(y_q, y_scale, topk_w, dst_row):
    """The FP8 combine in fp32 (coefficient w*scale, then an FMA chain in j
    order), rounded to bf16: uint16 [T,H]."""
    q = _c(y_q, np.uint8)
    sc = _c(y_scale, np.float32)
    w = _c(topk_w, np.float32)
    dst = _c(dst_row, np.int32)
    T, k = dst.shape
    H = q.shape[1]
    out = np.zeros((T, H), np.uint16)
    _load().oracle_combine_fp8_fp32_seq(_p(q), _p(sc), _p(w), _p(dst), T, H, k, _p(out))
    return out


def rank_layout(topk_idx, E, R):
    """Returns dict(rank_counts, rank_offsets, rank_dst_row, pair_rank_row,
    rank_row_token, flags); rank_row_token has rank_offsets[R] entries."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    rc = np.zeros(R, np.int32)
    ro = np.zeros(R + 1, np.int32)
    rdst = np.zeros((T, k), np.int32)
    prr = np.zeros((T, k), np.int32)
    tok = np.full(max(1, T * min(k, R)), -1, np.int32)
    flags = _load().oracle_rank_layout(_p(idx), T, k, E, R, _p(rc), _p(ro), _p(rdst), _p(prr), _p(tok))
    if flags == 0xFFFFFFFF:
        raise ValueError("oracle_rank_layout: invalid sizes")
    return dict(rank_counts=rc, rank_offsets=ro, rank_dst_row=rdst, pair_rank_row=prr,
                rank_row_token=tok[:int(ro[R])], flags=int(flags))


def expand(rank_buf, pair_rank_row, dst_row, rows, recv=None):
    rank_buf = _c(rank_buf, np.uint16)
    prr = _c(pair_rank_row, np.int32)
    dst = _c(dst_row, np.int32)
    T, k = dst.shape
    H = rank_buf.shape[1]
    if recv is None:
        recv = np.zeros((rows, H), np.uint16)
    _load().oracle_expand(_p(rank_buf), _p(prr), _p(dst), T, H, k, _p(recv))
    return recv


def combine_partial(y, topk_w, dst_row, pair_rank_row, rank_row_token):
    y = _c(y, np.uint16)
    w = _c(topk_w, np.float32)
    dst = _c(dst_row, np.int32)
    prr = _c(pair_rank_row, np.int32)
    tok = _c(rank_row_token, np.int32)
    k = dst.shape[1]
    H = y.shape[1]
    n = tok.shape[0]
    part = np.zeros((max(n, 1), H), np.uint16)
    _load().oracle_combine_partial(_p(y), _p(w), _p(dst), _p(prr), _p(tok), n, H, k, _p(part))
    return part[:n]


def combine_reduce(partial, rank_dst_row, H):
    part = _c(partial, np.uint16)
    rdst = _c(rank_dst_row, np.int32)
    T, k = rdst.shape
    out = np.zeros((T, H), np.uint16)
    if part.size == 0:
        part = np.zeros((1, H), np.uint16)
    _load().oracle_combine_reduce(_p(part), _p(rdst), T, H, k, _p(out))
    return out


def library_path():
    return _build.build()


__all__ = [
    "LAYOUT_CONTIGUOUS", "LAYOUT_MASKED", "FLAG_BAD_EXPERT", "FLAG_OVERFLOW",
    "bf16_to_float", "bf16_from_double", "e4m3_decode", "e4m3_encode",
    "layout", "layout_aligned", "dispatch_bf16", "quantize_row_fp8", "dispatch_fp8",
    "combine_f64", "combine_fp32_seq", "rank_layout", "expand", "combine_partial",
    "combine_reduce", "library_path",
]
