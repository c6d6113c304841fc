"""The C-ABI library builds, loads and exports every symbol that
include/ep.h declares; host-side argument validation rejects bad calls
before anything is enqueued (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from combine_ep_layout_02_gb300 import build as cuda_build
    cuda_build.build()
    from combine_ep_layout_02_gb300 import binding
    return binding.load()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(ROOT, "include", fn)) as f:
            text = f.read()
        names += re.findall(r"^EP_API\s+[\w\s\*]+?\b(ep_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_hot_path():
    names = declared_functions()
    for required in ("ep_layout", "ep_dispatch", "ep_dispatch_fp8", "ep_combine"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_binding_constants_match_the_header():
    from combine_ep_layout_02_gb300 import binding
    with open(os.path.join(ROOT, "include", "ep.h")) as f:
        text = f.read()
    consts = dict(re.findall(r"\b(EP_(?:FLAG|ERR|OK)\w*)\s*=\s*(\d+)u?\b", text))
    assert {"EP_FLAG_BAD_EXPERT", "EP_FLAG_OVERFLOW", "EP_FLAG_BAD_ROW",
            "EP_ERR_INVALID_ARG", "EP_ERR_ALIGNMENT", "EP_ERR_WORKSPACE", "EP_ERR_CUDA"} <= set(consts)
    for name, value in consts.items():
        assert getattr(binding, name) == int(value), name


def test_version_and_status_strings(lib):
    assert lib.ep_version() >> 16 == 1
    assert lib.ep_status_string(0) == b"EP_OK"
    assert lib.ep_status_string(3) == b"EP_ERR_WORKSPACE"
    assert lib.ep_status_string(99) == b"EP_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    assert lib.ep_layout_workspace_bytes(0, 8, 256, 16, 1) == 0
    # 65536 tokens -> 512 chunks of 128; (256 + 16) columns of int32
    assert lib.ep_layout_workspace_bytes(65536, 8, 256, 16, 1) == 512 * 272 * 4
    assert lib.ep_layout_workspace_bytes(65536, 8, 256, 16, 0) == 512 * 256 * 4
    assert lib.ep_layout_workspace_bytes(1, 8, 3, 1, 0) == 256   # rounded up to 256 bytes


FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails validation


def test_layout_argument_validation(lib):
    def call(T=16, k=8, E=256, R=16, kind=0, cap=0, ws=FAKE, wsb=1 << 30, idx=FAKE, cnt=FAKE,
             off=FAKE, dst=FAKE):
        return lib.ep_layout(idx, T, k, E, R, kind, cap, cnt, off, dst, None, None, ws, wsb, None)
    assert call(E=255) == 1           # E % R != 0
    assert call(k=0) == 1
    assert call(k=33) == 1
    assert call(E=2048, R=1) == 1     # E > EP_MAX_EXPERTS
    assert call(T=-1) == 1
    assert call(kind=7) == 1
    assert call(kind=1, cap=-1) == 1
    assert call(kind=1, cap=1 << 24) == 1      # E * capacity >= 2^31
    assert call(cnt=None) == 1
    assert call(idx=None) == 1
    assert call(ws=None) == 3
    assert call(wsb=16) == 3
    assert call(idx=ctypes.c_void_p((1 << 20) + 2)) == 2
    assert call(ws=ctypes.c_void_p((1 << 20) + 4)) == 2


def test_layout_dispatch_argument_validation(lib):
    def call(fp8=False, T=16, k=8, E=256, R=16, kind=0, cap=0, H=64, x=FAKE, idx=FAKE, ws=FAKE,
             wsb=1 << 30, recv=FAKE, rows=128):
        if fp8:
            return lib.ep_layout_dispatch_fp8(idx, T, k, E, R, kind, cap, x, H, FAKE, FAKE, FAKE,
                                              None, recv, FAKE, rows, None, ws, wsb, None)
        return lib.ep_layout_dispatch(idx, T, k, E, R, kind, cap, x, H, FAKE, FAKE, FAKE, None,
                                      recv, rows, None, ws, wsb, None)
    assert call(E=255) == 1                    # the layout's checks: E % R != 0
    assert call(k=33) == 1
    assert call(ws=None) == 3
    assert call(H=100) == 2                    # the dispatch's: H % 8
    assert call(fp8=True, H=64) == 2           # FP8: H % 128
    assert call(x=None) == 1
    assert call(recv=None) == 1
    assert call(x=ctypes.c_void_p((1 << 20) + 8)) == 2
    assert call(fp8=True, H=128, recv=ctypes.c_void_p((1 << 20) + 4)) == 2


def test_dispatch_combine_argument_validation(lib):
    assert lib.ep_dispatch(FAKE, 4, 100, 8, FAKE, FAKE, 32, None, None) == 2        # H % 8
    assert lib.ep_dispatch(FAKE, 4, 64, 0, FAKE, FAKE, 32, None, None) == 1          # k
    assert lib.ep_dispatch(None, 4, 64, 8, FAKE, FAKE, 32, None, None) == 1
    assert lib.ep_dispatch(ctypes.c_void_p((1 << 20) + 8), 4, 64, 8, FAKE, FAKE, 32, None, None) == 2
    assert lib.ep_dispatch(FAKE, 0, 64, 8, FAKE, FAKE, 32, None, None) == 0          # T == 0: no-op
    assert lib.ep_dispatch_fp8(FAKE, 4, 64, 8, FAKE, FAKE, FAKE, 32, None, None) == 2  # H % 128
    assert lib.ep_dispatch_fp8(FAKE, 4, 256, 8, FAKE, FAKE, ctypes.c_void_p((1 << 20) + 2), 32,
                               None, None) == 2
    assert lib.ep_combine(FAKE, FAKE, FAKE, 4, 64, 8, 32, None, None, None) == 1      # out NULL
    assert lib.ep_combine(FAKE, FAKE, FAKE, 4, 60, 8, 32, FAKE, None, None) == 2
    assert lib.ep_combine(FAKE, FAKE, FAKE, -1, 64, 8, 32, FAKE, None, None) == 1
    assert lib.ep_status_read(None, None, None) == 1


def test_combine_fp8_argument_validation(lib):
    # (y_q, y_scale, topk_w, dst_row, T, H, k, rows, out, status, stream)
    assert lib.ep_combine_fp8(FAKE, FAKE, FAKE, FAKE, 4, 64, 8, 32, FAKE, None, None) == 2    # H % 128
    assert lib.ep_combine_fp8(FAKE, FAKE, FAKE, FAKE, 4, 256, 0, 32, FAKE, None, None) == 1   # k
    assert lib.ep_combine_fp8(FAKE, FAKE, FAKE, FAKE, 4, 256, 8, 32, None, None, None) == 1   # out NULL
    assert lib.ep_combine_fp8(None, FAKE, FAKE, FAKE, 4, 256, 8, 32, FAKE, None, None) == 1   # codes NULL
    assert lib.ep_combine_fp8(FAKE, None, FAKE, FAKE, 4, 256, 8, 32, FAKE, None, None) == 1   # scales NULL
    assert lib.ep_combine_fp8(ctypes.c_void_p((1 << 20) + 8), FAKE, FAKE, FAKE, 4, 256, 8, 32, FAKE,
                              None, None) == 2                                                 # codes not 16-B aligned
    assert lib.ep_combine_fp8(FAKE, ctypes.c_void_p((1 << 20) + 2), FAKE, FAKE, 4, 256, 8, 32, FAKE,
                              None, None) == 2                                                 # scales not 4-B aligned
    assert lib.ep_combine_fp8(FAKE, FAKE, FAKE, FAKE, 0, 256, 8, 32, FAKE, None, None) == 0   # T == 0: no-op


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from combine_ep_layout_02_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.load()


def test_pipeline_argument_validation(lib):
    assert lib.ep_pipeline_create(0, ctypes.byref(ctypes.c_void_p())) == 1
    assert lib.ep_pipeline_create(5000, ctypes.byref(ctypes.c_void_p())) == 1
    assert lib.ep_pipeline_destroy(None) == 1
    args = [FAKE] * 4 + [16, 64, 8, 256, 16, 0, 0, 4] + [FAKE] * 4 + [None, None] + \
        [32, None, FAKE] + [FAKE] * 3 + [None, None, FAKE, 1 << 20]
    assert lib.ep_roundtrip_host(None, None, *args) == 1     # no handle


def test_aligned_layout_argument_validation(lib):
    def call(T=16, k=8, E=256, R=16, align=8, ws=FAKE):
        return lib.ep_layout_aligned(FAKE, T, k, E, R, align, FAKE, FAKE, FAKE, None, None, ws,
                                     1 << 30, None)
    assert call(align=0) == 1
    assert call(align=-3) == 1
    assert call(T=1 << 27, k=8, E=1024, R=1, align=1 << 21) == 1   # padded rows >= 2^31
    assert call(E=255) == 1
    assert call(ws=None) == 3


def test_two_stage_argument_validation(lib):
    assert lib.ep_rank_layout_workspace_bytes(0, 8, 256, 16) == 0
    assert lib.ep_rank_layout_workspace_bytes(65536, 8, 256, 16) >= 65536 * 8 * 4
    assert lib.ep_rank_layout(FAKE, 16, 8, 255, 16, FAKE, FAKE, FAKE, FAKE, FAKE, 128, None, FAKE,
                              1 << 30, None) == 1   # E % R
    assert lib.ep_rank_layout(FAKE, 16, 8, 256, 16, FAKE, FAKE, FAKE, FAKE, FAKE, 128, None, None,
                              0, None) == 3         # workspace
    assert lib.ep_expand(FAKE, FAKE, 0, 10, FAKE, FAKE, FAKE, 4, 64, 8, FAKE, 32, None, None) == 1
    assert lib.ep_expand(FAKE, FAKE, 4, 10, FAKE, FAKE, FAKE, 4, 60, 8, FAKE, 32, None, None) == 2
    assert lib.ep_combine_partial(FAKE, 32, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 4, 64, 8, None,
                                  None, None) == 1  # partial NULL
    assert lib.ep_combine_reduce(FAKE, 10, FAKE, 4, 64, 8, None, None, None) == 1


def test_expand_fp8_argument_validation(lib):
    assert lib.ep_expand_fp8(FAKE, FAKE, FAKE, 4, 10, FAKE, FAKE, FAKE, 4, 64, 8, FAKE, FAKE, 32,
                             None, None) == 2       # H % 128
    assert lib.ep_expand_fp8(FAKE, FAKE, FAKE, 0, 10, FAKE, FAKE, FAKE, 4, 128, 8, FAKE, FAKE, 32,
                             None, None) == 1       # R < 1
    assert lib.ep_expand_fp8(None, FAKE, FAKE, 4, 10, FAKE, FAKE, FAKE, 4, 128, 8, FAKE, FAKE, 32,
                             None, None) == 1
