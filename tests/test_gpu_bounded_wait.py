"""The library's only device-side wait (the mbarrier wait of the optional
bulk-copy dispatch) is bounded: on a barrier that nothing completes it gives
up after its limit, raises EP_FLAG_TIMEOUT in the status word and returns,
and the context stays usable.  The kernel that runs it is built here from
tests/selftest/bounded_wait.cu against the library's device header."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import build as B
from combine_ep_layout_02_gb300 import workloads as W

from gpu_helpers import DEV

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def selftest_lib():
    import __graft_entry__
    __graft_entry__.build()
    out = tempfile.mkdtemp(prefix="ep_selftest_")
    lib = os.path.join(out, "libep_selftest.so")
    cmd = [B._nvcc()] + B.NVCC_FLAGS + ["-shared", os.path.join(HERE, "selftest", "bounded_wait.cu"),
                                        "-o", lib]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    so = ctypes.CDLL(lib)
    so.selftest_bounded_wait.restype = ctypes.c_int
    so.selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return so


def test_bounded_wait_gives_up_flags_and_leaves_context_usable(selftest_lib):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    elapsed = torch.zeros(1, dtype=torch.int64, device=DEV)
    stream = torch.cuda.current_stream(DEV)
    rc = selftest_lib.selftest_bounded_wait(status.data_ptr(), elapsed.data_ptr(), stream.cuda_stream)
    assert rc == 0
    torch.cuda.synchronize(DEV)
    assert ep.status_read(status) == ep.EP_FLAG_TIMEOUT
    ns = int(elapsed.item())
    assert 1.9e9 <= ns <= 10e9            # the 2 s limit, then return
    # the context is intact: the whole path still matches the oracle
    wl = W.WORKLOADS["small"].scaled(T=64, H=256)
    x, idx = W.hidden_states(wl, device=DEV), W.route(wl, device=DEV)
    lay = ep.layout(idx, wl.E, wl.R)
    recv = ep.dispatch(x, lay.dst_row, wl.rows, status=lay.status)
    ref = oracle.dispatch_bf16(W.bf16_bits(x), lay.dst_row.cpu().numpy(), wl.rows)
    assert np.array_equal(W.bf16_bits(recv), ref)
    assert ep.status_read(lay.status) == 0
