"""ep_layout_static_ws: the routing layout for callers that cannot allocate
device memory (a plug-in whose host application owns all device memory, a
loop that must not allocate once running).  Its scratch is a fixed array in
the library's own device memory; it must give exactly what ep_layout gives
with a caller-provided workspace, call after call.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import binding
from combine_ep_layout_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _same(a, b):
    for name in ("expert_counts", "expert_offsets", "dst_row", "rank_token_counts", "status"):
        ta, tb = getattr(a, name), getattr(b, name)
        assert torch.equal(ta, tb), name


def test_static_scratch_layout_matches_workspace_layout_twice():
    dev = torch.device("cuda:0")
    # Both chunked-path cases use the scratch; the second has fewer chunks and
    # fewer columns (72 x 32 against 288 x 1024 int32 counters), so the first
    # call's counters are still in the array at other positions and any entry
    # the second call failed to rewrite would be read stale.  decode_fp8 takes
    # the one-launch path, which needs no scratch.
    cases = [W.WORKLOADS["prefill_fp8"],
             W.WORKLOADS["prefill"].scaled(T=4096, E=64, R=8),
             W.WORKLOADS["decode_fp8"]]
    for wl in cases:
        idx = W.route(wl, device=dev)
        for _ in range(2):                                            # two calls in a row
            ref = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
            got = binding.layout_static_ws(idx, wl.E, wl.R, wl.kind, wl.capacity)
            torch.cuda.synchronize()
            _same(ref, got)
            assert ep.status_read(got.status) == 0


def test_static_scratch_rejects_sizes_beyond_its_limit():
    lib = binding.load()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the call is rejected on the host
    T, k, E, R = 1 << 20, 8, 1024, 1024          # needs 2048 columns x 2048 chunks x 4 B = 16 MiB
    need = lib.ep_layout_workspace_bytes(T, k, E, R, 1)
    assert need > (2 << 20)
    rc = lib.ep_layout_static_ws(fake, T, k, E, R, 0, 0, fake, fake, fake, fake, None, None)
    assert rc == binding.EP_ERR_WORKSPACE


def test_static_scratch_reports_bad_arguments_like_ep_layout():
    lib = binding.load()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the call is rejected on the host
    T, k, E, R = 1 << 20, 8, 2048, 1024          # E above EP_MAX_EXPERTS, and too large for the array
    rc = lib.ep_layout_static_ws(fake, T, k, E, R, 0, 0, fake, fake, fake, fake, None, None)
    assert rc == binding.EP_ERR_INVALID_ARG
    rc = lib.ep_layout(fake, T, k, E, R, 0, 0, fake, fake, fake, fake, None, fake, 1 << 30, None)
    assert rc == binding.EP_ERR_INVALID_ARG
