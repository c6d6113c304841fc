"""Shared helpers for the GPU parity tests: draw a workload, run the CUDA path
through the C ABI and the oracle on the same inputs, and compare."""
import numpy as np
import torch

import oracle
from combine_ep_layout_02_gb300 import workloads as W

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

# Combine tolerance (stated per element): |gpu - ref| <= 2^-7 * max(|ref|, 2^-12 * S)
# with ref the fp64 sum and S = sum_j |w_j y_j|.  The fp32-FMA + bf16-RNE path
# errs by at most 2^-8 |ref| (one bf16 rounding) + k * 2^-24 * S (k fp32
# roundings), well inside this bound for k <= 32.
COMBINE_REL = 2.0 ** -7
COMBINE_FLOOR = 2.0 ** -12


def oracle_kind(wl):
    return oracle.LAYOUT_MASKED if wl.kind == "masked" else oracle.LAYOUT_CONTIGUOUS


def draw(wl, device):
    """Inputs of a workload on `device` (the route and weights also on host)."""
    x = W.hidden_states(wl, device=device)
    idx = W.route(wl, device=device)
    w = W.topk_weights(wl, device=device)
    return x, idx, w


def bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def check_combine(out_bits, ref, absum, what=""):
    got = bf16_to_f64(out_bits)
    denom = np.maximum(np.abs(ref), COMBINE_FLOOR * absum)
    err = np.abs(got - ref)
    bad = err > COMBINE_REL * denom
    assert not bad.any(), "%s: %d elements outside 2^-7 (max rel %.3g)" % (
        what, int(bad.sum()), float((err / np.maximum(denom, 1e-300)).max()))
    return float((err / np.maximum(denom, 1e-300)).max())


def rows_of(dst_row):
    d = np.asarray(dst_row).reshape(-1)
    return d[d >= 0]
