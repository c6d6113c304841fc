"""Seeded synthetic workloads for MoE layout / dispatch / combine.

This module only draws inputs: hidden states, top-k routes, top-k weights,
per-expert scales and independent expert outputs.  It holds none of the
method's arithmetic (no layout, no dispatch, no quantisation, no combine) and
serves both the CUDA path and the CPU oracle, which never import each other.

The five named workloads follow the shapes the pages measure:
  * afdEP-comm validation record, "setup": one NVLink domain of 4 GPUs, BF16,
    hidden 2048, top-8 of 128 experts, capacity 2048   -> ``small``, ``masked``
  * awsome-distributed-ai PR #1238, Decode-like profile: 128 tokens per rank,
    EP16, hidden 7168, top-8 of 256                     -> ``decode_fp8``
  * the same PR, Prefill-like profile: 4096 tokens per rank, EP16 / EP32,
    layout included                                     -> ``prefill``, ``prefill_fp8``
Routes are uniform or Zipf-skewed instead of the PR's perfectly balanced
``(t*17 + j*31 + seed) mod 256`` route, which is kept as an extra test input
(``balanced_route``).  A sixth workload, ``prefill_grouped``, limits each
token to 4 of 8 virtual ranks (group-limited routing, the reason DeepEP-style
dispatch sends one copy per destination and expands it there), so that the
two-stage path has real per-rank deduplication to exploit.

Seeds: workload ``i`` (1-based, in the order above) uses seed ``0xEB00 + i``;
each quantity has its own sub-stream.  Random draws use ``torch.Generator``
on the requested device, so the same seed gives the same values on the same
device type and PyTorch build; both sides of every comparison always receive
the very same tensors.
"""
from dataclasses import dataclass, field, replace
import hashlib

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens
    H: int                 # hidden size
    E: int                 # experts
    k: int                 # top-k
    R: int                 # virtual ranks (a grouping of experts only)
    kind: str              # "contiguous" | "masked"
    capacity: int          # rows per expert in the masked layout (0 for contiguous)
    payload: str           # "bf16" | "fp8"
    route: str             # "uniform" | "zipf" | "balanced" | "grouped"
    zipf_s: float = 0.0
    groups_per_token: int = 0   # "grouped": virtual ranks a token's experts may span
    outlier_frac: float = 0.0   # fraction of channels scaled x100
    expert_out: str = "independent"  # "independent" | "recv" | "scaled_recv"
    seed: int = 0
    notes: str = field(default="", compare=False)

    @property
    def rows(self):
        """Rows of the dispatch buffer."""
        return self.T * self.k if self.kind == "contiguous" else self.E * self.capacity

    def logical_bytes(self):
        """Useful payload per dispatch+combine call: each (token, expert)
        assignment counted once; FP8 adds a 4-byte scale per 128 channels."""
        n = self.T * self.k
        disp = n * (self.H + 4 * (self.H // 128)) if self.payload == "fp8" else n * self.H * 2
        comb = n * self.H * 2
        return disp, comb

    def scaled(self, T=None, H=None, capacity=None, **kw):
        """A smaller copy of the same workload (same distributions)."""
        return replace(self, T=self.T if T is None else T, H=self.H if H is None else H,
                       capacity=self.capacity if capacity is None else capacity, **kw)


WORKLOADS = {
    "small": Workload("small", T=128, H=2048, E=128, k=8, R=4, kind="contiguous", capacity=0,
                      payload="bf16", route="uniform", expert_out="scaled_recv", seed=0xEB01,
                      notes="4 virtual ranks x 32 experts; y = dispatched rows x per-expert U(0.5,1.5)"),
    "masked": Workload("masked", T=2048, H=2048, E=128, k=8, R=4, kind="masked", capacity=2048,
                       payload="bf16", route="uniform", seed=0xEB02,
                       notes="masked [128, 2048, 2048]; independent N(0,1) expert outputs"),
    "decode_fp8": Workload("decode_fp8", T=2048, H=7168, E=256, k=8, R=16, kind="masked",
                           capacity=2048, payload="fp8", route="uniform", seed=0xEB03,
                           notes="16 virtual ranks x 128 tokens; FP8 dispatch; BF16 combine"),
    "prefill": Workload("prefill", T=65536, H=7168, E=256, k=8, R=16, kind="contiguous",
                        capacity=0, payload="bf16", route="zipf", zipf_s=1.0,
                        expert_out="recv", seed=0xEB04,
                        notes="16 virtual ranks x 4096 tokens; Zipf(1.0); combine of the dispatched rows"),
    "prefill_fp8": Workload("prefill_fp8", T=131072, H=7168, E=256, k=8, R=32,
                            kind="contiguous", capacity=0, payload="fp8", route="zipf",
                            zipf_s=1.2, outlier_frac=0.01, seed=0xEB05,
                            notes="32 virtual ranks x 4096 tokens; Zipf(1.2); 1% outlier channels"),
    "prefill_grouped": Workload("prefill_grouped", T=65536, H=7168, E=256, k=8, R=8,
                                kind="contiguous", capacity=0, payload="bf16", route="grouped",
                                groups_per_token=4, expert_out="recv", seed=0xEB06,
                                notes="8 virtual ranks x 32 experts; each token's 8 experts "
                                      "within 4 ranks (at least 2 pairs per rank copy)"),
}

_STREAMS = {"x": 1, "route": 2, "logits": 3, "y": 4, "scale": 5, "outliers": 6,
            "y_q": 7, "y_scale": 8}


def _gen(seed, stream, device):
    g = torch.Generator(device=device)
    g.manual_seed((seed * 0x9E3779B1 + _STREAMS[stream] * 0x85EBCA77) & 0x7FFFFFFFFFFFFFFF)
    return g


def hidden_states(wl, device="cpu", chunk_rows=8192):
    """x [T, H] bf16: N(0,1) rounded to bf16; with ``outlier_frac`` > 0 a fixed
    set of channels (chosen once per seed) holds bf16(100 * z) instead."""
    g = _gen(wl.seed, "x", device)
    x = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=device)
    cols = None
    if wl.outlier_frac > 0:
        n_out = int(round(wl.outlier_frac * wl.H))
        go = _gen(wl.seed, "outliers", "cpu")
        cols = torch.randperm(wl.H, generator=go)[:n_out].sort().values.to(device)
    for r0 in range(0, wl.T, chunk_rows):
        r1 = min(wl.T, r0 + chunk_rows)
        z = torch.randn(r1 - r0, wl.H, generator=g, device=device, dtype=torch.float32)
        if cols is not None:
            z[:, cols] *= 100.0
        x[r0:r1] = z.to(torch.bfloat16)
    return x


def balanced_route(T, k, E, seed=0):
    """The perfectly balanced route printed in PR #1238's methodology review:
    expert (t*17 + j*31 + seed) mod E.  With E = 256 and 31 coprime to it the
    k ids of a token are distinct and every expert carries T*k/E pairs when T
    is a multiple of E."""
    t = torch.arange(T, dtype=torch.int64).view(T, 1)
    j = torch.arange(k, dtype=torch.int64).view(1, k)
    return ((t * 17 + j * 31 + seed) % E).to(torch.int32)


def route(wl, device="cpu", chunk_rows=16384):
    """topk_idx [T, k] int32: k distinct experts per token.

    uniform: a uniformly random k-subset in random order (top-k of i.i.d.
    uniform keys).  zipf: successive draws without replacement with expert
    popularity p_e proportional to (e+1)^-s (expert 0 hottest), via the
    Gumbel-top-k construction: top-k of log p_e + Gumbel noise.  grouped:
    first a uniformly random set of ``groups_per_token`` of the R virtual
    ranks (top of i.i.d. uniform rank keys), then a uniformly random k-subset
    of those ranks' experts (their uniform keys; the other experts' keys are
    set below every draw)."""
    if wl.route == "balanced":
        return balanced_route(wl.T, wl.k, wl.E, wl.seed).to(device)
    g = _gen(wl.seed, "route", device)
    out = torch.empty(wl.T, wl.k, dtype=torch.int32, device=device)
    if wl.route == "zipf":
        logp = -wl.zipf_s * torch.log(torch.arange(1, wl.E + 1, device=device, dtype=torch.float64))
        logp = logp.to(torch.float32)
    for r0 in range(0, wl.T, chunk_rows):
        r1 = min(wl.T, r0 + chunk_rows)
        u = torch.rand(r1 - r0, wl.E, generator=g, device=device, dtype=torch.float32)
        if wl.route == "uniform":
            keys = u
        elif wl.route == "grouped":
            per = wl.E // wl.R
            if wl.groups_per_token * per < wl.k:
                raise ValueError("grouped route: the chosen ranks hold fewer than k experts")
            ru = torch.rand(r1 - r0, wl.R, generator=g, device=device, dtype=torch.float32)
            chosen = torch.zeros(r1 - r0, wl.R, dtype=torch.bool, device=device)
            chosen.scatter_(1, torch.topk(ru, wl.groups_per_token, dim=1).indices, True)
            keys = torch.where(chosen.repeat_interleave(per, dim=1), u, torch.full_like(u, -1.0))
        elif wl.route == "zipf":
            u = u.clamp_min(torch.finfo(torch.float32).tiny)
            keys = logp.view(1, -1) - torch.log(-torch.log(u))
        else:
            raise ValueError(wl.route)
        out[r0:r1] = torch.topk(keys, wl.k, dim=1, largest=True, sorted=True).indices.to(torch.int32)
    return out


def topk_weights(wl, device="cpu"):
    """topk_w [T, k] float32: softmax over the k chosen of N(0,1) logits."""
    g = _gen(wl.seed, "logits", device)
    logits = torch.randn(wl.T, wl.k, generator=g, device=device, dtype=torch.float32)
    return torch.softmax(logits, dim=1)


def expert_scales(wl, device="cpu"):
    """Per-expert fp32 scale U(0.5, 1.5) used to make ``scaled_recv`` outputs."""
    g = _gen(wl.seed, "scale", device)
    return 0.5 + torch.rand(wl.E, generator=g, device=device, dtype=torch.float32)


def independent_expert_outputs(wl, device="cpu", chunk_rows=8192):
    """y [rows, H] bf16 with i.i.d. N(0,1) entries (rounded to bf16)."""
    g = _gen(wl.seed, "y", device)
    y = torch.empty(wl.rows, wl.H, dtype=torch.bfloat16, device=device)
    for r0 in range(0, wl.rows, chunk_rows):
        r1 = min(wl.rows, r0 + chunk_rows)
        y[r0:r1] = torch.randn(r1 - r0, wl.H, generator=g, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
    return y


def fp8_expert_outputs(wl, device="cpu", chunk_rows=8192):
    """Expert outputs already in the FP8 payload encoding, for the FP8
    combine: codes y_q [rows, H] uint8 drawn uniformly from the 254 finite
    e4m3 codes (0x7F and 0xFF, the NaN codes, excluded), and one float32
    scale per row and 128 channels, y_scale [rows, H/128] = (2 + U(0,2)) / 448
    (the scale of a block whose largest magnitude is 2..4, as N(0,1) rows
    give).  Plain random draws: no quantisation happens here."""
    g = _gen(wl.seed, "y_q", device)
    gs = _gen(wl.seed, "y_scale", device)
    q = torch.empty(wl.rows, wl.H, dtype=torch.uint8, device=device)
    for r0 in range(0, wl.rows, chunk_rows):
        r1 = min(wl.rows, r0 + chunk_rows)
        c = torch.randint(0, 254, (r1 - r0, wl.H), generator=g, device=device, dtype=torch.int32)
        q[r0:r1] = (c + (c >= 127).to(torch.int32)).to(torch.uint8)   # skip 0x7F
    sc = (2.0 + 2.0 * torch.rand(wl.rows, wl.H // 128, generator=gs, device=device,
                                 dtype=torch.float32)) / 448.0
    return q, sc


def scale_rows(recv, row_expert, scales):
    """bf16(float(recv[row]) * scales[row_expert[row]]); rows with
    row_expert < 0 are left as they are.  Builds the ``scaled_recv`` expert
    outputs from a dispatched buffer."""
    y = recv.clone()
    valid = row_expert >= 0
    s = scales[row_expert.clamp_min(0).long()]
    y[valid] = (recv[valid].float() * s[valid].view(-1, 1)).to(torch.bfloat16)
    return y


def sha256_of(*tensors):
    """SHA-256 over the raw bytes of host copies of the given tensors."""
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()


def bf16_bits(t):
    """View a bf16 tensor as its uint16 bit patterns (numpy, host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
