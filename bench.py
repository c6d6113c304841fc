"""Benchmark: one step = routing layout + dispatch + combine on one batch.

Default workload: the Prefill-like shape (65,536 tokens = 16 virtual ranks x
4,096, hidden 7168, 256 experts, top-8 with Zipf(1.0) popularity, contiguous
layout, BF16 dispatch and combine; combine runs over the dispatched rows,
i.e. identity experts).  Inputs are generated on the device before timing
and are far larger than L2 (x 0.94 GB, dispatch buffer 7.5 GB), so no L2
flush is inserted between steps.  Workloads whose working set is under four
times the L2 size get a 2 x L2 buffer written between steps, outside the
timed events (one event pair per step).

Prints ONE JSON line (rank 0).  `value` is the logical throughput: the
useful payload of one dispatch plus one combine (each (token, expert)
assignment counted once; BF16 T*k*H*2 each way, FP8 dispatch T*k*(H + H/32))
divided by the device time of the whole step, summed over all ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from combine_ep_layout_02_gb300 import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
LEAD_CYCLES = 1 << 20   # GPU spin (about 0.5 ms) queued ahead of each individually timed step
METRIC = "dispatch+combine logical GB/s per call (layout+dispatch+combine, one event pair)"
KERNEL_SOURCES = {
    "layout": "combine_ep_layout_02_gb300/csrc/ep_layout.cu",
    "dispatch": "combine_ep_layout_02_gb300/csrc/ep_dispatch.cu",
    "dispatch_fp8": "combine_ep_layout_02_gb300/csrc/ep_dispatch_fp8.cu",
    "combine": "combine_ep_layout_02_gb300/csrc/ep_combine.cu",
    "combine_fp8": "combine_ep_layout_02_gb300/csrc/ep_combine_fp8.cu",
}


# ----------------------------------------------------------------------------- helpers

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="prefill", choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=None,
                    help="override the workload's seed (inputs are drawn from it)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="scale the workload to this many tokens (profiling captures)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--chunk-tokens", type=int, default=2048,
                    help="token chunk of the host-buffer executor (e2e)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the timed oracle sample (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--path", default="direct", choices=["direct", "two_stage"],
                    help="direct: layout, dispatch, combine; two_stage: one copy per (token, rank), "
                         "expansion into experts, rank-local partial combine, final reduce")
    ap.add_argument("--l2-flush", action="store_true",
                    help="flush L2 between steps even when the working set is far larger than L2")
    ap.add_argument("--no-l2-flush", action="store_true",
                    help="never flush L2 (warm-L2 numbers for working sets that fit in L2)")
    ap.add_argument("--layout-only", action="store_true",
                    help="time only the routing layout (20 calls captured in one CUDA graph)")
    ap.add_argument("--fused", action="store_true",
                    help="layout + dispatch through ep_layout_dispatch (one launch up to 128 tokens)")
    ap.add_argument("--combine", default="bf16", choices=["bf16", "fp8"],
                    help="fp8: expert outputs held as e4m3 codes + per-128-channel scales, "
                         "combined by ep_combine_fp8")
    ap.add_argument("--graph", action="store_true",
                    help="replay the step as one captured CUDA graph (launch-bound small shapes)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def max_over_ranks(value, world, device=None):
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world, device=None):
    if world > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate_value(logical_bytes_per_step, steps, max_seconds, world):
    """Whole-job logical GB/s: every rank processes its own step each time."""
    return world * logical_bytes_per_step * steps / max_seconds / 1e9


def provenance(dev, idx, w, x):
    """Versions, git revision and input hashes recorded with every result."""
    info = {"torch": torch.__version__, "cuda": torch.version.cuda,
            "device": torch.cuda.get_device_name(dev)}
    try:
        info["git"] = subprocess.run(["git", "rev-parse", "--short", "HEAD"], cwd=ROOT,
                                     capture_output=True, text=True, timeout=10).stdout.strip() or None
    except (OSError, subprocess.TimeoutExpired):
        info["git"] = None
    try:
        info["driver"] = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                                        capture_output=True, text=True, timeout=10).stdout.split()[0]
    except (OSError, subprocess.TimeoutExpired, IndexError):
        info["driver"] = None
    try:
        info["nvcc"] = subprocess.run(["nvcc", "--version"], capture_output=True, text=True,
                                      timeout=10).stdout.strip().splitlines()[-1]
    except (OSError, subprocess.TimeoutExpired, IndexError):
        info["nvcc"] = None
    try:  # digest of the CUDA sources and flags the library was built from
        with open(os.path.join(ROOT, "combine_ep_layout_02_gb300", "_build", "stamp")) as f:
            info["library_source_digest"] = f.read().strip()[:16]
    except OSError:
        info["library_source_digest"] = None
    info["sha256_route_weights"] = W.sha256_of(idx, w)
    info["sha256_x_first_64MB"] = W.sha256_of(x.view(-1)[: (64 << 20) // 2])
    return info


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        for key in ("hbm_gbs", "hbm_copy_gbs", "hbm_GBs"):
            if key in peaks and peaks[key]:
                return float(peaks[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def source_hash(rel):
    """Hash of a kernel's source file and the device helpers it includes."""
    h = hashlib.sha256()
    for path in (rel, "combine_ep_layout_02_gb300/csrc/ep_internal.cuh"):
        with open(os.path.join(ROOT, path), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, wl):
    """DRAM bytes per launch of `kernel` on workload `wl`, from the committed
    ncu capture (profiles/traffic.json), or None.  Captures are taken on a
    smaller case of the same shape (same H and k, fewer tokens) and scaled
    by the token count: a launch's reads and writes are per-token rows.  Only
    used while the kernel's source is the one the capture was taken on."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            tab = json.load(f)
    except (OSError, ValueError):
        return None
    ent = tab.get("kernels", {}).get(kernel)
    if not ent or kernel not in KERNEL_SOURCES:
        return None
    if ent.get("source_sha256_16") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    if ent.get("H") != wl.H or ent.get("k") != wl.k or not ent.get("tokens"):
        return None
    lo, hi = ent.get("valid_tokens", [0, 1 << 62])  # the token range that runs the captured instance
    if not lo <= wl.T <= hi:
        return None
    per_launch = ent["dram_bytes_read"] + ent["dram_bytes_write"]
    return {"bytes": per_launch * wl.T / ent["tokens"], "captured_tokens": ent["tokens"],
            "captured_workload": ent.get("workload"), "scale": wl.T / ent["tokens"]}


def algorithmic_bytes(wl, path="direct", fused=False, rank_rows=0, combine="bf16"):
    """Algorithmic HBM bytes of each timed part of a step: what the method
    must read and write once.  Direct path: the layout reads the ids and
    writes dst_row; dispatch reads x and writes k rows per token (FP8: codes
    plus a 4-byte scale per 128 channels); combine reads k rows and writes
    one per token (FP8 expert outputs: codes plus a 4-byte scale per 128
    channels).  `fused`: layout and dispatch timed as one call.  Two-stage
    path (`rank_rows` rank rows filled): the copy to ranks plus the expansion,
    and the rank-local partials plus the final reduce."""
    Tk = wl.T * wl.k
    row = wl.H + wl.H // 32 if wl.payload == "fp8" else wl.H * 2  # bytes of a dispatched row
    if path == "two_stage":
        nr = rank_rows
        return {
            "layout": 2 * Tk * 4 + Tk * 4 + 2 * Tk * 4 + nr * 4,
            "dispatch": (wl.T * wl.H * 2 + nr * row + Tk * 4)               # copy to ranks
                        + (nr * row + Tk * row + 2 * Tk * 4),               # expansion
            "combine": (Tk * wl.H * 2 + nr * wl.H * 2 + Tk * 12 + nr * 4)   # rank-local partials
                       + (nr * wl.H * 2 + wl.T * wl.H * 2 + Tk * 4),       # final reduce
        }
    in_row = wl.H + wl.H // 32 if combine == "fp8" else wl.H * 2  # bytes of an expert-output row
    alg = {"layout": 2 * Tk * 4,
           "dispatch": wl.T * wl.H * 2 + Tk * row + Tk * 4,
           "combine": Tk * in_row + wl.T * wl.H * 2 + Tk * 8}
    if fused:
        return {"layout_dispatch": alg["layout"] + alg["dispatch"], "combine": alg["combine"]}
    return alg


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ident = vis.split(",")[device_index] if vis else str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, IndexError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle timing

def host_cpu():
    """Cores and model of the host CPU (for the CPU-baseline record)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.TimeoutExpired):
        pass
    import platform
    return {"host_cores": os.cpu_count(), "cpu_model": model or platform.processor() or None,
            "machine": platform.machine()}


def oracle_sample(wl, x_host_bits, idx_host, w_host, tokens, seconds, combine="bf16"):
    """Time the CPU oracle (layout + dispatch + combine of the first `tokens`
    tokens) in repeated passes until `seconds` elapse; return logical GB/s and
    details.  The expert outputs combined are the dispatched BF16 rows, built
    once outside the timed passes (FP8 combine: seeded codes and scales)."""
    import oracle
    T = min(tokens, wl.T)
    idx = idx_host[:T]
    xb = x_host_bits[:T]
    w = w_host[:T]
    kind = oracle.LAYOUT_MASKED if wl.kind == "masked" else oracle.LAYOUT_CONTIGUOUS
    cap = min(wl.capacity, T) if wl.kind == "masked" else 0
    rows = T * wl.k if wl.kind == "contiguous" else wl.E * cap
    sub = wl.scaled(T=T, capacity=cap or None)
    disp_b, comb_b = sub.logical_bytes()
    lay0 = oracle.layout(idx, wl.E, wl.R, kind, cap)
    y = oracle.dispatch_bf16(xb, lay0["dst_row"], rows)
    if combine == "fp8":
        yq, ys = W.fp8_expert_outputs(sub)
        yq, ys = yq.numpy(), ys.numpy()
    passes, t_lay, t_disp, t_comb = 0, 0.0, 0.0, 0.0
    t0 = time.perf_counter()
    while True:
        a = time.perf_counter()
        lay = oracle.layout(idx, wl.E, wl.R, kind, cap)
        b = time.perf_counter()
        if wl.payload == "fp8":
            oracle.dispatch_fp8(xb, lay["dst_row"], rows)
        else:
            oracle.dispatch_bf16(xb, lay["dst_row"], rows)
        c = time.perf_counter()
        if combine == "fp8":
            oracle.combine_fp8_f64(yq, ys, w, lay["dst_row"])
        else:
            oracle.combine_f64(y, w, lay["dst_row"])
        d = time.perf_counter()
        passes += 1
        t_lay, t_disp, t_comb = t_lay + b - a, t_disp + c - b, t_comb + d - c
        if d - t0 >= seconds:
            break
    total = t_lay + t_disp + t_comb
    return {
        "value": passes * (disp_b + comb_b) / total / 1e9,
        "unit": "GB/s",
        "cores": 1,
        "kind": "oracle",
        "sample": "%d passes of layout+dispatch+combine over the first %d of %d tokens "
                  "(%.1f s, single-threaded C; time.perf_counter around each step)" % (
                      passes, T, wl.T, total),
        "us_per_call": total / passes * 1e6,
        "us_layout": t_lay / passes * 1e6,
        "us_dispatch": t_disp / passes * 1e6,
        "us_combine": t_comb / passes * 1e6,
        **host_cpu(),
    }


# ----------------------------------------------------------------------------- arms

def run_reference(args, rank, world):
    """--impl reference: the oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    from oracle import build as oracle_build
    oracle_build.build()
    wl = W.WORKLOADS[args.workload]
    tokens = 512
    sub = wl.scaled(T=tokens)
    x = W.bf16_bits(W.hidden_states(sub))
    idx = W.route(sub).numpy()
    w = W.topk_weights(sub).numpy()
    for _ in range(args.warmup):
        oracle_sample(wl, x, idx, w, tokens, 0.0, args.combine)
    vals, secs = [], 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = oracle_sample(wl, x, idx, w, tokens, 0.0, args.combine)
        vals.append(r["us_per_call"])
    secs = time.perf_counter() - t0
    disp_b, comb_b = sub.logical_bytes()
    us = float(np.mean(vals))
    value = (disp_b + comb_b) / (us * 1e-6) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.payload,
        "data": "synthetic",
        "config": {"workload": wl.name, "T_sampled": tokens, "T": wl.T, "H": wl.H, "E": wl.E,
                   "k": wl.k, "R": wl.R, "layout": wl.kind, "payload": wl.payload,
                   "route": wl.route, "zipf_s": wl.zipf_s, "combine": args.combine},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "each step: layout+dispatch+combine of the first %d of %d "
                                   "tokens (single-threaded C oracle); %.1f s total" % (
                                       tokens, wl.T, secs), **host_cpu()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_layout_only(args, rank, world, local):
    """The routing layout alone: `--steps` replays of a CUDA graph holding 20
    layout calls on the workload's route (a few MB on the device)."""
    import combine_ep_layout_02_gb300 as ep
    if not os.path.exists(ep.binding.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.scaled(T=args.tokens, capacity=min(wl.capacity, args.tokens) or None)
    idx = W.route(wl, device=dev)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    ws = torch.empty(max(16, ep.layout_workspace_bytes(wl.T, wl.k, wl.E, wl.R)), dtype=torch.uint8,
                     device=dev)
    for _ in range(max(3, args.warmup)):
        ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity, out=lay, workspace=ws)
    torch.cuda.synchronize(dev)
    calls = 20
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(calls):
            ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity, out=lay, workspace=ws)
    graph.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        graph.replay()
    b.record()
    torch.cuda.synchronize(dev)
    if ep.status_read(lay.status) != 0:
        raise SystemExit("device status flags set by the layout")
    us = a.elapsed_time(b) * 1e3 / (args.steps * calls)
    pairs = wl.T * wl.k
    if rank == 0:
        print(json.dumps({"metric": "routing layout us per call (CUDA graph of %d calls)" % calls,
                          "value": us, "unit": "us", "higher_is_better": False, "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup,
                          "config": {"workload": wl.name, "T": wl.T, "k": wl.k, "E": wl.E,
                                     "R": wl.R, "layout": wl.kind},
                          "pairs_per_us": pairs / us,
                          "launches_per_call": 1 if wl.T <= 2048 else 3}), flush=True)


def run_ours(args, rank, world, local):
    import combine_ep_layout_02_gb300 as ep
    if not os.path.exists(ep.binding.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    ep.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.scaled(T=args.tokens, capacity=min(wl.capacity, args.tokens) or None)
    if args.seed is not None:
        wl = wl.scaled(seed=args.seed)
    torch.manual_seed(0)

    # ---- inputs resident in HBM
    x = W.hidden_states(wl, device=dev)
    idx = W.route(wl, device=dev)
    w = W.topk_weights(wl, device=dev)
    lay = ep.LayoutOut(torch.empty(wl.E, dtype=torch.int32, device=dev),
                       torch.empty(wl.E + 1, dtype=torch.int32, device=dev),
                       torch.empty(wl.T, wl.k, dtype=torch.int32, device=dev),
                       torch.empty(wl.R, dtype=torch.int32, device=dev),
                       torch.zeros(1, dtype=torch.int32, device=dev))
    ws = torch.empty(max(16, ep.layout_workspace_bytes(wl.T, wl.k, wl.E, wl.R)), dtype=torch.uint8,
                     device=dev)
    if wl.payload == "fp8":
        recv_q = torch.empty(wl.rows, wl.H, dtype=torch.uint8, device=dev)
        recv_s = torch.empty(wl.rows, wl.H // 128, dtype=torch.float32, device=dev)
    recv = None
    if wl.payload == "bf16" or wl.expert_out == "recv":
        recv = torch.empty(wl.rows, wl.H, dtype=torch.bfloat16, device=dev)
    y_q = y_s = None
    if args.combine == "fp8":
        if args.path != "direct":
            raise SystemExit("--combine fp8 applies to the direct path")
        # expert outputs in the FP8 payload encoding: independent draws of
        # codes and per-128-channel scales (no bf16 expert outputs exist)
        y_q, y_s = W.fp8_expert_outputs(wl, device=dev)
        y = None
    elif wl.expert_out == "recv":
        y = recv
    elif wl.expert_out == "independent":
        y = W.independent_expert_outputs(wl, device=dev)
    else:  # scaled_recv: expert outputs = dispatched rows x per-expert scale
        lay0 = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
        r0 = ep.dispatch(x, lay0.dst_row, wl.rows)
        row_expert = torch.full((wl.rows,), -1, dtype=torch.int64, device=dev)
        row_expert[lay0.dst_row.view(-1).long()] = idx.view(-1).long()
        y = W.scale_rows(r0, row_expert, W.expert_scales(wl, device=dev))
        del r0, lay0
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    if args.fused and args.path != "direct":
        raise SystemExit("--fused applies to the direct path")
    if args.path == "two_stage":
        cap = ep.rank_rows_bound(wl.T, wl.k, wl.R)
        rl = ep.rank_layout(idx, wl.E, wl.R)
        if wl.payload == "fp8":   # rank rows hold e4m3 codes and scales
            rank_q = torch.empty(cap, wl.H, dtype=torch.uint8, device=dev)
            rank_s = torch.empty(cap, wl.H // 128, dtype=torch.float32, device=dev)
        else:
            rank_buf = torch.empty(cap, wl.H, dtype=torch.bfloat16, device=dev)
        partial = torch.empty(cap, wl.H, dtype=torch.bfloat16, device=dev)
        rws = torch.empty(max(16, ep.load().ep_rank_layout_workspace_bytes(wl.T, wl.k, wl.E, wl.R)),
                          dtype=torch.uint8, device=dev)

    def step_two_stage(ev=None):
        if ev:
            ev[0].record(stream)
        ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity, out=lay, workspace=ws)
        ep.rank_layout(idx, wl.E, wl.R, out=rl, workspace=rws)
        if ev:
            ev[1].record(stream)
        if wl.payload == "fp8":
            ep.dispatch_fp8(x, rl.rank_dst_row, cap, recv_q=rank_q, recv_scale=rank_s,
                            status=lay.status)
            ep.expand_fp8(rank_q, rank_s, rl, lay.dst_row, wl.rows, recv_q=recv_q,
                          recv_scale=recv_s, status=lay.status)
        else:
            ep.dispatch(x, rl.rank_dst_row, cap, recv=rank_buf, status=lay.status)
            ep.expand(rank_buf, rl, lay.dst_row, wl.rows, recv=recv, status=lay.status)
        if ev:
            ev[2].record(stream)
        ep.combine_partial(y, w, lay.dst_row, rl, cap, partial=partial, status=lay.status)
        ep.combine_reduce(partial, rl, wl.T, out=out, status=lay.status)
        if ev:
            ev[3].record(stream)

    def step(ev=None):
        if args.path == "two_stage":
            return step_two_stage(ev)
        if ev:
            ev[0].record(stream)
        if args.fused:
            # one call; its time is reported under "layout" + "dispatch" together
            if wl.payload == "fp8":
                ep.layout_dispatch(x, idx, wl.E, wl.R, wl.kind, wl.capacity, wl.rows, out=lay,
                                   workspace=ws, fp8=True, recv_q=recv_q, recv_scale=recv_s)
            else:
                ep.layout_dispatch(x, idx, wl.E, wl.R, wl.kind, wl.capacity, wl.rows, out=lay,
                                   recv=recv, workspace=ws)
            if ev:
                ev[1].record(stream)
                ev[2].record(stream)
        else:
            ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity, out=lay, workspace=ws)
            if ev:
                ev[1].record(stream)
            if wl.payload == "fp8":
                ep.dispatch_fp8(x, lay.dst_row, wl.rows, recv_q=recv_q, recv_scale=recv_s,
                                status=lay.status)
            else:
                ep.dispatch(x, lay.dst_row, wl.rows, recv=recv, status=lay.status)
            if ev:
                ev[2].record(stream)
        if y_q is not None:
            ep.combine_fp8(y_q, y_s, w, lay.dst_row, out=out, status=lay.status)
        else:
            ep.combine(y, w, lay.dst_row, out=out, status=lay.status)
        if ev:
            ev[3].record(stream)

    # launches of our kernels per step: 3 layout kernels (1 when T <= 2048) +
    # dispatch + combine; the two-stage path adds the rank layout (keys, the
    # layout over keys, finish), the expansion and the final reduce
    lay_launches = 1 if wl.T <= 2048 else 3  # one launch (single block or one cluster) up to 2048 tokens
    launches_per_step = lay_launches + 2
    fused_one = args.fused and 1 <= wl.T <= 128   # layout and dispatch in one launch
    if fused_one:
        launches_per_step = 2
    if args.path == "two_stage":
        launches_per_step = 2 * lay_launches + 2 + 4

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    run_step = step
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize(dev)
        run_step = graph.replay
    if ep.status_read(lay.status) != 0:
        raise SystemExit("device status flags set during warm-up")

    # L2 policy: the working set of a step must exceed L2 by a wide margin,
    # else L2 is flushed between steps: a buffer twice its size is written and
    # then another one twice its size is read, so that L2 holds clean lines of
    # neither the inputs nor the written buffer (with the write alone, L2 is
    # left full of dirty lines that the next timed kernel has to write back:
    # measured +2.7 us on the 2,048-token masked dispatch, +6.8 us on the
    # 2,048 x 7168 FP8 dispatch)
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20)
    elem = 1 if wl.payload == "fp8" else 2
    celem = 1 if args.combine == "fp8" else 2
    touched = (x.numel() * 2 + wl.T * wl.k * wl.H * elem + wl.T * wl.k * wl.H * celem
               + out.numel() * 2)
    flush = args.l2_flush or (touched < 4 * l2_bytes and not args.no_l2_flush)
    if flush:
        flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        flush_rd = torch.ones(2 * l2_bytes // 4, dtype=torch.float32, device=dev)
        l2_note = ("L2 flushed between steps (%d MB written, then %d MB read, outside the timed "
                   "events); working set %.0f MB" % (flush_buf.numel() >> 20,
                                                     flush_rd.numel() * 4 >> 20, touched / 1e6))
    elif touched < 4 * l2_bytes:
        l2_note = "warm L2 (no flush requested); working set %.0f MB" % (touched / 1e6)
    else:
        l2_note = ("inputs larger than L2 (x %.2f GB, dispatch buffer %.2f GB, working set %.1f GB); "
                   "no flush" % (x.numel() * 2 / 1e9, wl.rows * wl.H * elem / 1e9, touched / 1e9))

    # timed region: K steps between one event pair, nothing else on the stream
    # (so consecutive kernels keep their programmatic-dependent-launch overlap);
    # with an L2 flush, one event pair per step and the flush outside it
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    time.sleep(0.3)  # let the sampler start
    def flush_l2(i):
        flush_buf.fill_(i & 0xFF)
        flush_rd.sum()

    # one event pair per step (flush or per-kernel pass): a GPU spin queued in
    # front of the step lets the host finish its launch calls before the GPU
    # reaches the step's first event, so the events time the device, not the
    # host's launch rate
    def gpu_lead():
        torch.cuda._sleep(LEAD_CYCLES)

    if flush:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2(i)
            gpu_lead()
            pairs[i][0].record(stream)
            run_step()
            pairs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        total_ms = sum(a.elapsed_time(b) for a, b in pairs)
    else:
        t_start.record(stream)
        for _ in range(args.steps):
            run_step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = t_start.elapsed_time(t_end)
    clocks = sampler.stop()
    barrier(world, dev)

    # per-kernel times: the same K steps again with an event pair around each
    # call (events between kernels, so no launch overlap at those boundaries)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        if flush:
            flush_l2(i)
        gpu_lead()
        step(evs[i])
    torch.cuda.synchronize(dev)
    lay_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    disp_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    comb_ms = sum(e[2].elapsed_time(e[3]) for e in evs)
    max_total_s = max_over_ranks(total_ms / 1e3, world, dev)
    disp_b, comb_b = wl.logical_bytes()
    logical = disp_b + comb_b
    value = aggregate_value(logical, args.steps, max_total_s, world)
    ms_per_step = max_total_s * 1e3 / args.steps

    # ---- roofline of the dominant kernel (algorithmic bytes / event time)
    per_launch_ms = {"layout": lay_ms / args.steps, "dispatch": disp_ms / args.steps,
                     "combine": comb_ms / args.steps}
    if args.fused:  # the fused call is timed as one
        per_launch_ms = {"layout_dispatch": (lay_ms + disp_ms) / args.steps,
                         "combine": comb_ms / args.steps}
    alg = algorithmic_bytes(wl, args.path, args.fused,
                            int(rl.rank_offsets[-1]) if args.path == "two_stage" else 0,
                            combine=args.combine)
    dominant = max((n for n in per_launch_ms if n != "layout"), key=lambda n: per_launch_ms[n])
    peak, peak_src = measured_peak()
    kname = "dispatch_fp8" if (dominant == "dispatch" and wl.payload == "fp8") else dominant
    if dominant == "combine" and args.combine == "fp8":
        kname = "combine_fp8"
    if args.path == "two_stage":
        kname = {"dispatch": "rank_copy+expand", "combine": "combine_partial+reduce"}[dominant]

    def roof(n):
        a = alg[n] / (per_launch_ms[n] * 1e-3) / 1e9
        return a, a / peak

    ach, frac = roof(dominant)
    roofline = {"bound": "hbm", "kernel": kname,
                "timing": "CUDA events around each call over a second pass of the K steps (each step "
                          "queued behind a GPU spin, so the events time the device)", "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": frac, "peak_source": peak_src + " (%s)" % (
                    "MEASURED_PEAKS.json hbm_gbs" if peak_src == "measured" else "6.8 TB/s"),
                "algorithmic_bytes_per_launch": alg[dominant],
                "traffic": None}
    tr = None if (args.path != "direct" or args.fused) else ncu_traffic(kname, wl)
    if tr is not None:
        roofline["traffic"] = tr["bytes"]
        roofline["traffic_note"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch "
                                    "at %d tokens (%s), scaled x%.3g by the token count" % (
                                        tr["captured_tokens"], tr["captured_workload"], tr["scale"]))
    kernels = {}
    step_sum = sum(per_launch_ms.values())
    for n in per_launch_ms:
        a, f = roof(n)
        kernels[n] = {"us_per_launch": per_launch_ms[n] * 1e3, "alg_bytes": alg[n],
                      "achieved_GBs": a, "frac_of_peak": f, "share": per_launch_ms[n] / step_sum}

    # ---- end to end through the public API with pinned host buffers: the
    # host-buffer executor (ep_roundtrip_host) copies the route, runs the
    # layout, streams x in token chunks overlapped with dispatch + combine, and
    # streams the output back, all inside the timed region
    e2e = None
    if not args.no_e2e and args.path == "direct" and args.combine == "bf16":
        xh = x.cpu().pin_memory()
        ih = idx.cpu().pin_memory()
        wh = w.cpu().pin_memory()
        oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
        pipe = ep.Pipeline(wl.T, wl.H, wl.k, wl.E, wl.R, wl.kind, wl.capacity,
                           chunk_tokens=args.chunk_tokens, device=dev,
                           y=None if wl.expert_out == "recv" else y, payload=wl.payload)
        for _ in range(3):
            pipe.run(xh, ih, wh, oh)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_ev.record(stream)
        for _ in range(args.e2e_steps):
            pipe.run(xh, ih, wh, oh)
        b_ev.record(stream)
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks(a_ev.elapsed_time(b_ev) / 1e3, world, dev)
        if not torch.equal(oh.view(torch.int16), out.cpu().view(torch.int16)):
            raise SystemExit("e2e output differs from the device-path output")
        if ep.status_read(pipe.layout.status) != 0:
            raise SystemExit("device status flags set during the e2e run")
        nch = (wl.T + args.chunk_tokens - 1) // args.chunk_tokens
        e2e = {"value": aggregate_value(logical, args.e2e_steps, e2e_s, world), "unit": "GB/s",
               "ms_per_step": e2e_s * 1e3 / args.e2e_steps,
               "h2d_bytes_per_step": x.numel() * 2 + idx.numel() * 4 + w.numel() * 4,
               "d2h_bytes_per_step": out.numel() * 2,
               "api": "ep_roundtrip_host (pinned host in/out, %d chunks of %d tokens)" % (
                   nch, args.chunk_tokens)}
        pipe.close()
        del pipe

    if ep.status_read(lay.status) != 0:
        raise SystemExit("device status flags set during the timed region")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tokens = 1024
        cpu = oracle_sample(wl, W.bf16_bits(x[:tokens]), idx[:tokens].cpu().numpy(),
                            w[:tokens].cpu().numpy(), tokens, args.cpu_seconds, args.combine)

    if rank == 0:
        props = torch.cuda.get_device_properties(dev)
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "us_per_call": ms_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.payload, "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "E": wl.E, "k": wl.k,
                       "R": wl.R, "layout": wl.kind, "payload": wl.payload, "route": wl.route,
                       "zipf_s": wl.zipf_s, "expert_outputs": wl.expert_out, "seed": wl.seed,
                       "logical_bytes_per_step": logical,
                       "l2": l2_note,
                       "parallelism": "replicas x%d" % world,
                       "launch": ("cuda graph" if args.graph else "stream (programmatic dependent launch)")
                                 + ("; layout+dispatch through ep_layout_dispatch" if args.fused else ""),
                       "path": args.path, "combine": args.combine},
            "roofline": roofline,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "device": props.name,
            "provenance": provenance(dev, idx, w, x),
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.layout_only:
            run_layout_only(args, rank, world, local)
        else:
            run_ours(args, rank, world, local)
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
