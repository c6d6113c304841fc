"""Host-side logic of bench.py: the max-over-ranks reduction and the
whole-job aggregation on world_size-2 gloo process groups (CPU), and the
CPU-only reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_seconds = 1.0 + rank          # rank 1 is the slowest
    m = bench.max_over_ranks(local_seconds, world)
    bench.barrier(world)
    v = bench.aggregate_value(15e9, 10, m, world)
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 2.0                                   # max over ranks
        assert v == pytest.approx(2 * 15e9 * 10 / 2.0 / 1e9)  # all ranks' bytes / slowest time


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_value(1e9, 4, 2.0, 1) == pytest.approx(2.0)
    peak, src = bench.measured_peak()
    assert peak > 0 and src in ("measured", "fallback")


def test_reference_arm_runs_on_cpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["host_cores"] == os.cpu_count()


def test_reference_arm_under_torchrun_two_ranks():
    # N > 1 launch of the reference arm: rank 0 runs and prints, rank 1 exits 0
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port),
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


def test_algorithmic_bytes_accounting():
    sys.path.insert(0, ROOT)
    import bench
    from combine_ep_layout_02_gb300 import workloads as W
    wl = W.WORKLOADS["prefill"]
    T, H, k = wl.T, wl.H, wl.k
    a = bench.algorithmic_bytes(wl)
    assert a["layout"] == 2 * T * k * 4
    assert a["dispatch"] == T * H * 2 + T * k * H * 2 + T * k * 4          # read x once, k rows out
    assert a["combine"] == T * k * H * 2 + T * H * 2 + T * k * 8           # k rows in, one out
    # the full-size prefill figures of the measurement table: 8,457.8 and 8,459.9 MB
    assert round(a["dispatch"] / 1e6, 1) == 8457.8 and round(a["combine"] / 1e6, 1) == 8459.9
    f = W.WORKLOADS["prefill_fp8"]
    af = bench.algorithmic_bytes(f)
    assert af["dispatch"] == f.T * f.H * 2 + f.T * f.k * (f.H + 4 * f.H // 128) + f.T * f.k * 4
    assert round(af["dispatch"] / 1e6, 1) == 9634.3
    fused = bench.algorithmic_bytes(wl, fused=True)
    assert fused == {"layout_dispatch": a["layout"] + a["dispatch"], "combine": a["combine"]}
    # two-stage with every pair in its own rank row equals the direct bytes plus
    # one more write and read of those rows in each direction
    nr = T * k
    t2 = bench.algorithmic_bytes(wl, path="two_stage", rank_rows=nr)
    assert t2["dispatch"] == a["dispatch"] + 2 * nr * H * 2 + 2 * T * k * 4
    assert t2["combine"] == a["combine"] + 2 * nr * H * 2 + T * k * 8 + nr * 4
    # FP8 expert outputs: codes plus a 4-byte scale per 128 channels in, bf16 out
    c8 = bench.algorithmic_bytes(f, combine="fp8")
    assert c8["combine"] == f.T * f.k * (f.H + f.H // 32) + f.T * f.H * 2 + f.T * f.k * 8
    assert c8["dispatch"] == af["dispatch"]


def test_host_cpu_record():
    sys.path.insert(0, ROOT)
    import bench
    info = bench.host_cpu()
    assert info["host_cores"] == os.cpu_count() and info["machine"]


def test_ncu_traffic_scales_by_tokens(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from combine_ep_layout_02_gb300 import workloads as W
    os.makedirs(tmp_path / "profiles")
    ent = {"kernel": "k", "workload": "prefill", "tokens": 16384, "H": 7168, "k": 8,
           "valid_tokens": [16384, 1 << 40], "dram_bytes_read": 100, "dram_bytes_write": 300,
           "source_sha256_16": "abc"}
    with open(tmp_path / "profiles" / "traffic.json", "w") as f:
        json.dump({"kernels": {"dispatch": ent}}, f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda rel: "abc")
    tr = bench.ncu_traffic("dispatch", W.WORKLOADS["prefill"])
    assert tr["bytes"] == 400 * 4 and tr["scale"] == 4          # 65,536 / 16,384 tokens
    assert bench.ncu_traffic("dispatch", W.WORKLOADS["prefill"].scaled(T=8192)) is None  # other instance
    assert bench.ncu_traffic("dispatch", W.WORKLOADS["masked"]) is None                  # other H
    assert bench.ncu_traffic("combine", W.WORKLOADS["prefill"]) is None                  # not captured
    monkeypatch.setattr(bench, "source_hash", lambda rel: "changed")
    assert bench.ncu_traffic("dispatch", W.WORKLOADS["prefill"]) is None                 # source changed
