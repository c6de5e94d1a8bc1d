"""Host-side logic of bench.py (CPU only): the replica aggregation over ranks
with gloo at world size 2, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    seconds = [0.010, 0.025][rank]
    value, slowest = bench.aggregate_throughput(1000.0, seconds, world, torch.device("cpu"))
    out[rank] = (value, slowest)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_throughput_takes_the_slowest_rank():
    port = 29500 + os.getpid() % 1000
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        value, slowest = res[r]
        assert abs(slowest - 0.025) < 1e-12
        assert abs(value - 2000.0 / 0.025) < 1e-6


def test_reference_arm_prints_one_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "1",
           "--workload", "f32_T256_d64_N4_k1_dff256_cf1.25", "--ref-budget", "3"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.strip().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    # the timing it reports is the time it spent: the whole small batch ran each step
    assert not d["extrapolated"] and d["tokens_per_timed_step"] == 256
    assert abs(d["timed_region_s"] - d["ms_per_step"] * 1e-3 * d["steps"]) < 1e-9


def test_gpus_flag_launches_one_rank_per_gpu():
    """bench.py --gpus 2 without a launcher re-runs itself under
    torch.distributed.run with two ranks; on the host-core arm rank 0 alone
    prints the line, which reports both ranks, and the other rank exits 0."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference", "--steps", "1",
           "--warmup", "1", "--workload", "f32_T256_d64_N4_k1_dff256_cf1.25", "--ref-budget", "2"]
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.strip().splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["config"]["parallelism"] == "replicas2"


def test_both_arms_report_the_same_config():
    """The reference arm's config is built by the same function as the GPU
    arm's, from the oracle's capacity and kept counts."""
    sys.path.insert(0, ROOT)
    import bench
    from sparse_mixture_experts_66_b300.workload import WORKLOADS

    w = WORKLOADS["f32_T256_d64_N4_k1_dff256_cf1.25"]
    cfg = bench.config_dict(w, 80, [64, 64, 64, 64], 1)
    assert cfg["kept_rows"] == 256 and cfg["active_experts"] == 4 and cfg["capacity"] == 80
    assert set(cfg) == {"workload", "T", "d", "N", "k", "d_ff", "capacity_factor", "router_bias", "capacity",
                        "kept_rows", "active_experts", "parallelism", "l2"}
