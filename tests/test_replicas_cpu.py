"""The multi-GPU path is replicas only: each rank runs its own token streams,
with no collective on the data path. What is left to test runs on the host and
is covered here on CPU, with world size 2 over `gloo`: the job's time is the
slowest rank's and its rate counts every rank's tokens (the same function the
bench uses after its timed region), and the reference arm under torchrun prints
one line from rank 0 while the other rank exits 0 without work.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r took 10 + 5r ms for its 100 tokens
        elapsed, rate = bench.replica_job_rate(10.0 + 5.0 * rank, 100, world)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
            json.dump({"elapsed": elapsed, "rate": rate}, fh)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_rate_is_max_over_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for g in got:
        assert g["elapsed"] == 15.0                       # the slowest rank
        assert g["rate"] == pytest.approx(world * 100 / 0.015)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_job_rate(20.0, 50, 1) == (20.0, 50 / 0.02)


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--workload",
           "relu_d512_f2048_fp32", "--steps", "2", "--warmup", "1", "--tokens", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_gpus_flag_without_a_launcher_starts_that_many_ranks():
    """`bench.py --gpus 2` run directly starts two replica processes itself
    (torch.distributed.run on 127.0.0.1); rank 0 prints the one line with
    n_gpus 2. A rank count that differs from --gpus is refused."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--workload",
           "relu_d512_f2048_fp32", "--steps", "2", "--warmup", "1", "--tokens", "2"]
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env.update(OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["config"]["parallelism"] == "replicas"
    bad = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                         env=dict(env, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert bad.returncode != 0 and "--gpus 2" in bad.stderr


def test_reference_arm_times_what_it_prints():
    """The reference arm runs every warm-up step, times whole tokens through
    the whole stack, and prints the config keys our arm prints."""
    sys.path.insert(0, ROOT)
    import bench
    from activation_sparse_ffn_gb300 import workload as W
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "relu_d512_f2048_fp32", "--steps", "3", "--warmup", "2", "--tokens", "4"]
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env.update(OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    assert d["steps"] == 3 and d["warmup"] == 2
    assert d["value"] == pytest.approx(1e3 / d["ms_per_step"], rel=1e-3)
    spec = W.spec_replace(W.WORKLOADS["relu_d512_f2048_fp32"], layers=4)
    want = bench.bench_config(spec, 1, 4, 4, False, False, 1,
                              "single-layer workload rotated over 4 independent layer replicas")
    assert d["config"] == json.loads(json.dumps(want))
