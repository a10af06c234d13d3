"""The N > 1 bench path on CPU: world-size-2 `gloo` process groups.

The layer does not shard: `bench.py --gpus N` runs N replicas
of the same per-GPU workload (weak scaling), with a barrier around the timed
region and the slowest rank's time. These tests exercise that host logic
without a GPU: the max-over-ranks reduction and the job throughput, each
rank's view of them, and the reference arm under torchrun, where rank 0
alone runs and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        dist.barrier()
        ms = bench.max_over_ranks(local_ms[rank])
        dist.barrier()
        value = bench.job_throughput(64, 10, w, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"rank": r, "world": w, "local": lr, "ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo_world2(tmp_path):
    world = 2
    local_ms = [3.0, 5.5]                 # rank 1 is the slow replica
    mp.start_processes(_rank_main, args=(world, _free_port(), local_ms, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, g in enumerate(got):
        assert (g["rank"], g["world"], g["local"]) == (r, world, r)
        assert g["ms"] == max(local_ms)   # every rank sees the job's time
        # 64 rows x 10 steps on each of 2 replicas in 5.5 ms
        assert g["value"] == pytest.approx(64 * 10 * 2 / 5.5e-3)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25) == 2.25
    assert bench.job_throughput(64, 100, 1, 10.0) == pytest.approx(640_000.0)


def test_reference_arm_under_torchrun_rank0_only(tmp_path):
    """Two ranks of the reference arm (the CPU oracle): rank 0 prints one JSON
    line for the job; rank 1 exits 0 without work."""
    env = dict(os.environ, PYTHONPATH=ROOT, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}",
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--config", "tiny", "--steps", "2", "--warmup", "1", "--reference-seconds", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=str(tmp_path), timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"] > 0
