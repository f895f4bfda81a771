"""The benchmark's multi-rank harness on CPU (gloo, world size 2).

bench.py runs one independent replica per GPU under torchrun (the path does
not shard across GPUs); across ranks it only needs a barrier and the maximum
of the per-rank step times, and under ``--impl reference`` rank 0 alone runs
the oracle and prints while the other ranks exit 0 without work.  Both are
checked here with two CPU processes; no GPU is involved.
"""
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


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(0.25 + rank, dist)   # rank 1 is the slower one
        alone = bench.max_over_ranks(3.0, None)
        dist.barrier()
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"max": got, "alone": alone}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d == {"max": 1.25, "alone": 3.0}


def test_reference_arm_rank0_only(tmp_path):
    """torchrun with two ranks: one JSON line (rank 0's), exit code 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--reference-budget-s", "1"]
    r = subprocess.run(cmd, cwd=str(tmp_path), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_rank_does_no_work():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, reference_budget_s = 1, 3, 1.0

    assert bench.run_reference(A(), rank=1, world=2) is None
