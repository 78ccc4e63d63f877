"""The multi-process (replicas) path of bench.py on the CPU: two gloo ranks.

The hot path has no exchange step, so N processes are N independent replicas;
the only cross-rank operations are the barrier around the timed region and the
max / sum reductions of the timings and the work done.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch

    import bench

    r, w, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist, w)
    mx = bench.max_over_ranks(dist, w, 1.5 + r, torch.device("cpu"))
    sm = bench.sum_over_ranks(dist, w, 10.0 * (r + 1), torch.device("cpu"))
    bench.barrier(dist, w)
    with open(f"{out_path}.{r}", "w") as f:
        json.dump({"rank": r, "world": w, "max": mx, "sum": sm}, f)
    dist.destroy_process_group()


def test_rank_reductions_over_gloo(tmp_path):
    import torch.multiprocessing as mp

    out = str(tmp_path / "rank")
    mp.spawn(_rank_main, args=(2, free_port(), out), nprocs=2, join=True)
    for r in range(2):
        with open(f"{out}.{r}") as f:
            got = json.load(f)
        assert got == {"rank": r, "world": 2, "max": 2.5, "sum": 30.0}


def test_reference_arm_under_torchrun():
    """Under torchrun only rank 0 times the oracle and prints the one JSON line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-seconds", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
