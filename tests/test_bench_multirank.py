"""bench.py's multi-rank plumbing on CPU: world size 2 over gloo.

The decode path shards into independent replicas, so the only cross-rank
steps are the barrier around the timed region and the max over ranks of the
elapsed time; the reference arm runs on rank 0 alone.  No GPU needed."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup(None)
    bench.barrier(w)
    elapsed = bench.max_over_ranks(1.5 + rank, w)   # rank 1 is the slow one
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "max": elapsed}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [g["rank"] for g in got] == [0, 1]
    assert all(g["world"] == world for g in got)
    assert all(g["max"] == 2.5 for g in got)   # every rank reports the slowest rank's time


def test_reference_arm_prints_once_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "2", "--warmup", "1", "--ref-seconds", "0.3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(l) for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout                  # rank 0 alone prints
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    cfg = line["config"]                                # the same workload keys as our arm's line
    assert cfg["workload"] == "tiny" and cfg["B"] == 4 and cfg["D"] == 64 and cfg["q_len"] == 1
