"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one process per GPU (torchrun); the work partitions by
independent (batch, head) replicas, so the only cross-rank steps are the
barrier around the timed region and the max-over-ranks of the step time.
These run here with the gloo backend (no GPU needed); the reference arm is
run under torchrun with two ranks, where rank 0 alone works and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    # Each rank's step time differs; every rank must see the largest.
    m = bench.max_over_ranks(1.5 + rank, w)
    # Replicas draw different inputs (seed + 7919 * rank), as bench.py does.
    wl = bench.workload("c1")
    q, *_ = bench.make_inputs(1, 1, 16, 16, "fp32", wl.seed + 7919 * rank)
    import torch.distributed as dist
    qs = [torch.empty_like(q) for _ in range(world)]
    dist.all_gather(qs, q)
    out[rank] = (m, bool(torch.equal(qs[0], qs[1])))
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5
    assert res[0][1] is False, "the two replicas must not draw the same inputs"


def test_reference_arm_under_torchrun_two_ranks():
    """Rank 0 alone times the oracle and prints one JSON line; rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "c1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
