"""The N > 1 path of bench.py on the CPU, over gloo with two ranks: the path shards into
independent replicas (no collective on the data path), so what N > 1 adds is the host
logic -- the rank setup, the barrier, the max over ranks of the timed region, and rank 0
alone printing the line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

# the gloo path: with a GPU visible the bench's helpers take NCCL, one device a rank
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="the CPU (gloo) path")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks_take_the_max(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # each rank's "timed region" differs; every rank gets the slowest
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_ranks_take_the_max, args=(2, _free_port(), out), nprocs=2,
                           start_method="spawn")
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "tiny_sliding", "--steps", "3",
           "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["scaling"] == "weak"
