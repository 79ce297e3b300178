"""The bench's multi-rank path on the CPU (gloo, world size 2), no GPU.

The path shards into independent (b, key-head group) units with no collective
on the data path; the only cross-rank operations are the harness's barrier and
the max over ranks of the step time.  These tests run them in two processes
over gloo, and the reference arm under torchrun, where rank 0 alone runs the
oracle and prints the one JSON line.
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        bench.barrier(2)
        ms = bench.max_over_ranks(1.0 + 2.0 * rank, 2)  # rank 0: 1 ms, rank 1: 3 ms
        out[rank] = ms
        bench.barrier(2)
    finally:
        dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU gloo test")
def test_barrier_and_max_over_ranks_gloo():
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(_free_port(), out), nprocs=2, join=True)
    assert dict(out) == {0: 3.0, 1: 3.0}


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU gloo test")
def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--workload", "toy_fp32", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
