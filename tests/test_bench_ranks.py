"""bench.py's multi-rank plumbing on CPU (gloo, world size 2): the barrier,
the max over ranks that sets the job time of N replicas, and the reference
arm doing its work on rank 0 only."""
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_path):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(ws),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench

    w, r, _ = bench.dist_env()
    assert (w, r) == (ws, rank)
    bench.init_dist(ws, rank, "gloo")
    bench.barrier(ws)
    mx = bench.max_over_ranks(1.5 + rank, ws)  # rank 1 is the slower replica
    # the reference arm: only rank 0 works and prints; the others return 0 at once
    import argparse

    rc = bench.run_reference(argparse.Namespace(gpus=ws, steps=0, warmup=0), None) if rank == 1 else 0
    bench.barrier(ws)
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(f"{mx} {rc}")
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_max_and_reference_rank_gate(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    out = str(tmp_path / "rank")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        mx, rc = open(f"{out}.{r}").read().split()
        assert float(mx) == 2.5
        assert int(rc) == 0
