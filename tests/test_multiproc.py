"""Multi-rank host logic of bench.py on CPU: world size 2 over gloo.

Every GPU machine in this setup has one GPU, so the N > 1 launch path (one process
per GPU under torchrun) is exercised here on the host: the rendezvous, the
barrier around the timed region, the max-over-ranks reduction of the timed
duration, and the rule that only rank 0 runs the reference arm and prints.
The attention path itself needs no collective (replicas shard by head/batch).
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                          LOCAL_RANK=str(rank))
        import bench
        w, r, local = bench.dist_setup()
        assert (w, r, local) == (world, rank, rank)
        bench.barrier(w)
        # each rank "timed" a different duration: everyone must see the slowest
        m = bench.max_over_ranks(10.0 + 5.0 * rank, w)

        class A:
            steps, warmup, beta, cpu_seconds = 1, 3, 1.0, 0.2
        ref = bench.run_reference(A, w, r) if r != 0 else "rank0-skipped"
        import torch.distributed as dist
        dist.destroy_process_group()
        q.put((rank, m, ref))
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, "error", repr(e)))


def test_two_ranks_gloo_barrier_max_and_rank0_only_reference():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(2):
        rank, m, ref = q.get(timeout=120)
        results[rank] = (m, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0][0] == 15.0 and results[1][0] == 15.0, results
    assert results[1][1] is None            # non-zero ranks do no reference work and print nothing
