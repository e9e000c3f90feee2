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


# ---------------------------------------------------------------- sharded cross attention (host logic, gloo)

def _oracle_partials(q, k, v, n_split, scale):
    import oracle
    o, l = oracle.split_partials(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, n_split)
    import torch
    return torch.from_numpy(o), torch.from_numpy(l)


def _oracle_merge(o_part, lse_part):
    import oracle
    import torch
    o, l = oracle.lse_merge(o_part.numpy(), lse_part.numpy())
    return torch.from_numpy(o), torch.from_numpy(l)


def _sharded_rank(rank, world, port, Skv, n_split, q):
    try:
        sys.path.insert(0, ROOT)
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        import numpy as np
        import torch
        import torch.distributed as dist
        from video_diffusion_transformer_block_gb300 import sharded
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", world_size=world, rank=rank)
        g = torch.Generator().manual_seed(31)
        B, H, Sq, d = 1, 2, 5, 16
        qq = torch.randn((B, H, Sq, d), generator=g, dtype=torch.float64)
        kk = torch.randn((B, H, Skv, d), generator=g, dtype=torch.float64)
        vv = torch.randn((B, H, Skv, d), generator=g, dtype=torch.float64)
        lo, hi = sharded.shard_bounds(Skv, world, rank)
        out, lse = sharded.cross_attention_sharded(qq, kk[:, :, lo:hi].contiguous(), vv[:, :, lo:hi].contiguous(),
                                                   n_split, scale=0.25, partials=_oracle_partials,
                                                   merge=_oracle_merge)
        dist.destroy_process_group()
        q.put((rank, out.numpy(), lse.numpy(), qq.numpy(), kk.numpy(), vv.numpy()))
    except Exception as e:
        q.put((rank, "error", repr(e), None, None, None))


@pytest.mark.parametrize("world,Skv,n_split", [(2, 1000, 3), (2, 7, 2), (3, 301, 1)])
def test_sharded_cross_attention_gathers_and_merges_exactly(world, Skv, n_split):
    import numpy as np
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sharded_rank, args=(r, world, port, Skv, n_split, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r = q.get(timeout=180)
        assert not isinstance(r[1], str), r
        res[r[0]] = r
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    _, out0, lse0, qq, kk, vv = res[0]
    ref_o, ref_l = oracle.attention(qq, kk, vv, 0.25)
    for r in range(world):
        # every rank holds the same exact answer over all keys
        np.testing.assert_allclose(res[r][1], ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(res[r][2], ref_l, rtol=0, atol=1e-12)


def test_shard_bounds_partition():
    sys.path.insert(0, ROOT)
    from video_diffusion_transformer_block_gb300.sharded import shard_bounds
    for S in (0, 1, 7, 1000, 32769):
        for world in (1, 2, 3, 8):
            b = [shard_bounds(S, world, r) for r in range(world)]
            assert b[0][0] == 0 and b[-1][1] == S
            assert all(b[i][1] == b[i + 1][0] for i in range(world - 1))
            assert max(h - l for l, h in b) - min(h - l for l, h in b) <= 1
    with pytest.raises(ValueError):
        shard_bounds(10, 2, 2)
