"""GPU parity of the sharded cross attention (video keys/values split over ranks).

One GPU per process here, so two rank layouts are checked on it: (a) the ranks'
work emulated in one process -- each shard's split-KV partials computed by the
CUDA library, concatenated in rank order exactly as the all-gather lays them
out, and merged by the library; (b) the real function over a one-rank NCCL
group.  No kernel waits on another rank.  The two-rank exchange itself is
tested over gloo on the CPU (tests/test_multiproc.py).
"""
import math
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
import video_diffusion_transformer_block_gb300 as vd
from video_diffusion_transformer_block_gb300 import sharded
from workloads import Workload, make_qkv
from parity_util import assert_close, host

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    torch.cuda.synchronize()
    yield
    assert vd.attn_last_device_status() == 0


@pytest.mark.parametrize("world,Skv,n_split", [(2, 32768, 4), (3, 4097, 2), (2, 300, 1)])
def test_sharded_partials_gathered_in_rank_order_merge_exactly(world, Skv, n_split):
    w = Workload("x", B=1, H=4, Sq=128, Skv=Skv, d=128, seed=40 + world)
    q, k, v = make_qkv(w, device="cuda")
    parts = []
    for r in range(world):
        lo, hi = sharded.shard_bounds(Skv, world, r)
        parts.append(vd.attn_cross_splitkv_fwd(q, k[:, :, lo:hi].contiguous(), v[:, :, lo:hi].contiguous(), n_split))
    o_all = torch.cat([p[0] for p in parts], dim=0)
    l_all = torch.cat([p[1] for p in parts], dim=0)
    out, lse = vd.attn_lse_merge(o_all, l_all)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(host(q), host(k), host(v), w.scale)
    assert_close(host(out), ro, "sharded merged out")
    assert_close(host(lse), rl, "sharded merged lse")


def test_sharded_function_over_one_rank_nccl_group():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", world_size=1, rank=0)
    try:
        w = Workload("x", B=1, H=4, Sq=100, Skv=5000, d=128, seed=44)
        q, k, v = make_qkv(w, device="cuda")
        out, lse = sharded.cross_attention_sharded(q, k, v, n_split=3)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    ro, rl = oracle.attention(host(q), host(k), host(v), w.scale)
    assert_close(host(out), ro, "sharded (1 rank) out")
    assert_close(host(lse), rl, "sharded (1 rank) lse")
