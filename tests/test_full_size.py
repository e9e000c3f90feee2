"""Full-size parity: the benchmark-size workloads in the launch configuration bench.py times.

The GPU runs each whole problem; the oracle recomputes sampled heads and
sampled query rows one by one (seeded), plus the complete routing of the
sampled heads.  Tolerances as in the small cases.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_block_gb300 as vd
from workloads import WORKLOADS, Workload, make_qkv
from parity_util import assert_close, compare_selection, gpu_selection, host

pytestmark = pytest.mark.gpu


def sample_heads(H, rng, n=4):
    extra = rng.choice(np.arange(1, H - 1), size=max(0, n - 2), replace=False)
    return sorted({0, H - 1, *extra.tolist()})


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.empty_cache()
    assert vd.attn_last_device_status() == 0


def test_dense16k_full_size_sampled_rows():
    w = WORKLOADS["dense16k"]
    q, k, v = make_qkv(w, device="cuda")
    out, lse = vd.attn_dense_fwd(q, k, v)
    torch.cuda.synchronize()
    rng = np.random.default_rng(102)
    hs = sample_heads(w.H, rng)
    qh, kh, vh = (host(x[:, hs].contiguous()) for x in (q, k, v))
    rows = np.sort(rng.choice(len(hs) * w.Sq, size=512, replace=False))
    ro, rl = oracle.attention(qh, kh, vh, w.scale, rows=rows)
    go = host(out[:, hs].contiguous()).reshape(-1, w.d)[rows]
    gl = host(lse[:, hs].contiguous()).reshape(-1)[rows]
    assert_close(go, ro, "dense16k out")
    assert_close(gl, rl, "dense16k lse")


@pytest.mark.parametrize("Skv", [32768, 32769])
def test_cross_full_size_split_merge(Skv):
    w = WORKLOADS["cross"]
    q, k, v = make_qkv(w, device="cuda", Skv=Skv)
    op, lp = vd.attn_cross_splitkv_fwd(q, k, v, w.n_split)
    out, lse = vd.attn_lse_merge(op, lp)
    dense, dlse = vd.attn_dense_fwd(q, k, v)
    torch.cuda.synchronize()
    # merged partials against the GPU's own unsplit attention (every head, every row)
    assert_close(host(out), host(dense), "merged vs unsplit (GPU)")
    assert_close(host(lse), host(dlse), "merged lse vs unsplit (GPU)")
    rng = np.random.default_rng(103 + Skv)
    hs = sample_heads(w.H, rng)
    qh, kh, vh = (host(x[:, hs].contiguous()) for x in (q, k, v))
    rop, rlp = oracle.split_partials(qh, kh, vh, w.scale, w.n_split)
    assert_close(host(op[:, :, hs].contiguous()), rop, "partials out")
    assert_close(host(lp[:, :, hs].contiguous()), rlp, "partials lse")
    ro, rl = oracle.attention(qh, kh, vh, w.scale)
    assert_close(host(out[:, hs].contiguous()), ro, "merged out")
    assert_close(host(lse[:, hs].contiguous()), rl, "merged lse")


def sparse_full_size(w, beta, n_rows, n_heads, seed, fn=None):
    fn = vd.attn_sparse_route_fwd if fn is None else fn
    q, k, v = make_qkv(w, device="cuda")
    out, lse, rt = fn(q, k, v, beta, block=w.block, route=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    hs = sample_heads(w.H, rng, n_heads)
    qh, kh, vh = (host(x[:, hs].contiguous()) for x in (q, k, v))
    del q, k, v
    qp, kp, vp = (oracle.block_pool(x, w.block) for x in (qh, kh, vh))
    ort = oracle.route(qp, kp, vp, w.Sq, w.block, w.scale, beta)
    gsel = gpu_selection(rt["sel_idx"][:, hs], rt["sel_cnt"][:, hs])
    flips = compare_selection(gsel, ort)
    st = host(rt["stats"][:, hs])
    np.testing.assert_allclose(st[..., 0], ort["mu"], atol=1e-4, rtol=1e-4)
    np.testing.assert_allclose(st[..., 1], ort["sigma"], atol=1e-4, rtol=1e-4)
    forced = oracle.route(qp, kp, vp, w.Sq, w.block, w.scale, beta, force_sel=gsel)
    np.testing.assert_allclose(st[..., 3], forced["W"], atol=2e-3, rtol=1e-3)
    np.testing.assert_allclose(host(rt["taylor_t"][:, hs]), forced["T"], atol=0.3, rtol=1e-3)
    rows = np.sort(rng.choice(len(hs) * w.Sq, size=n_rows, replace=False))
    ro, rl = oracle.sparse_attention(qh, kh, vh, w.block, w.block, gsel, forced["mu"], forced["W"], forced["T"],
                                     w.scale, rows=rows)
    go = host(out[:, hs].contiguous()).reshape(-1, w.d)[rows]
    gl = host(lse[:, hs].contiguous()).reshape(-1)[rows]
    assert_close(go, ro, f"{w.name} beta={beta} out")
    assert_close(gl, rl, f"{w.name} beta={beta} lse")
    return flips, float(gsel.mean())


def test_sparse64k_full_size():
    w = WORKLOADS["sparse64k"]
    flips, density = sparse_full_size(w, w.beta, n_rows=4096, n_heads=4, seed=104)
    assert 0.0 < density < 1.0


@pytest.mark.parametrize("H,S,d,beta", [(8, 128 * 301 - 37, 128, 0.5), (12, 128 * 201 - 5, 64, 1.0)])
def test_fused_routing_odd_block_count_mid_size(H, S, d, beta):
    # routing folded into the forward at a size between the small cases and the benchmark: an odd
    # query-block count leaves the second tile of the last CTA of every head without a block, and
    # the last key block is short
    nqb = -(-S // 128)
    assert nqb % 2 == 1
    w0 = WORKLOADS["sparse64k"]
    w = Workload("fp", B=1, H=H, Sq=S, Skv=S, d=d, seed=43 + d, q_std=0.5, k_std=0.5, grid=w0.grid,
                 audio_per_frame=8, pe=True, block=128, beta=beta)
    flips, density = sparse_full_size(w, beta, n_rows=2048, n_heads=3, seed=108 + d, fn=vd.attn_sparse_fused_fwd)
    assert 0.0 < density < 1.0


@pytest.mark.parametrize("H,S,d,beta", [(8, 128 * 301 - 37, 128, 0.5), (12, 128 * 201 - 5, 64, 1.0)])
def test_sparse_two_launch_mid_size_odd_block_count(H, S, d, beta):
    # pool + route + forward at a size between the small cases and the benchmark (the sizes of the
    # folded-routing case above): an odd query-block count leaves the second tile of the last CTA
    # of every head without a block, and the last key block is short
    w0 = WORKLOADS["sparse64k"]
    w = Workload("tp", B=1, H=H, Sq=S, Skv=S, d=d, seed=47 + d, q_std=0.5, k_std=0.5, grid=w0.grid,
                 audio_per_frame=8, pe=True, block=128, beta=beta)
    flips, density = sparse_full_size(w, beta, n_rows=2048, n_heads=3, seed=112 + d)
    assert 0.0 < density < 1.0


def test_sparse64k_full_size_fused_routing():
    w = WORKLOADS["sparse64k"]
    flips, density = sparse_full_size(w, w.beta, n_rows=4096, n_heads=4, seed=106, fn=vd.attn_sparse_fused_fwd)
    assert 0.0 < density < 1.0


@pytest.mark.parametrize("beta", [-math.inf, 0.0, 0.5, 1.0, 2.0])
def test_sweep128k_full_size(beta):
    w = WORKLOADS["sweep128k"]
    flips, density = sparse_full_size(w, beta, n_rows=512, n_heads=2, seed=105)
    if beta == -math.inf:
        assert density == 1.0


def test_na3d_full_size_sampled_rows():
    w = WORKLOADS["na3d"]
    q, k, v = make_qkv(w, device="cuda")
    out, lse = vd.attn_na3d_fwd(q, k, v, w.grid, w.extra["kernel"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(107)
    hs = sample_heads(w.H, rng)
    qh, kh, vh = (host(x[:, hs].contiguous()) for x in (q, k, v))
    # every row of the first and last sampled head, 4096 sampled rows of the others
    rows = np.concatenate([np.arange(w.Sq), (len(hs) - 1) * w.Sq + np.arange(w.Sq),
                           rng.choice(np.arange(w.Sq, (len(hs) - 1) * w.Sq), size=4096, replace=False)])
    rows = np.sort(rows)
    ro, rl = oracle.na3d_attention(qh, kh, vh, w.grid, w.extra["kernel"], w.scale, rows=rows)
    go = host(out[:, hs].contiguous()).reshape(-1, w.d)[rows]
    gl = host(lse[:, hs].contiguous()).reshape(-1)[rows]
    assert_close(go, ro, "na3d out")
    assert_close(gl, rl, "na3d lse")


def test_na3d_full_size_e5m2_window_same_bits_as_library_plan():
    # plan 6 (E5M2 window operands, asked for) at the full na3d size: the raw scores of the
    # synthetic recipe are far inside its exact range, so it must give the library's plan 5
    # bit for bit (plan 5 is checked against the oracle above); the same launch bench.py times
    w = WORKLOADS["na3d"]
    q, k, v = make_qkv(w, device="cuda")
    assert vd.attn_na3d_plan(w.grid, w.extra["kernel"])[:2] == (3, 5)
    o5, l5 = vd.attn_na3d_fwd(q, k, v, w.grid, w.extra["kernel"])
    o6, l6 = vd.attn_na3d_fwd(q, k, v, w.grid, w.extra["kernel"], brick=3, pair_axis=6)
    torch.cuda.synchronize()
    assert torch.equal(o6, o5) and torch.equal(l6, l5)
