"""GPU parity: every kernel of the hot path against the fp64 oracle, through the C ABI.

Small cases (seconds of oracle time) cover several tiles, ragged tails, odd
key counts, d = 64/128, B > 1 and the degenerate cases; they compare every
output element.  Tolerances: max-abs 2e-2 and relative L2 5e-3 on outputs
(bf16 inputs, fp32 accumulation), selection lists exact outside the 1e-4
band around tau.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_block_gb300 as vd
from workloads import WORKLOADS, Workload, make_qkv
from parity_util import assert_close, compare_selection, gpu_selection, host

pytestmark = pytest.mark.gpu

DEV = "cuda"


def rnd_qkv(B, H, Sq, Skv, d, seed, std=1.0):
    w = Workload("t", B=B, H=H, Sq=Sq, Skv=Skv, d=d, seed=seed, q_std=std, k_std=std)
    return make_qkv(w, device=DEV)


@pytest.fixture(autouse=True)
def _status_clean():
    torch.cuda.synchronize()
    yield
    assert vd.attn_last_device_status() == 0, "device status word set (timeout or bad list)"


# ---------------------------------------------------------------- pool

@pytest.mark.parametrize("B,H,S,d,block", [(1, 2, 1024, 64, 64), (2, 3, 1000, 128, 128), (1, 1, 77, 128, 64),
                                           (1, 2, 129, 64, 128)])
def test_block_pool(B, H, S, d, block):
    x, _, _ = rnd_qkv(B, H, S, S, d, seed=11)
    xp = vd.attn_block_pool(x, block)
    torch.cuda.synchronize()
    ref = oracle.block_pool(host(x), block)
    np.testing.assert_allclose(host(xp), ref, rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------- merge

@pytest.mark.parametrize("n,d", [(1, 128), (3, 64), (8, 128), (5, 128)])
def test_lse_merge(n, d):
    g = torch.Generator(device="cpu").manual_seed(5 + n)
    B, H, Sq = 1, 3, 37
    o = torch.randn((n, B, H, Sq, d), generator=g)
    lse = torch.randn((n, B, H, Sq), generator=g) * 3
    lse[:, 0, 0, 0] = -math.inf                      # a row whose partials are all empty
    if n > 1:
        lse[0, 0, 1, 2] = -math.inf                  # one empty partial
        lse[1, 0, 2, 3] = 80.0                       # dominant partial
    out, l = vd.attn_lse_merge(o.to(DEV), lse.to(DEV))
    torch.cuda.synchronize()
    ro, rl = oracle.lse_merge(o.double().numpy(), lse.double().numpy())
    assert_close(host(out), ro, "merge out")
    lg = host(l)
    assert lg[0, 0, 0] == -np.inf and np.all(host(out)[0, 0, 0] == 0)
    fin = np.isfinite(rl)
    np.testing.assert_allclose(lg[fin], rl[fin], atol=1e-5, rtol=1e-6)


# ---------------------------------------------------------------- dense

@pytest.mark.parametrize("B,H,Sq,Skv,d", [
    (1, 2, 256, 256, 128),      # exact tiles
    (1, 2, 300, 517, 64),       # ragged query and key tails
    (2, 1, 1, 1, 128),          # single token
    (1, 1, 129, 1000, 128),     # one full + one 1-row query tile
    (1, 3, 513, 255, 64),       # three query-tile pairs, odd keys
    (1, 1, 640, 2049, 128),     # odd key count across many tiles
])
def test_dense(B, H, Sq, Skv, d):
    q, k, v = rnd_qkv(B, H, Sq, Skv, d, seed=21 + Sq)
    out, lse = vd.attn_dense_fwd(q, k, v)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(host(q), host(k), host(v), 1 / math.sqrt(d))
    assert_close(host(out), ro, "dense out")
    assert_close(host(lse), rl, "dense lse")


def test_dense_large_scores_rescale():
    # peaked rows: the running max grows by far more than the lazy-rescale threshold across tiles
    B, H, S, d = 1, 2, 1024, 128
    q, k, v = rnd_qkv(B, H, S, S, d, seed=3, std=3.0)
    out, lse = vd.attn_dense_fwd(q, k, v, scale=0.3)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(host(q), host(k), host(v), 0.3)
    assert_close(host(out), ro, "dense peaked out")
    assert_close(host(lse), rl, "dense peaked lse", max_abs=2e-2 * max(1.0, float(np.abs(rl).max()) / 10))


# ---------------------------------------------------------------- split-KV + merge

@pytest.mark.parametrize("H,Sq,Skv,d,n", [(2, 128, 4096, 128, 8), (2, 128, 4097, 128, 3), (1, 100, 1000, 64, 7),
                                          (2, 130, 2000, 128, 1), (1, 128, 5, 128, 5)])
def test_splitkv_and_merge(H, Sq, Skv, d, n):
    q, k, v = rnd_qkv(1, H, Sq, Skv, d, seed=31 + Skv)
    scale = 1 / math.sqrt(d)
    op, lp = vd.attn_cross_splitkv_fwd(q, k, v, n)
    out, lse = vd.attn_lse_merge(op, lp)
    torch.cuda.synchronize()
    qh, kh, vh = host(q), host(k), host(v)
    rop, rlp = oracle.split_partials(qh, kh, vh, scale, n)
    assert_close(host(op), rop, "partials out")
    assert_close(host(lp), rlp, "partials lse")
    ro, rl = oracle.attention(qh, kh, vh, scale)
    assert_close(host(out), ro, "merged out")
    assert_close(host(lse), rl, "merged lse")


def test_splitkv_partials_16_byte_aligned():
    # the partial rows are written as whole 32-byte sectors when they start on a 32-byte boundary
    # and as 16-byte pieces otherwise: partials 16 bytes past a boundary take the second path
    H, Sq, Skv, d, n = 2, 130, 2000, 128, 4
    q, k, v = rnd_qkv(1, H, Sq, Skv, d, seed=61)
    op, lp = vd.attn_cross_splitkv_fwd(q, k, v, n)
    buf = torch.empty(n * H * Sq * d + 4, dtype=torch.float32, device=q.device)
    op16 = buf[4:].view(n, 1, H, Sq, d)
    assert op16.data_ptr() % 32 == 16
    _, lp16 = vd.attn_cross_splitkv_fwd(q, k, v, n, out_part=op16)
    torch.cuda.synchronize()
    assert torch.equal(op16, op) and torch.equal(lp16, lp)


# ---------------------------------------------------------------- block-sparse

def sparse_check(q, k, v, block, beta, scale=None, rows=None, heads_idx=None, fn=None):
    """Runs a GPU block-sparse path (two-kernel by default, or ``fn``) with route outputs and
    checks route + output against the oracle.  Returns (n_flips, density, errors)."""
    B, H, S, d = q.shape
    scale = 1 / math.sqrt(d) if scale is None else scale
    fn = vd.attn_sparse_route_fwd if fn is None else fn
    out, lse, rt = fn(q, k, v, beta, block=block, scale=scale, route=True)
    torch.cuda.synchronize()
    hs = list(range(H)) if heads_idx is None else list(heads_idx)
    qh, kh, vh = (host(x[:, hs].contiguous()) for x in (q, k, v))
    o_out, o_lse, ort, (qp, kp, vp) = oracle.sparse_route_attention(qh, kh, vh, block, block, scale, beta, rows=[0])
    gsel = gpu_selection(rt["sel_idx"][:, hs], rt["sel_cnt"][:, hs])
    flips = compare_selection(gsel, ort)
    st = host(rt["stats"][:, hs])
    np.testing.assert_allclose(st[..., 0], ort["mu"], atol=1e-4, rtol=1e-4)
    np.testing.assert_allclose(st[..., 1], ort["sigma"], atol=1e-4, rtol=1e-4)
    if beta != -math.inf:
        np.testing.assert_allclose(st[..., 2], ort["tau"], atol=1e-4, rtol=1e-4)
    # Taylor aggregates and outputs for the GPU's own selection (separates near-tau flips from arithmetic)
    forced = oracle.route(qp, kp, vp, S, block, scale, beta, force_sel=gsel)
    np.testing.assert_allclose(st[..., 3], forced["W"], atol=2e-3, rtol=1e-3)
    np.testing.assert_allclose(host(rt["taylor_t"][:, hs]), forced["T"], atol=2e-3 * block, rtol=1e-3)
    nsel = len(hs) * S
    rws = np.arange(nsel) if rows is None else np.asarray(rows)
    ro, rl = oracle.sparse_attention(qh, kh, vh, block, block, gsel, forced["mu"], forced["W"], forced["T"], scale,
                                     rows=rws)
    go = host(out[:, hs].contiguous()).reshape(-1, d)[rws]
    gl = host(lse[:, hs].contiguous()).reshape(-1)[rws]
    e1 = assert_close(go, ro, "sparse out")
    assert_close(gl, rl, "sparse lse")
    density = float(gsel.mean())
    return flips, density, e1


@pytest.mark.parametrize("beta", [0.5, -math.inf, 0.0, 3.0])
def test_sparse_tiny_config(beta):
    w = WORKLOADS["tiny"]
    q, k, v = make_qkv(w, device=DEV)
    flips, density, _ = sparse_check(q, k, v, w.block, beta)
    if beta == -math.inf:
        assert density == 1.0


def test_sparse_beta_minus_inf_equals_dense():
    for d, block in [(64, 64), (128, 128)]:
        q, k, v = rnd_qkv(1, 2, 1000, 1000, d, seed=41)
        out_s, lse_s = vd.attn_sparse_route_fwd(q, k, v, -math.inf, block=block)
        out_d, lse_d = vd.attn_dense_fwd(q, k, v)
        torch.cuda.synchronize()
        if block == 128:
            # same kernel main loop over the same tiles: bitwise equal
            assert torch.equal(out_s, out_d) and torch.equal(lse_s, lse_d)
        else:
            assert_close(host(out_s), host(out_d), "sparse(-inf) vs dense")


@pytest.mark.parametrize("d", [128, 64])
def test_sparse_all_blocks_equals_dense_over_many_ctas(d):
    # 6 heads x 52 two-tile CTAs (more than two waves of CTAs), each head ending in a short query
    # block and a short key block; with every key block selected the sparse walk does the dense
    # kernel's arithmetic in the same order, bit for bit
    S = 128 * 103 - 11
    q, k, v = rnd_qkv(1, 6, S, S, d, seed=53)
    out_s, lse_s = vd.attn_sparse_route_fwd(q, k, v, -math.inf, block=128)
    out_d, lse_d = vd.attn_dense_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(out_s, out_d) and torch.equal(lse_s, lse_d)


@pytest.mark.parametrize("d", [128, 64])
def test_sparse_query_block_order_balances_pairs_and_changes_no_bits(d):
    # the routing's query-block order: per head a permutation, sorted by list length (longest
    # first) within each run of 128 blocks; the forward runs neighbours in it on one CTA, which
    # changes which CTA computes a row but not a bit of any row
    B, H, S, block = 1, 4, 128 * 300 - 11, 128
    w0 = WORKLOADS["sparse64k"]
    w = Workload("ord", B=B, H=H, Sq=S, Skv=S, d=d, seed=59, q_std=0.5, k_std=0.5, grid=w0.grid,
                 audio_per_frame=8, pe=True, block=block, beta=1.0)
    q, k, v = make_qkv(w, device=DEV)
    rt = vd.attn_sparse_route(q, k, v, 1.0, block=block)
    out, lse = vd.attn_sparse_fwd(q, k, v, rt, block=block)
    plain = {key: val for key, val in rt.items() if key != "qb_order"}
    out0, lse0 = vd.attn_sparse_fwd(q, k, v, plain, block=block)
    torch.cuda.synchronize()
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
    order = rt["qb_order"].cpu().numpy().reshape(H, -1)
    cnt = rt["sel_cnt"].cpu().numpy().reshape(H, -1)
    nqb = order.shape[1]
    for h in range(H):
        assert sorted(order[h]) == list(range(nqb))
        for c0 in range(0, nqb, 128):
            chunk = order[h, c0:c0 + 128]
            assert set(chunk) == set(range(c0, min(c0 + 128, nqb)))
            lens = cnt[h, chunk]
            assert np.all(np.diff(lens) <= 0)
            ties = np.diff(lens) == 0
            assert np.all(np.diff(chunk)[ties] > 0)
    # the pairs' longer lists: never more than the plain pairing's
    def pair_max(o):
        return sum(int(max(cnt[h, o[h, i:i + 2]])) for h in range(H) for i in range(0, nqb, 2))
    assert pair_max(order) <= pair_max(np.tile(np.arange(nqb), (H, 1)))


def test_sparse_forward_reports_corrupt_lists_and_keeps_other_rows():
    # an empty list and an entry past the last key block: the forward reports both; the empty
    # list's rows become zeros (lse -inf), the bad entry is clamped to the last key block, and every
    # other query block's rows are exactly those of the intact routing
    B, H, S, d, block = 1, 2, 1000, 128, 128
    q, k, v = rnd_qkv(B, H, S, S, d, seed=57)
    rt = vd.attn_sparse_route(q, k, v, 1.0, block=block)
    ref_o, ref_l = vd.attn_sparse_fwd(q, k, v, rt, block=block)
    assert vd.attn_last_device_status() == 0
    nkb = rt["sel_idx"].shape[-1]
    bad = {key: val.clone() for key, val in rt.items()}
    bad["sel_cnt"][0, 0, 3] = 0
    bad["sel_idx"][0, 1, 2, 0] = nkb + 5
    out, lse = vd.attn_sparse_fwd(q, k, v, bad, block=block)
    assert vd.attn_last_device_status() == 1     # ATTN_ERR_INVALID_ARG
    rows3 = slice(3 * block, 4 * block)
    assert torch.all(out[0, 0, rows3] == 0) and torch.all(torch.isneginf(lse[0, 0, rows3]))
    # the clamped list now holds the last key block where it held its first entry
    fixed = {key: val.clone() for key, val in rt.items()}
    fixed["sel_idx"][0, 1, 2, 0] = nkb - 1
    fo, fl = vd.attn_sparse_fwd(q, k, v, fixed, block=block)
    assert vd.attn_last_device_status() == 0
    rows2 = slice(2 * block, 3 * block)
    assert torch.equal(out[0, 1, rows2], fo[0, 1, rows2]) and torch.equal(lse[0, 1, rows2], fl[0, 1, rows2])
    keep = torch.ones(H, S, dtype=torch.bool, device=out.device)
    keep[0, rows3] = False
    keep[1, rows2] = False
    assert torch.equal(out[0][keep], ref_o[0][keep]) and torch.equal(lse[0][keep], ref_l[0][keep])
    # an order entry past the last query block is clamped and reported too; the blocks the
    # order still names come out as with the intact routing
    odd = {key: val.clone() for key, val in rt.items()}
    nqb = odd["qb_order"].shape[-1]
    lost = int(odd["qb_order"][0, 1, 0])
    odd["qb_order"][0, 1, 0] = nqb + 3
    o2, l2 = vd.attn_sparse_fwd(q, k, v, odd, block=block)
    assert vd.attn_last_device_status() == 1
    named = [b for b in range(nqb) if b != lost]
    for b in named:
        rows = slice(b * block, min((b + 1) * block, S))
        assert torch.equal(o2[0, 1, rows], ref_o[0, 1, rows]) and torch.equal(l2[0, 1, rows], ref_l[0, 1, rows])


@pytest.mark.parametrize("d,block,beta", [(128, 128, 1.0), (128, 64, 0.5), (64, 128, 1.5)])
def test_sparse_local_workload_ragged(d, block, beta):
    # the Stage-2 generator (noise + 3D position code, interleaved audio) truncated to two frames: S = 8208
    w = WORKLOADS["sparse64k"]
    w2 = Workload("s2", B=1, H=2, Sq=8208, Skv=8208, d=d, seed=7, q_std=0.5, k_std=0.5, grid=w.grid,
                  audio_per_frame=8, pe=True, block=block, beta=beta)
    q, k, v = make_qkv(w2, device=DEV)
    flips, density, _ = sparse_check(q, k, v, block, beta)
    assert 0.0 < density < 1.0


def test_sparse_batch_gt_one():
    q, k, v = rnd_qkv(2, 2, 640, 640, 128, seed=43)
    out, lse, rt = vd.attn_sparse_route_fwd(q, k, v, 0.7, block=128, route=True)
    torch.cuda.synchronize()
    for b in range(2):
        qh, kh, vh = (host(x[b:b + 1]) for x in (q, k, v))
        _, _, ort, (qp, kp, vp) = oracle.sparse_route_attention(qh, kh, vh, 128, 128, 1 / math.sqrt(128), 0.7,
                                                                rows=[0])
        gsel = gpu_selection(rt["sel_idx"][b:b + 1], rt["sel_cnt"][b:b + 1])
        compare_selection(gsel, ort)
        forced = oracle.route(qp, kp, vp, 640, 128, 1 / math.sqrt(128), 0.7, force_sel=gsel)
        ro, rl = oracle.sparse_attention(qh, kh, vh, 128, 128, gsel, forced["mu"], forced["W"], forced["T"],
                                         1 / math.sqrt(128))
        assert_close(host(out[b:b + 1]), ro, f"batch {b} out")
        assert_close(host(lse[b:b + 1]), rl, f"batch {b} lse")


@pytest.mark.parametrize("d,block", [(128, 128), (128, 64), (64, 128)])
def test_sparse_given_lists_uneven_between_paired_tiles(d, block):
    # Hand-made selections through attn_sparse_fwd: neighbouring query tiles (the two
    # tiles a dense/sparse CTA holds) get lists of very different lengths (all key
    # blocks against one, one against none-but-the-last, ...), so one tile's walk ends
    # long before the other's.  The Taylor aggregates for the forced selection come
    # from the oracle's routing, and the oracle computes the same attention.
    B, H, S = 1, 2, 1000
    q, k, v = rnd_qkv(B, H, S, S, d, seed=61 + d + block)
    nqb = (S + block - 1) // block
    rng = np.random.default_rng(5)
    sel = np.zeros((B, H, nqb, nqb), dtype=bool)
    for h in range(H):
        for i in range(nqb):
            kind = (i + h) % 4
            if kind == 0:
                sel[0, h, i, :] = True                       # every key block
            elif kind == 1:
                sel[0, h, i, nqb - 1] = True                 # only the ragged last block
            elif kind == 2:
                sel[0, h, i, i] = True                       # only the diagonal
            else:
                sel[0, h, i, rng.choice(nqb, size=max(1, nqb // 3), replace=False)] = True
    qh, kh, vh = host(q), host(k), host(v)
    qp, kp, vp = (oracle.block_pool(x, block) for x in (qh, kh, vh))
    scale = 1 / math.sqrt(d)
    forced = oracle.route(qp, kp, vp, S, block, scale, 0.0, force_sel=sel)
    rt = vd.sparse_route_buffers(B, H, S, d, block, DEV)
    idx = np.zeros((B, H, nqb, nqb), dtype=np.int32)
    cnt = sel.sum(-1).astype(np.int32)
    for h in range(H):
        for i in range(nqb):
            lst = np.flatnonzero(sel[0, h, i])
            idx[0, h, i, :lst.size] = lst
    stats = np.stack([forced["mu"], forced["sigma"], forced["tau"], forced["W"]], axis=-1)
    rt["sel_idx"].copy_(torch.from_numpy(idx))
    rt["sel_cnt"].copy_(torch.from_numpy(cnt))
    rt["stats"].copy_(torch.from_numpy(stats.astype(np.float32)))
    rt["taylor_t"].copy_(torch.from_numpy(np.ascontiguousarray(forced["T"], dtype=np.float32)))
    out, lse = vd.attn_sparse_fwd(q, k, v, rt, block=block)
    torch.cuda.synchronize()
    ro, rl = oracle.sparse_attention(qh, kh, vh, block, block, sel, forced["mu"], forced["W"], forced["T"], scale)
    assert_close(host(out), ro, "sparse given-lists out")
    assert_close(host(lse), rl, "sparse given-lists lse")


# ---------------------------------------------------------------- routing folded into the forward

@pytest.mark.parametrize("beta", [0.5, -math.inf, 3.0])
def test_fused_tiny_config(beta):
    w = WORKLOADS["tiny"]
    q, k, v = make_qkv(w, device=DEV)
    _, density, _ = sparse_check(q, k, v, w.block, beta, fn=vd.attn_sparse_fused_fwd)
    if beta == -math.inf:
        assert density == 1.0


@pytest.mark.parametrize("d,block,beta", [(128, 128, 1.0), (128, 64, 0.5), (64, 128, 1.5), (64, 64, 0.0)])
def test_fused_local_workload_ragged(d, block, beta):
    w = WORKLOADS["sparse64k"]
    w2 = Workload("s2", B=1, H=2, Sq=8208, Skv=8208, d=d, seed=8, q_std=0.5, k_std=0.5, grid=w.grid,
                  audio_per_frame=8, pe=True, block=block, beta=beta)
    q, k, v = make_qkv(w2, device=DEV)
    _, density, _ = sparse_check(q, k, v, block, beta, fn=vd.attn_sparse_fused_fwd)
    assert 0.0 < density < 1.0


def test_fused_agrees_with_two_kernel_path_and_dense():
    B, H, S, d, block, beta = 2, 2, 1000, 128, 128, 0.6
    scale = 1 / math.sqrt(d)
    q, k, v = rnd_qkv(B, H, S, S, d, seed=47, std=1.0)
    o1, l1, r1 = vd.attn_sparse_route_fwd(q, k, v, beta, block=block, route=True)
    o2, l2, r2 = vd.attn_sparse_fused_fwd(q, k, v, beta, block=block, route=True)
    torch.cuda.synchronize()
    s1 = gpu_selection(r1["sel_idx"], r1["sel_cnt"])
    s2 = gpu_selection(r2["sel_idx"], r2["sel_cnt"])
    np.testing.assert_allclose(host(r1["stats"])[..., 0], host(r2["stats"])[..., 0], atol=1e-5, rtol=1e-5)
    if np.array_equal(s1, s2):
        assert_close(host(o2), host(o1), "fused vs two-kernel")
        np.testing.assert_allclose(host(r2["taylor_t"]), host(r1["taylor_t"]), atol=1e-2, rtol=1e-4)
    # whether or not the two selections agree: each may differ from the oracle's only inside the
    # near-tau band, and each path's output must match the oracle evaluated on its own selection
    for b in range(B):
        qh, kh, vh = (host(x[b:b + 1]) for x in (q, k, v))
        _, _, ort, (qp, kp, vp) = oracle.sparse_route_attention(qh, kh, vh, block, block, scale, beta, rows=[0])
        for name, o, l, sel in (("two-kernel", o1, l1, s1), ("fused", o2, l2, s2)):
            compare_selection(sel[b:b + 1], ort)
            forced = oracle.route(qp, kp, vp, S, block, scale, beta, force_sel=sel[b:b + 1])
            ro, rl = oracle.sparse_attention(qh, kh, vh, block, block, sel[b:b + 1], forced["mu"], forced["W"],
                                             forced["T"], scale)
            assert_close(host(o[b:b + 1]), ro, f"{name} out, batch {b}")
            assert_close(host(l[b:b + 1]), rl, f"{name} lse, batch {b}")
    # with every block kept, the fused path runs exactly the dense arithmetic
    od, ld = vd.attn_dense_fwd(q, k, v)
    of, lf = vd.attn_sparse_fused_fwd(q, k, v, -math.inf, block=block)
    torch.cuda.synchronize()
    assert torch.equal(of, od) and torch.equal(lf, ld)


# ---------------------------------------------------------------- status word

def test_bounded_wait_reports_timeout_and_context_survives():
    vd.attn_selftest_wait_timeout(2000)
    assert vd.attn_last_device_status() == 5
    assert vd.attn_last_device_status() == 0          # cleared on read
    q, k, v = rnd_qkv(1, 1, 128, 128, 64, seed=1)
    out, _ = vd.attn_dense_fwd(q, k, v)
    torch.cuda.synchronize()
    ro, _ = oracle.attention(host(q), host(k), host(v), 1 / 8)
    assert_close(host(out), ro, "dense after timeout self-test")


def test_launch_wide_abort_ends_a_broken_launch_quickly():
    # 16 waves of one CTA per SM, every CTA waiting on a barrier nothing arrives on with a 20 ms limit:
    # waited out wave by wave that would take >= 320 ms; with the launch-wide abort the first timeout
    # stops the CTAs still waiting and the later waves return at once, so the launch takes ~20 ms
    vd.attn_selftest_wait_timeout(10)                    # loads the module; its timeout is read and cleared
    assert vd.attn_last_device_status() == 5
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    limit_us, waves = 20000, 16
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    vd.attn_selftest_wait_timeout_grid(limit_us, waves * n_sm)
    status = vd.attn_last_device_status()
    elapsed = time.perf_counter() - t0
    assert status == 5
    assert elapsed < 0.1, f"aborted launch took {elapsed * 1e3:.1f} ms"
    print(f"aborted launch of {waves * n_sm} CTAs ended after {elapsed * 1e3:.1f} ms (wait limit {limit_us / 1e3} ms)")
    assert vd.attn_last_device_status() == 0
    # later launches carry their own ids and are not affected
    q, k, v = rnd_qkv(1, 2, 300, 517, 128, seed=2)
    out, lse = vd.attn_dense_fwd(q, k, v)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(host(q), host(k), host(v), 1 / math.sqrt(128))
    assert_close(host(out), ro, "dense after an aborted launch")
    assert_close(host(lse), rl, "dense lse after an aborted launch")


# ---------------------------------------------------------------- split-KV with the merge in the tail

@pytest.mark.parametrize("H,Sq,Skv,d,n", [(2, 128, 4096, 128, 8), (2, 300, 4097, 128, 3), (1, 100, 1000, 64, 7),
                                          (3, 129, 517, 128, 1), (2, 1, 2, 64, 2)])
def test_cross_fused_merge_matches_two_launch_path_and_oracle(H, Sq, Skv, d, n):
    q, k, v = rnd_qkv(1, H, Sq, Skv, d, seed=77 + Sq + n)
    ws = torch.zeros(vd.attn_cross_workspace_bytes(1, H, Sq, d, n), dtype=torch.uint8, device=DEV)
    out, lse = vd.attn_cross_fwd(q, k, v, n, workspace=ws)
    op, lp = vd.attn_cross_splitkv_fwd(q, k, v, n)
    out2, lse2 = vd.attn_lse_merge(op, lp)
    # the workspace is ready for the next call: a second call gives the same bits
    out3, lse3 = vd.attn_cross_fwd(q, k, v, n, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert torch.equal(out, out3) and torch.equal(lse, lse3)
    tiles = H * ((Sq + 127) // 128)                       # counters: the workspace's last 256-aligned region
    off = ws.numel() - ((4 * tiles + 255) // 256) * 256
    assert int(ws[off:off + 4 * tiles].view(torch.int32).abs().sum()) == 0      # counters back at zero
    ro, rl = oracle.attention(host(q), host(k), host(v), 1 / math.sqrt(d))
    assert_close(host(out), ro, "fused cross out")
    assert_close(host(lse), rl, "fused cross lse")


# ---------------------------------------------------------------- degenerate routing cases

@pytest.mark.parametrize("fn", [None, "fused"])
def test_sparse_identical_pooled_keys_select_everything(fn):
    # every key block holds the same rows, so all pooled keys are equal: sigma = 0, tau = mu, and
    # every proxy ties with tau and is selected; the result is dense attention
    B, H, S, d, block = 1, 2, 1024, 128, 128
    q, k, v = rnd_qkv(B, H, S, S, d, seed=61)
    k = k[:, :, :block].repeat(1, 1, S // block, 1).contiguous()
    f = vd.attn_sparse_fused_fwd if fn == "fused" else None
    # an exact tie: the GPU's fp32 Welford mean of identical proxies is exact (sigma = 0, all selected),
    # while the fp64 oracle's two-pass mean may round by an ulp and put tau a hair above them; such
    # flips lie inside the 1e-4 band that sparse_check accepts
    flips, density, _ = sparse_check(q, k, v, block, 1.5, fn=f)
    if fn == "fused":
        return   # the prologue's two-pass fp32 mean can round the tie too (checked against the band above)
    assert density == 1.0
    out, lse, _ = vd.attn_sparse_route_fwd(q, k, v, 1.5, block=block, route=True)
    dense, dlse = vd.attn_dense_fwd(q, k, v)
    torch.cuda.synchronize()
    assert_close(host(out), host(dense), "identical keys vs dense (GPU)")


@pytest.mark.parametrize("S,block", [(100, 128), (64, 64), (1, 64)])
def test_sparse_shorter_than_one_block(S, block):
    # one query block and one key block: the argmax keeps it, there is nothing to reject
    q, k, v = rnd_qkv(1, 2, S, S, 64, seed=62 + S)
    flips, density, _ = sparse_check(q, k, v, block, 2.0)
    assert flips == 0 and density == 1.0
