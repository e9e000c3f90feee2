"""Pins for the fp64 oracle: closed forms, library routines and invariants.

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (a dropped term, a wrong sign or index, a transposed
operand, an off-by-one chunk bound) fails at least one of them.  CPU only.
"""
import bisect
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle

RNG = np.random.default_rng(1234)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def sdpa64(q, k, v, scale, mask=None):
    """torch's own attention routine in float64 on the CPU (a library routine the oracle does not use)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    out = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=None if mask is None else t(mask),
                                                           scale=scale)
    return out.numpy()


# ---------------------------------------------------------------- dense attention

@pytest.mark.parametrize("B,H,Sq,Skv,d", [(1, 2, 33, 57, 64), (2, 1, 128, 256, 128), (1, 1, 1, 1, 64), (1, 3, 200, 7, 16)])
def test_dense_matches_library_sdpa(B, H, Sq, Skv, d):
    q, k, v = rand(B, H, Sq, d), rand(B, H, Skv, d), rand(B, H, Skv, d)
    scale = 1 / math.sqrt(d)
    out, lse = oracle.attention(q, k, v, scale)
    ref = sdpa64(q, k, v, scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # lse against scipy's logsumexp of the explicit score matrix
    scores = scale * np.einsum("bhqd,bhkd->bhqk", q, k)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(scores, axis=-1), rtol=0, atol=1e-12)


def test_dense_two_keys_closed_form():
    # with two keys the softmax is a logistic function of the score difference
    d = 4
    q = rand(1, 1, 5, d)
    k = rand(1, 1, 2, d)
    v = rand(1, 1, 2, d)
    scale = 0.7
    out, lse = oracle.attention(q, k, v, scale)
    x = scale * q[0, 0] @ k[0, 0].T                      # [5, 2]
    s1 = 1.0 / (1.0 + np.exp(-(x[:, 0] - x[:, 1])))
    expect = s1[:, None] * v[0, 0, 0] + (1 - s1)[:, None] * v[0, 0, 1]
    np.testing.assert_allclose(out[0, 0], expect, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.logaddexp(x[:, 0], x[:, 1]), atol=1e-13)


def test_dense_identical_keys_give_mean_value():
    d, Skv = 8, 37
    q = rand(1, 1, 3, d)
    k = np.repeat(rand(1, 1, 1, d), Skv, axis=2)
    v = rand(1, 1, Skv, d)
    out, lse = oracle.attention(q, k, v, 0.5)
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(v[0, 0].mean(0), (3, d)), atol=1e-13)
    x = 0.5 * q[0, 0] @ k[0, 0, 0]
    np.testing.assert_allclose(lse[0, 0], x + math.log(Skv), atol=1e-12)


def test_dense_large_scores_are_stable_and_one_hot():
    d = 4
    k = np.zeros((1, 1, 5, d))
    k[0, 0, :, 0] = [-3, 1, 7, 2, 0]
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 400.0                               # scores up to 2800: exp overflows without the max shift
    v = rand(1, 1, 5, d)
    out, lse = oracle.attention(q, k, v, 1.0)
    assert np.all(np.isfinite(out)) and np.isfinite(lse).all()
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, 2], atol=1e-12)
    np.testing.assert_allclose(lse[0, 0, 0], 2800.0, atol=1e-9)


def test_dense_rows_sum_to_one_before_v():
    q, k = rand(1, 2, 40, 16), rand(1, 2, 90, 16)
    out, _ = oracle.attention(q, k, np.ones((1, 2, 90, 16)), 0.25)
    np.testing.assert_allclose(out, 1.0, atol=1e-14)
    # one-hot value columns expose the weights themselves: each row of weights sums to 1
    v = np.zeros((1, 2, 90, 90))
    v[0, :, np.arange(90), np.arange(90)] = 1.0
    w, _ = oracle.attention(np.pad(q, ((0, 0), (0, 0), (0, 0), (0, 74))), np.pad(k, ((0, 0), (0, 0), (0, 0), (0, 74))),
                            v, 0.25)
    np.testing.assert_allclose(w.sum(-1), 1.0, atol=1e-13)
    assert (w >= 0).all()


def test_dense_key_permutation_invariance_and_row_subset():
    q, k, v = rand(1, 1, 20, 8), rand(1, 1, 50, 8), rand(1, 1, 50, 8)
    perm = RNG.permutation(50)
    a, la = oracle.attention(q, k, v, 0.3)
    b, lb = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.3)
    np.testing.assert_allclose(a, b, atol=1e-13)
    np.testing.assert_allclose(la, lb, atol=1e-13)
    rows = np.array([19, 0, 7])
    c, lc = oracle.attention(q, k, v, 0.3, rows=rows)
    np.testing.assert_array_equal(c, a[0, 0, rows])
    np.testing.assert_array_equal(lc, la[0, 0, rows])


# ---------------------------------------------------------------- split-KV + merge

@pytest.mark.parametrize("Skv,n", [(257, 1), (257, 2), (257, 3), (257, 8), (32769 // 64, 8), (5, 5), (3, 7)])
def test_split_merge_equals_unsplit(Skv, n):
    q, k, v = rand(1, 2, 9, 16), rand(1, 2, Skv, 16), rand(1, 2, Skv, 16)
    full, lfull = oracle.attention(q, k, v, 0.25)
    op, lp = oracle.split_partials(q, k, v, 0.25, n)
    out, lse = oracle.lse_merge(op, lp)
    np.testing.assert_allclose(out, full, atol=1e-12)
    np.testing.assert_allclose(lse, lfull, atol=1e-12)
    # every chunk is plain attention over its balanced, unpadded key range
    for c in range(n):
        lo, hi = (c * Skv) // n, ((c + 1) * Skv) // n
        if hi == lo:
            assert np.all(lp[c] == -np.inf) and np.all(op[c] == 0)
            continue
        np.testing.assert_allclose(op[c], sdpa64(q, k[:, :, lo:hi], v[:, :, lo:hi], 0.25), atol=1e-12)


def test_split_single_chunk_is_identity():
    q, k, v = rand(1, 1, 4, 8), rand(1, 1, 31, 8), rand(1, 1, 31, 8)
    op, lp = oracle.split_partials(q, k, v, 0.5, 1)
    full, lfull = oracle.attention(q, k, v, 0.5)
    np.testing.assert_array_equal(op[0], full)
    np.testing.assert_array_equal(lp[0], lfull)


def test_unpadded_odd_length_equals_padded_and_masked():
    # the padded key, masked out, changes nothing: attention over the odd-length sequence is the same
    Skv = 65
    q, k, v = rand(1, 2, 6, 8), rand(1, 2, Skv, 8), rand(1, 2, Skv, 8)
    kp = np.concatenate([k, rand(1, 2, 1, 8)], axis=2)
    vp = np.concatenate([v, rand(1, 2, 1, 8)], axis=2)
    mask = np.ones((6, Skv + 1), dtype=bool)
    mask[:, -1] = False
    padded = sdpa64(q, kp, vp, 0.4, mask=mask)
    out, _ = oracle.attention(q, k, v, 0.4)
    np.testing.assert_allclose(out, padded, atol=1e-12)


def test_merge_closed_form_two_partials():
    # two partials with lse a, b: weights are the logistic function of a - b
    o1, o2 = rand(3, 4), rand(3, 4)
    a, b = np.array([0.0, 3.0, -700.0]), np.array([1.0, -2.0, -701.0])
    out, lse = oracle.lse_merge(np.stack([o1, o2]), np.stack([a, b]))
    w1 = 1.0 / (1.0 + np.exp(b - a))
    np.testing.assert_allclose(out, w1[:, None] * o1 + (1 - w1)[:, None] * o2, atol=1e-13)
    np.testing.assert_allclose(lse, np.logaddexp(a, b), atol=1e-12)


def test_merge_all_empty_and_one_empty():
    o = rand(2, 3, 4)
    out, lse = oracle.lse_merge(np.zeros((2, 3, 4)), np.full((2, 3), -np.inf))
    assert np.all(out == 0) and np.all(lse == -np.inf)
    out, lse = oracle.lse_merge(np.stack([o[0], np.zeros((3, 4))]), np.stack([np.array([0.5, 1.0, 2.0]), np.full(3, -np.inf)]))
    np.testing.assert_allclose(out, o[0], atol=1e-15)
    np.testing.assert_allclose(lse, [0.5, 1.0, 2.0], atol=1e-15)


# ---------------------------------------------------------------- pooling

@pytest.mark.parametrize("S,block", [(256, 64), (300, 64), (129, 128), (1, 64), (1024, 128)])
def test_pool_matches_numpy_mean(S, block):
    x = rand(2, 3, S, 16)
    xp = oracle.block_pool(x, block)
    nb = -(-S // block)
    assert xp.shape == (2, 3, nb, 16)
    for i in range(nb):
        np.testing.assert_allclose(xp[:, :, i], x[:, :, i * block:(i + 1) * block].mean(axis=2), atol=1e-14)


def test_pool_constant_blocks():
    x = np.repeat(np.arange(5.0)[None, None, :, None], 64, axis=2).reshape(1, 1, 320, 1) * np.ones((1, 1, 1, 4))
    xp = oracle.block_pool(x, 64)
    np.testing.assert_array_equal(xp[0, 0, :, 0], np.arange(5.0))


# ---------------------------------------------------------------- routing

def brute_route(q, k, v, block_q, block_k, scale, beta, clamp=True):
    """Direct enumeration from raw tokens: proxy = mean token-pair score of each block pair."""
    B, H, S, d = q.shape
    nq, nk = -(-S // block_q), -(-S // block_k)
    out = {}
    scores = scale * np.einsum("bhqd,bhkd->bhqk", q, k)
    proxy = np.zeros((B, H, nq, nk))
    for i in range(nq):
        for j in range(nk):
            proxy[:, :, i, j] = scores[:, :, i * block_q:(i + 1) * block_q, j * block_k:(j + 1) * block_k].mean(axis=(2, 3))
    mu = proxy.mean(-1)
    sigma = proxy.std(-1)
    tau = np.full_like(mu, -np.inf) if beta == -np.inf else mu + beta * sigma
    sel = proxy >= tau[..., None]
    am = proxy.argmax(-1)
    for b in range(B):
        for h in range(H):
            for i in range(nq):
                sel[b, h, i, am[b, h, i]] = True
    sizes = np.array([min(block_k, S - j * block_k) for j in range(nk)], dtype=float)
    w = sizes * (1 + proxy - mu[..., None])
    if clamp:
        w = np.maximum(w, 0)
    w = np.where(sel, 0.0, w)
    vbar = np.stack([v[:, :, j * block_k:(j + 1) * block_k].mean(axis=2) for j in range(nk)], axis=2)
    out.update(proxy=proxy, mu=mu, sigma=sigma, tau=tau, sel=sel, W=w.sum(-1), T=np.einsum("bhij,bhjd->bhid", w, vbar))
    return out


@pytest.mark.parametrize("S,bq,bk,beta", [(256, 64, 64, 0.5), (300, 64, 128, 0.0), (512, 128, 64, 1.3), (256, 64, 64, -0.7)])
def test_route_matches_brute_force_enumeration(S, bq, bk, beta):
    d = 16
    q, k, v = rand(1, 2, S, d), rand(1, 2, S, d), rand(1, 2, S, d)
    scale = 1 / math.sqrt(d)
    _, _, rt, _ = oracle.sparse_route_attention(q, k, v, bq, bk, scale, beta, rows=np.arange(2))
    ref = brute_route(q, k, v, bq, bk, scale, beta)
    np.testing.assert_allclose(rt["proxy"], ref["proxy"], atol=1e-12)
    np.testing.assert_allclose(rt["mu"], ref["mu"], atol=1e-12)
    np.testing.assert_allclose(rt["sigma"], ref["sigma"], atol=1e-12)
    np.testing.assert_allclose(rt["tau"], ref["tau"], atol=1e-12)
    # selection must agree exactly away from the threshold
    near = np.abs(ref["proxy"] - ref["tau"][..., None]) < 1e-9
    assert np.array_equal(rt["sel"] | near, ref["sel"] | near)
    np.testing.assert_array_equal(rt["sel_cnt"], rt["sel"].sum(-1))
    np.testing.assert_allclose(rt["W"], ref["W"], atol=1e-10)
    np.testing.assert_allclose(rt["T"], ref["T"], atol=1e-10)


def test_route_beta_minus_inf_selects_all():
    q, k, v = rand(1, 1, 256, 8), rand(1, 1, 256, 8), rand(1, 1, 256, 8)
    _, _, rt, _ = oracle.sparse_route_attention(q, k, v, 64, 64, 0.3, -np.inf, rows=np.arange(1))
    assert rt["sel"].all()
    assert np.all(rt["tau"] == -np.inf)
    assert np.all(rt["W"] == 0) and np.all(rt["T"] == 0)


def test_route_constant_keys_zero_sigma_selects_all():
    # identical pooled keys (dyadic values, exact mean) -> sigma = 0 -> every block meets tau = mu
    q = rand(1, 1, 256, 8)
    k = np.tile(np.array([0.5, -0.25, 1.0, 0.0, 0.125, 2.0, -1.0, 0.75]), (1, 1, 256, 1))
    v = rand(1, 1, 256, 8)
    qp, kp, vp = oracle.block_pool(q, 64), oracle.block_pool(k, 64), oracle.block_pool(v, 64)
    rt = oracle.route(qp, kp, vp, 256, 64, 1.0, 2.0)
    assert np.all(rt["sigma"] == 0)
    assert rt["sel"].all()


def test_route_density_monotone_in_beta_and_argmax_kept():
    q, k, v = rand(1, 2, 512, 16), rand(1, 2, 512, 16), rand(1, 2, 512, 16)
    qp, kp, vp = oracle.block_pool(q, 64), oracle.block_pool(k, 64), oracle.block_pool(v, 64)
    prev = None
    for beta in [-np.inf, -2, -1, 0, 0.5, 1, 2, 5, 1e9]:
        rt = oracle.route(qp, kp, vp, 512, 64, 0.25, beta)
        dens = rt["sel"].sum()
        if prev is not None:
            assert dens <= prev
        prev = dens
        am = rt["proxy"].argmax(-1)
        assert np.take_along_axis(rt["sel"], am[..., None], -1).all()
    assert prev == 2 * 8                                 # beta -> inf keeps only the argmax block of each row


# ---------------------------------------------------------------- sparse attention + Taylor term

def test_sparse_beta_minus_inf_equals_dense_bitwise():
    q, k, v = rand(1, 2, 300, 16), rand(1, 2, 300, 16), rand(1, 2, 300, 16)
    out, lse, rt, _ = oracle.sparse_route_attention(q, k, v, 64, 64, 0.25, -np.inf)
    dense, ldense = oracle.attention(q, k, v, 0.25)
    assert np.array_equal(out, dense)
    assert np.array_equal(lse, ldense)


def test_sparse_without_taylor_equals_masked_library_attention():
    # zero Taylor aggregates: the output is softmax attention restricted to the selected blocks
    S, b = 256, 64
    q, k, v = rand(1, 1, S, 8), rand(1, 1, S, 8), rand(1, 1, S, 8)
    qp, kp, vp = oracle.block_pool(q, b), oracle.block_pool(k, b), oracle.block_pool(v, b)
    rt = oracle.route(qp, kp, vp, S, b, 0.5, 0.8)
    assert not rt["sel"].all()
    out, _ = oracle.sparse_attention(q, k, v, b, b, rt["sel"], rt["mu"], np.zeros_like(rt["W"]),
                                     np.zeros_like(rt["T"]), 0.5)
    mask = np.repeat(np.repeat(rt["sel"][0, 0], b, axis=0), b, axis=1)
    np.testing.assert_allclose(out, sdpa64(q, k, v, 0.5, mask=mask), atol=1e-12)


def load_taylor_fixture():
    path = os.path.join(GOLDEN, "taylor_closed_form.txt")
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, rhs = line.split("=", 1)
                vals[key.strip()] = np.array([float(t) for t in rhs.split()])
    return vals


def test_taylor_hand_derived_closed_form():
    """Two query blocks x two key blocks with identical tokens inside each block.

    Every token score then equals its block proxy, so the Taylor-corrected
    row has a two-term closed form (derivation in the fixture file)."""
    g = load_taylor_fixture()
    a, bq = g["q_block0"], g["q_block1"]
    alpha, gamma = g["k_block0"], g["k_block1"]
    vA, vB = g["v_block0"], g["v_block1"]
    beta, scale = float(g["beta"][0]), float(g["scale"][0])
    q = np.array([a, a, bq, bq])[None, None]
    k = np.array([alpha, alpha, gamma, gamma])[None, None]
    v = np.array([vA, vA, vB, vB])[None, None]
    out, lse, rt, _ = oracle.sparse_route_attention(q, k, v, 2, 2, scale, beta)
    # row block 0: s00 = 0.6, s01 = 0.2 -> mu = 0.4, sigma = 0.2, only block 0 kept
    # row block 1: s10 = 0.2, s11 = 0.4 -> mu = 0.3, sigma = 0.1, only block 1 kept
    np.testing.assert_allclose(rt["mu"][0, 0], [0.4, 0.3], atol=1e-14)
    np.testing.assert_allclose(rt["sigma"][0, 0], [0.2, 0.1], atol=1e-14)
    assert rt["sel"][0, 0].tolist() == [[True, False], [False, True]]
    np.testing.assert_allclose(rt["W"][0, 0], [2 * 0.8, 2 * 0.9], atol=1e-14)
    r0 = math.exp(-0.2) * 0.8
    r1 = math.exp(-0.1) * 0.9
    exp0 = (vA + r0 * vB) / (1 + r0)
    exp1 = (vB + r1 * vA) / (1 + r1)
    np.testing.assert_allclose(out[0, 0, 0], exp0, atol=1e-14)
    np.testing.assert_allclose(out[0, 0, 1], exp0, atol=1e-14)
    np.testing.assert_allclose(out[0, 0, 2], exp1, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], 0.6 + math.log(2 + 2 * r0), atol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 3], 0.4 + math.log(2 + 2 * r1), atol=1e-14)


def test_taylor_term_converges_quadratically_to_exact_attention():
    """The Taylor term is a first-order expansion of exp about the row-mean proxy
    score, so it must agree with exact softmax attention up to second-order terms.

    Self-attention over S = 90 tokens in blocks of 16 (the last block ragged, 10
    tokens).  Every query row is the same unit vector and the keys are identical
    inside each key block, so every token score equals its block's proxy score,
    mu + delta * t_j (t_j fixed, |t_j| <= 1), for every row.  Query block i keeps
    only key block i; the others go through the Taylor term.  Exact attention over
    all keys and the Taylor-corrected output then differ by O(delta^2): shrinking
    delta tenfold must shrink the error about a hundredfold.  A dropped term, a
    wrong sign or a missing block-size factor n_j would leave an error of order
    delta or 1."""
    b, d, S = 16, 8, 90
    nkb = (S + b - 1) // b
    t = np.array([0.9, -0.5, 0.3, -0.8, 0.6, -0.2])
    rng = np.random.default_rng(11)
    vblk = rng.standard_normal((nkb, d))
    rest = rng.standard_normal((nkb, d - 1))
    sel = np.eye(nkb, dtype=bool)[None, None]
    errs, lerrs = [], []
    for delta in (1e-1, 1e-2, 1e-3):
        q = np.zeros((1, 1, S, d))
        q[..., 0] = 1.0                                   # score = the key's first coordinate
        kblk = np.concatenate([(0.7 + delta * t)[:, None], rest], axis=1)
        k = np.repeat(kblk, b, axis=0)[:S][None, None]
        v = np.repeat(vblk, b, axis=0)[:S][None, None]
        qp, kp, vp = (oracle.block_pool(x, b) for x in (q, k, v))
        forced = oracle.route(qp, kp, vp, S, b, 1.0, 0.0, force_sel=sel)
        np.testing.assert_allclose(forced["proxy"][0, 0], np.tile(0.7 + delta * t, (nkb, 1)), atol=1e-14)
        out, lse = oracle.sparse_attention(q, k, v, b, b, sel, forced["mu"], forced["W"], forced["T"], 1.0)
        s_tok = np.repeat(0.7 + delta * t, b)[:S]
        p = np.exp(s_tok - s_tok.max())
        exact = (p[:, None] * v[0, 0]).sum(0) / p.sum()
        exact_lse = s_tok.max() + math.log(p.sum())
        errs.append(np.abs(out[0, 0] - exact).max())
        lerrs.append(np.abs(lse[0, 0] - exact_lse).max())
    for e in (errs, lerrs):
        assert e[2] < 1e-6, e
        for m in (0, 1):
            ratio = e[m] / e[m + 1]
            assert 60 < ratio < 160, (e, ratio)


def test_taylor_constant_v_and_unit_mass():
    # with V constant, num = c * den exactly in exact arithmetic: the output is that constant,
    # i.e. the selected probabilities plus the Taylor mass sum to one
    S = 320
    q, k = rand(1, 2, S, 16, scale=0.5), rand(1, 2, S, 16, scale=0.5)
    cst = rand(16)
    v = np.tile(cst, (1, 2, S, 1))
    out, _, rt, _ = oracle.sparse_route_attention(q, k, v, 64, 64, 0.25, 0.5)
    assert not rt["sel"].all()
    np.testing.assert_allclose(out, np.broadcast_to(cst, out.shape), atol=1e-13)
    out1, _, _, _ = oracle.sparse_route_attention(q, k, np.ones((1, 2, S, 16)), 64, 64, 0.25, 0.5)
    np.testing.assert_allclose(out1, 1.0, atol=1e-14)


def test_taylor_unclamped_switch_and_clamp_count():
    # strongly peaked rows: some rejected blocks fall below mu - 1 and get clamped
    S, b, d = 512, 64, 16
    q, k, v = rand(1, 1, S, d, scale=3), rand(1, 1, S, d, scale=3), rand(1, 1, S, d)
    qp, kp, vp = oracle.block_pool(q, b), oracle.block_pool(k, b), oracle.block_pool(v, b)
    rc = oracle.route(qp, kp, vp, S, b, 1.0, 0.5, clamp=True)
    ru = oracle.route(qp, kp, vp, S, b, 1.0, 0.5, clamp=False)
    low = (~rc["sel"]) & (rc["proxy"] < rc["mu"][..., None] - 1)
    assert rc["n_clamped"] == int(low.sum()) > 0
    assert np.all(rc["W"] >= ru["W"])


def test_route_forced_selection_matches_threshold_rule_on_its_own_selection():
    # forcing the selection the threshold rule would take reproduces W and T exactly
    q, k, v = rand(1, 2, 384, 16), rand(1, 2, 384, 16), rand(1, 2, 384, 16)
    qp, kp, vp = oracle.block_pool(q, 64), oracle.block_pool(k, 64), oracle.block_pool(v, 64)
    rt = oracle.route(qp, kp, vp, 384, 64, 0.25, 0.3)
    rf = oracle.route(qp, kp, vp, 384, 64, 0.25, 0.3, force_sel=rt["sel"])
    assert np.array_equal(rf["sel"], rt["sel"])
    np.testing.assert_array_equal(rf["W"], rt["W"])
    np.testing.assert_array_equal(rf["T"], rt["T"])
    flip = rt["sel"].copy()
    flip[0, 0, 0, 0] = ~flip[0, 0, 0, 0]
    ff = oracle.route(qp, kp, vp, 384, 64, 0.25, 0.3, force_sel=flip)
    assert ff["sel_cnt"][0, 0, 0] == rt["sel_cnt"][0, 0, 0] + (1 if flip[0, 0, 0, 0] else -1)


# ---------------------------------------------------------------- 3D neighbourhood attention

def nearest_window(p, K, L):
    """Start of the K-position window nearest to p: among all starts whose window
    lies inside [0, L), the one whose centre p' = s + K//2 is closest to p
    (a search over feasible windows, not the clamp formula)."""
    starts = np.arange(L - K + 1)
    return int(starts[np.argmin(np.abs(starts + K // 2 - p))])


def na_mask(grid, kernel):
    """Boolean [S, S] key mask of 3D neighbourhood attention, built token by token."""
    T, Y, X = grid
    S = T * Y * X
    coords = [(t, y, x) for t in range(T) for y in range(Y) for x in range(X)]
    mask = np.zeros((S, S), dtype=bool)
    for i, c in enumerate(coords):
        lo = [nearest_window(c[a], kernel[a], grid[a]) for a in range(3)]
        for j, e in enumerate(coords):
            mask[i, j] = all(lo[a] <= e[a] < lo[a] + kernel[a] for a in range(3))
    return mask


NA_CASES = [((3, 5, 6), (3, 3, 3)), ((4, 6, 5), (2, 4, 3)), ((1, 7, 9), (1, 5, 4)), ((5, 4, 4), (3, 4, 1)),
            ((2, 3, 8), (2, 1, 8))]


@pytest.mark.parametrize("grid,kernel", NA_CASES)
def test_na3d_matches_masked_library_attention(grid, kernel):
    S = int(np.prod(grid))
    d = 8
    q, k, v = rand(1, 2, S, d), rand(1, 2, S, d), rand(1, 2, S, d)
    scale = 0.45
    out, lse = oracle.na3d_attention(q, k, v, grid, kernel, scale)
    mask = na_mask(grid, kernel)
    add = np.where(mask, 0.0, -np.inf)[None, None]
    np.testing.assert_allclose(out, sdpa64(q, k, v, scale, mask=add), rtol=0, atol=1e-12)
    scores = scale * np.einsum("bhqd,bhkd->bhqk", q, k) + add
    np.testing.assert_allclose(lse, scipy.special.logsumexp(scores, axis=-1), rtol=0, atol=1e-12)


@pytest.mark.parametrize("grid,kernel", NA_CASES[:3])
def test_na3d_window_indicator(grid, kernel):
    # uniform scores and one-hot values: row i of the output is the window of
    # query i divided by its size, so the exact key set is visible
    S = int(np.prod(grid))
    q = np.zeros((1, 1, S, S))
    v = np.eye(S)[None, None]
    out, lse = oracle.na3d_attention(q, q, v, grid, kernel, 1.0)
    n = int(np.prod(kernel))
    np.testing.assert_allclose(out[0, 0], na_mask(grid, kernel) / n, rtol=0, atol=1e-15)
    np.testing.assert_array_equal((out[0, 0] > 0).sum(axis=1), n)
    np.testing.assert_allclose(lse, math.log(n), atol=1e-14)


def test_na3d_single_token_window_returns_own_value():
    grid = (2, 3, 4)
    S, d = 24, 16
    q, k, v = rand(2, 1, S, d), rand(2, 1, S, d), rand(2, 1, S, d)
    out, lse = oracle.na3d_attention(q, k, v, grid, (1, 1, 1), 0.3)
    np.testing.assert_array_equal(out, v)
    np.testing.assert_allclose(lse, 0.3 * np.einsum("bhsd,bhsd->bhs", q, k), rtol=0, atol=1e-13)


def test_na3d_full_window_equals_library_dense():
    grid = (3, 4, 5)
    S, d = 60, 32
    q, k, v = rand(1, 3, S, d), rand(1, 3, S, d), rand(1, 3, S, d)
    out, lse = oracle.na3d_attention(q, k, v, grid, grid, 0.2)
    np.testing.assert_allclose(out, sdpa64(q, k, v, 0.2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(0.2 * np.einsum("bhqd,bhkd->bhqk", q, k), axis=-1),
                               rtol=0, atol=1e-12)


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_na3d_mirror_symmetry_odd_window(axis):
    # an odd window is centred, so mirroring the volume along an axis mirrors the output
    grid, kernel = (5, 6, 7), (3, 3, 5)
    S, d = 210, 8
    q, k, v = rand(1, 1, S, d), rand(1, 1, S, d), rand(1, 1, S, d)
    flip = lambda a: np.flip(a.reshape(1, 1, *grid, -1), axis=2 + axis).reshape(1, 1, S, -1)
    out, lse = oracle.na3d_attention(q, k, v, grid, kernel, 0.5)
    fo, fl = oracle.na3d_attention(flip(q), flip(k), flip(v), grid, kernel, 0.5)
    np.testing.assert_allclose(flip(fo), out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(flip(fl[..., None])[..., 0], lse, rtol=0, atol=1e-13)


def test_na3d_row_subset_matches_full():
    grid, kernel = (3, 5, 6), (2, 3, 3)
    S, d = 90, 8
    q, k, v = rand(2, 2, S, d), rand(2, 2, S, d), rand(2, 2, S, d)
    out, lse = oracle.na3d_attention(q, k, v, grid, kernel, 0.4)
    rows = np.array([0, 17, 89, 90, 200, 359])
    ro, rl = oracle.na3d_attention(q, k, v, grid, kernel, 0.4, rows=rows)
    np.testing.assert_array_equal(ro, out.reshape(-1, d)[rows])
    np.testing.assert_array_equal(rl, lse.reshape(-1)[rows])


# ---------------------------------------------------------------- FP8 (E4M3) codec, quantiser and scaled product

def torch_e4m3_values(codes):
    """torch's own decoding of E4M3 codes (a library routine the oracle does not use)."""
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).float().double().numpy()


def test_e4m3_decode_matches_library_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours, lib = oracle.e4m3_decode(codes), torch_e4m3_values(codes)
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(lib))
    np.testing.assert_array_equal(ours[~np.isnan(ours)], lib[~np.isnan(lib)])
    assert np.isnan(ours[[0x7f, 0xff]]).all() and np.isnan(ours).sum() == 2
    assert ours[0x7e] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6 and ours[0x38] == 1.0


def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7f, 0xff)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(vals), codes)


def test_e4m3_encode_matches_library_conversion():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-0.02, 0.02, 20000),
                        np.exp(rng.uniform(-12, 6, 20000)) * rng.choice([-1, 1], 20000)]).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), lib)


def test_e4m3_encode_is_the_nearest_value_ties_to_even():
    # brute force: search the whole finite code table for the nearest value
    table_codes = np.array([c for c in range(128) if c != 0x7f], dtype=np.uint8)
    table = oracle.e4m3_decode(table_codes)
    rng = np.random.default_rng(6)
    mids = (table[:-1] + table[1:]) / 2                     # exact ties between neighbours
    v = np.concatenate([rng.uniform(0, 448, 3000), np.exp(rng.uniform(-14, 6, 3000)), mids]).astype(np.float32)
    v = v[v.astype(np.float64) <= 448]
    got = oracle.e4m3_encode(v)
    for x, g in zip(v.astype(np.float64), got):
        dist = np.abs(table - x)
        best = np.flatnonzero(dist == dist.min())
        if len(best) == 1:
            assert g == table_codes[best[0]], (x, g)
        else:                                               # a tie: the even code wins
            assert g == [table_codes[b] for b in best if table_codes[b] % 2 == 0][0], (x, g)
    # negative values mirror the positive ones with the sign bit
    np.testing.assert_array_equal(oracle.e4m3_encode(-v), got | 0x80)


def test_e4m3_encode_saturates():
    big = np.array([448.0, 449.0, 463.9, 464.0, 470.0, 479.9, 500.0, 1e6, 3.4e38], dtype=np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(big), 0x7e)
    np.testing.assert_array_equal(oracle.e4m3_encode(-big), 0xfe)


# Positive finite E4M3 values in code order (codes 0x00..0x7e are increasing), decoded by torch.
_E4M3_POS = [Fraction(float(v)) for v in torch_e4m3_values(np.arange(0x7f))]


def exact_e4m3_code(value: Fraction, negative: bool) -> int:
    """E4M3 code of an exact rational: the nearest value, ties to the even code, saturating at 448
    (a search over torch's decoding of the code table, in exact arithmetic)."""
    a = abs(value)
    sgn = 0x80 if negative else 0
    if a >= _E4M3_POS[-1]:
        return sgn | 0x7e
    hi = bisect.bisect_left(_E4M3_POS, a)
    if _E4M3_POS[hi] == a:
        return sgn | hi
    lo = hi - 1
    dlo, dhi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    if dlo != dhi:
        return sgn | (lo if dlo < dhi else hi)
    return sgn | (lo if lo % 2 == 0 else hi)


def exact_quantize_row(row):
    """The per-row quantiser's definition in exact rational arithmetic: s = amax / 448 (nearest
    float), codes nearest to x * 448 / amax.  Returns (codes, s, amax) for a row with a normal scale."""
    amax = max(abs(Fraction(float(x))) for x in row)
    codes = np.array([exact_e4m3_code(Fraction(float(x)) * 448 / amax, math.copysign(1.0, float(x)) < 0)
                      for x in row], dtype=np.uint8)
    return codes, np.float32(float(amax / 448)), amax


def near_midpoint_rows():
    """Rows whose values sit exactly on, or one float step either side of, the inputs whose exact
    quotient x * 448 / amax is an E4M3 rounding midpoint; each row holds its amax as the row max."""
    mids = [(a + b) / 2 for a, b in zip(_E4M3_POS[:-1], _E4M3_POS[1:])]
    rows = []
    for amax in (3.0, 5.0, 7.0, 11.0, 0.3, 1.7, 2.9, 6.1, 123.456, 0.0123, 1.1e-3, 37.5):
        a32 = np.float32(amax)
        row = [a32]
        for m in mids[::3]:
            t = np.float32(float(m * Fraction(float(a32)) / 448))
            for c in (np.nextafter(t, np.float32(-np.inf)), t, np.nextafter(t, np.float32(np.inf))):
                if 0 < c < a32:
                    row += [c, -c]
        rows.append(np.array(row, dtype=np.float32))
    return rows


def test_quantize_rows_codes_are_the_exact_quotients_nearest_value():
    """Codes against the definition in exact rational arithmetic, on inputs placed next to rounding
    midpoints: there a float-rounded scale or inverse scale would move the quotient across the
    midpoint, so this separates the exact quotient from single-precision shortcuts."""
    rows = near_midpoint_rows()
    n_product_differs = n_quotient_differs = 0
    for row in rows:
        q, s = oracle.fp8_quantize_rows(row[None, :])
        codes, s_exact, amax = exact_quantize_row(row)
        assert s[0] == s_exact
        np.testing.assert_array_equal(q[0], codes)
        # how often the two single-precision shortcuts would decide otherwise (the pin must see some)
        a32 = np.float32(float(amax))
        inv32 = np.float32(448.0) / a32
        for x, c in zip(row, codes):
            by_product = exact_e4m3_code(Fraction(float(np.float32(x * inv32))), x < 0)
            by_quotient = exact_e4m3_code(Fraction(float(np.float32(x / s_exact))), x < 0)
            n_product_differs += by_product != c
            n_quotient_differs += by_quotient != c
    assert n_product_differs >= 5 and n_quotient_differs >= 5, (n_product_differs, n_quotient_differs)


def test_quantize_rows_error_bound_and_row_max():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((37, 300)).astype(np.float32) * np.exp(rng.uniform(-8, 8, (37, 1))).astype(np.float32)
    x[3] = 0.0                                             # a row of zeros
    x[4, :] = 0.0
    x[4, 17] = -2.5                                        # a single non-zero
    x[6] = torch.from_numpy(x[6]).bfloat16().float().numpy()     # bf16 values, as the GPU's inputs are
    q, s = oracle.fp8_quantize_rows(x)
    dq = oracle.e4m3_decode(q) * s[:, None].astype(np.float64)
    amax = np.abs(x).max(axis=1)
    for m in range(x.shape[0]):
        if amax[m] == 0:
            assert s[m] == 0 and (q[m] == 0).all()
            continue
        # the definition in exact arithmetic: scale = amax / 448 (nearest float), codes nearest to x * 448 / amax
        codes, s_exact, _ = exact_quantize_row(x[m])
        assert s[m] == s_exact
        np.testing.assert_array_equal(q[m], codes)
        # and against torch's float -> E4M3 conversion of the quotient (in double, then to float: no value
        # of this row lies next to a midpoint)
        lib = torch.from_numpy(x[m].astype(np.float64) * 448.0 / float(amax[m])).float().clamp(-448, 448)
        np.testing.assert_array_equal(q[m], lib.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        j = int(np.argmax(np.abs(x[m])))
        assert q[m, j] & 0x7f == 0x7e
        # relative error <= 2^-4 for normal codes, absolute <= scale * 2^-10 on the subnormal grid (+ the
        # rounding of the scale to float)
        err = np.abs(dq[m] - x[m].astype(np.float64))
        bound = np.maximum(np.abs(x[m]) * 2.0 ** -4, s[m] * 2.0 ** -10) * (1 + 1e-6)
        assert (err <= bound).all()
    # a row whose scale amax / 448 is below the smallest normal float (2^-126) is treated as zero;
    # one just above it is quantised
    tiny = np.zeros((3, 32), dtype=np.float32)
    tiny[0, 5] = np.float32(1e-39)
    tiny[1, 5] = np.float32(448 * 2.0 ** -126 * 0.999)
    tiny[2, 5], tiny[2, 6] = np.float32(448 * 2.0 ** -126 * 1.001), np.float32(448 * 2.0 ** -126 * 0.3)
    tq, ts = oracle.fp8_quantize_rows(tiny)
    assert ts[0] == 0 and ts[1] == 0 and (tq[:2] == 0).all()
    assert ts[2] >= np.float32(2.0 ** -126) and tq[2, 5] == 0x7e and tq[2, 6] == exact_quantize_row(tiny[2])[0][6]
    # the lone non-zero is the row max: code -448, dequantised to -448 * fl32(2.5 / 448)
    assert q[4, 17] == 0xfe and dq[4, 17] == -448.0 * float(s[4]) and abs(dq[4, 17] + 2.5) < 2.5 * 2.0 ** -23
    assert (q[4, np.arange(300) != 17] == 0).all()


def test_fp8_gemm_matches_library_matmul_of_decoded_operands():
    rng = np.random.default_rng(8)
    M, N, K = 23, 41, 96
    aq = rng.integers(0, 256, (M, K), dtype=np.uint8)
    wq = rng.integers(0, 256, (N, K), dtype=np.uint8)
    aq[(aq & 0x7f) == 0x7f] = 0x10                          # no NaN codes
    wq[(wq & 0x7f) == 0x7f] = 0x22
    sa = rng.uniform(0.01, 2.0, M).astype(np.float32)
    sw = rng.uniform(0.01, 2.0, N).astype(np.float32)
    y, ya = oracle.fp8_gemm(aq, sa, wq, sw)
    A, W = torch_e4m3_values(aq), torch_e4m3_values(wq)
    ref = (sa[:, None].astype(np.float64) * (A @ W.T)) * sw[None, :].astype(np.float64)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    np.testing.assert_allclose(ya, np.abs(sa)[:, None] * (np.abs(A) @ np.abs(W).T) * np.abs(sw)[None, :],
                               rtol=1e-12)


def test_fp8_gemm_identity_weight_returns_dequantised_rows():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((9, 32)).astype(np.float32)
    q, s = oracle.fp8_quantize_rows(x)
    eye = np.where(np.eye(32, dtype=bool), np.uint8(0x38), np.uint8(0))   # 0x38 = 1.0
    y, _ = oracle.fp8_gemm(q, s, eye, np.ones(32, dtype=np.float32))
    np.testing.assert_array_equal(y, oracle.e4m3_decode(q) * s[:, None].astype(np.float64))
