"""GPU parity of 3D neighbourhood attention against the fp64 oracle, through the C ABI.

Every output element of small volumes is compared: ragged volumes (bricks cut
by the borders), every brick shape and pair axis (and one brick per CTA, and
the persistent one-brick tiles, also with several bricks per tile), d = 64/128,
B > 1, a single frame, even windows, windows of one token and of the whole volume.
Tolerances as for dense attention (max-abs 2e-2, relative L2 5e-3).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_block_gb300 as vd
from workloads import Workload, make_qkv
from parity_util import assert_close, host

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    torch.cuda.synchronize()
    yield
    assert vd.attn_last_device_status() == 0


def na_inputs(B, H, grid, d, seed, pe=True):
    S = int(np.prod(grid))
    w = Workload("na", B=B, H=H, Sq=S, Skv=S, d=d, seed=seed, grid=tuple(grid), pe=pe)
    return make_qkv(w, device="cuda")


# lse is computed in fp32 from fp32 scores and an fp32 row sum of unrounded
# probabilities: a few units in the sixth digit at most, while one key wrongly
# inside or outside a window of ~100 keys moves it by ~1e-2
LSE_ATOL = 1e-4


def check(B, H, grid, kernel, d, brick=0, pair=-1, seed=7, scale=None, out_max_abs=None):
    q, k, v = na_inputs(B, H, grid, d, seed)
    scale = 1 / math.sqrt(d) if scale is None else scale
    out, lse = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=brick, pair_axis=pair)
    torch.cuda.synchronize()
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
    tag = f"grid {grid} window {kernel} d {d} brick {brick} pair {pair}"
    if out_max_abs is None:
        assert_close(host(out), ro, f"na3d out ({tag})")
    else:
        assert_close(host(out), ro, f"na3d out ({tag})", max_abs=out_max_abs)
    assert_close(host(lse), rl, f"na3d lse ({tag})")
    np.testing.assert_allclose(host(lse), rl, atol=LSE_ATOL, rtol=0, err_msg=f"na3d lse ({tag})")
    return q, k, v, out, lse


@pytest.mark.parametrize("brick", [1, 2, 3])
@pytest.mark.parametrize("pair", [0, 1, 2, 3, 4, 5, 6])
def test_na3d_every_plan_ragged_volume(brick, pair):
    if pair in (5, 6) and brick != 3:
        pytest.skip("plans 5 and 6 take the 4x4x8 brick only")
    check(1, 2, (5, 11, 19), (3, 5, 4), 64, brick, pair, seed=brick * 3 + pair)


@pytest.mark.parametrize("grid,kernel,d", [
    ((1, 20, 24), (1, 9, 9), 128),     # one frame: 4-frame key boxes mostly outside the volume
    ((3, 13, 21), (3, 5, 7), 128),     # ragged in y and x, fewer frames than a key box
    ((6, 9, 10), (4, 2, 6), 64),       # even windows, several box rows
    ((4, 32, 32), (3, 31, 31), 128),   # a window wider than two key boxes
])
def test_na3d_wide_key_boxes(grid, kernel, d):
    # plan 5: 4x4x8 query bricks against 4x2x16 key boxes (the window step covers 4 frames, 2 rows
    # and 16 columns of a box)
    check(1, 2, grid, kernel, d, brick=3, pair=5, seed=19)


@pytest.mark.parametrize("B,H,grid,kernel,d", [
    (1, 2, (3, 13, 21), (3, 5, 7), 128),     # ragged in y and x, odd windows
    (2, 2, (4, 16, 32), (2, 7, 7), 128),     # whole bricks, B > 1
    (1, 2, (1, 20, 24), (1, 9, 9), 128),     # a single frame
    (1, 1, (6, 9, 10), (4, 2, 6), 64),       # even windows
    (1, 2, (4, 32, 32), (3, 31, 31), 128),   # large spatial window
    (1, 1, (2, 5, 6), (2, 5, 6), 128),       # the window is the whole volume (smaller than one brick)
])
def test_na3d_shapes(B, H, grid, kernel, d):
    check(B, H, grid, kernel, d)


def test_na3d_whole_volume_window_equals_dense():
    grid = (3, 16, 24)
    q, k, v, out, lse = check(1, 2, grid, grid, 128)
    dense, dlse = vd.attn_dense_fwd(q, k, v)
    torch.cuda.synchronize()
    assert_close(host(out), host(dense), "whole-volume window vs dense (GPU)")
    assert_close(host(lse), host(dlse), "whole-volume window lse vs dense (GPU)")


def test_na3d_single_token_window_returns_v():
    grid = (3, 9, 20)
    q, k, v = na_inputs(1, 2, grid, 128, seed=11)
    out, lse = vd.attn_na3d_fwd(q, k, v, grid, (1, 1, 1))
    torch.cuda.synchronize()
    assert torch.equal(out, v)
    expect = (q.float() * k.float()).sum(-1) / math.sqrt(128)
    torch.testing.assert_close(lse, expect, atol=1e-3, rtol=1e-4)


@pytest.mark.parametrize("pair", [-1, 3, 4, 5, 6])
def test_na3d_peaked_scores_rescale(pair):
    # large scores: the running max moves by more than the lazy-rescale threshold between boxes.
    # Each output is then close to one value row (|out| up to ~5), so the bf16 rounding of the
    # output (2^-8 |out|) and of the probabilities the PV product multiplies (2^-8 max|v|) bound
    # the error, not the fixed 2e-2 of flatter softmaxes; the lse bound is unchanged
    grid, kernel, d = (4, 16, 32), (3, 9, 9), 128
    q, k, v = na_inputs(1, 2, grid, d, 5)
    ro, _ = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, 0.6)
    bound = 2.0 ** -8 * (np.abs(ro).max() + np.abs(host(v)).max()) + 1e-3
    check(1, 2, grid, kernel, d, pair=pair, scale=0.6, seed=5, out_max_abs=bound)


def test_na3d_persistent_plan_tiny_scale_same_bits():
    # below scale * log2(e) = 2^-80 the window bias of the persistent plan could leave
    # masked keys a weight; the library then runs the one-brick CTAs, whose bits are the same
    grid, kernel = (3, 13, 21), (3, 5, 7)
    q, k, v = na_inputs(1, 2, grid, 128, seed=13)
    scale = 2.0 ** -90
    o4, l4 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=4)
    o5, l5 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=5)
    o3, l3 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=3)
    torch.cuda.synchronize()
    assert torch.equal(o4, o3) and torch.equal(l4, l3)
    assert torch.equal(o5, o3) and torch.equal(l5, l3)
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
    assert_close(host(o4), ro, "na3d tiny scale out")
    assert_close(host(l4), rl, "na3d tiny scale lse")


@pytest.mark.parametrize("brick,grid,kernel,H,d", [
    (3, (5, 37, 45), (3, 7, 7), 12, 128),   # 1440 bricks of 4x4x8, ragged in every axis
    (1, (3, 40, 50), (3, 5, 9), 16, 64),    # 960 bricks of 1x8x16
    (2, (6, 37, 45), (3, 7, 7), 8, 128),    # 720 bricks of 2x8x8; one window buffer per tile at d = 128
])
def test_na3d_persistent_tiles_walk_several_bricks(brick, grid, kernel, H, d):
    # plan 4: each tile of a persistent CTA runs bricks one after another (the
    # epilogue of one brick, the Q load of the next); enough bricks that every
    # tile takes several.  With one window buffer (2x8x8 at d = 128) the window
    # step runs first in each score MMA, which must not change a bit either
    B = {1: (1, 8, 16), 2: (2, 8, 8), 3: (4, 4, 8)}[brick]
    units = H * int(np.prod([-(-grid[a] // B[a]) for a in range(3)]))
    assert units > 2 * 2 * torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v = na_inputs(1, H, grid, d, seed=31 + brick)
    scale = 1 / math.sqrt(d)
    out4, lse4 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=brick, pair_axis=4)
    out3, lse3 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=brick, pair_axis=3)
    torch.cuda.synchronize()
    # the same boxes in the same order through the same arithmetic as the one-brick CTAs: identical bits
    assert torch.equal(out4, out3)
    assert torch.equal(lse4, lse3)
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
    assert_close(host(out4), ro, f"na3d persistent out (grid {grid} brick {brick})")
    assert_close(host(lse4), rl, f"na3d persistent lse (grid {grid} brick {brick})")


def test_na3d_wide_key_boxes_tiles_walk_several_bricks():
    # plan 5 with enough bricks (1440 of 4x4x8 over 12 heads) that every tile of a persistent CTA
    # takes several, ragged in every axis; checked against the oracle and against plan 4, whose
    # key boxes differ (so the two agree up to the rounding of the accumulation order)
    grid, kernel, H, d = (5, 37, 45), (3, 7, 7), 12, 128
    q, k, v = na_inputs(1, H, grid, d, seed=37)
    scale = 1 / math.sqrt(d)
    out5, lse5 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=5)
    out4, lse4 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=4)
    torch.cuda.synchronize()
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
    assert_close(host(out5), ro, "na3d wide key boxes out")
    assert_close(host(lse5), rl, "na3d wide key boxes lse")
    assert_close(host(out5), host(out4), "na3d plan 5 vs plan 4")
    torch.testing.assert_close(lse5, lse4, atol=1e-5, rtol=1e-5)


def test_na3d_persistent_output_16_byte_aligned():
    # the persistent plan writes whole 32-byte sectors when the output starts on a 32-byte
    # boundary and 16-byte pieces otherwise: an output 16 bytes past a boundary takes the second path
    grid, kernel, H, d = (3, 13, 21), (3, 5, 7), 2, 128
    S = int(np.prod(grid))
    q, k, v = na_inputs(1, H, grid, d, seed=17)
    buf = torch.empty(H * S * d + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(1, H, S, d)
    assert out.data_ptr() % 32 == 16
    vd.attn_na3d_fwd(q, k, v, grid, kernel, brick=3, pair_axis=4, out=out)
    o3, _ = vd.attn_na3d_fwd(q, k, v, grid, kernel, brick=3, pair_axis=3)
    torch.cuda.synchronize()
    assert torch.equal(out, o3)
    # plan 5 through the same two store paths: identical bits either way
    vd.attn_na3d_fwd(q, k, v, grid, kernel, brick=3, pair_axis=5, out=out)
    o5, _ = vd.attn_na3d_fwd(q, k, v, grid, kernel, brick=3, pair_axis=5)
    torch.cuda.synchronize()
    assert torch.equal(out, o5)


# Plan 6: plan 5's key boxes with the window added through E5M2 operands (-57344 per missed
# coordinate against one-hots of 57344).  Wherever both encodings are exact (raw scores
# |q.k| < 2^30, scale * log2(e) >= 2^-22) every in-window score is left unchanged and every
# other key gets an exact zero weight, with the same boxes in the same order: the bits of plan 5.

@pytest.mark.parametrize("grid,kernel,d,H", [
    ((1, 20, 24), (1, 9, 9), 128, 2),     # one frame: 4-frame key boxes mostly outside the volume
    ((3, 13, 21), (3, 5, 7), 128, 2),     # ragged in y and x
    ((6, 9, 10), (4, 2, 6), 64, 2),       # even windows, d = 64
    ((4, 32, 32), (3, 31, 31), 128, 2),   # a window wider than two key boxes
    ((5, 37, 45), (3, 7, 7), 128, 12),    # 1440 bricks: every tile of a persistent CTA takes several
])
def test_na3d_e5m2_window_same_bits_as_plan5(grid, kernel, d, H):
    q, k, v = na_inputs(1, H, grid, d, seed=41)
    scale = 1 / math.sqrt(d)
    o6, l6 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=6)
    o5, l5 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=5)
    torch.cuda.synchronize()
    assert torch.equal(o6, o5) and torch.equal(l6, l5)
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
    assert_close(host(o6), ro, f"na3d plan 6 out (grid {grid})")
    np.testing.assert_allclose(host(l6), rl, atol=LSE_ATOL, rtol=0, err_msg=f"na3d plan 6 lse (grid {grid})")


def test_na3d_e5m2_window_large_scores_same_bits():
    # raw scores of ~1e5 (inputs scaled by 40, softmax scale divided by 1600): still far inside
    # the E5M2 window's exact range, so plan 6 keeps plan 5's bits and both match the oracle
    grid, kernel, d = (4, 16, 32), (3, 9, 9), 128
    q, k, v = na_inputs(1, 2, grid, d, seed=43)
    q, k = (q.float() * 40).bfloat16(), (k.float() * 40).bfloat16()
    scale = 1 / (1600 * math.sqrt(d))
    raw = (q[0, 0].float() @ k[0, 0].float().T).abs().max().item()
    assert 1e4 < raw < 2.0 ** 30
    o6, l6 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=6)
    o5, l5 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=5)
    torch.cuda.synchronize()
    assert torch.equal(o6, o5) and torch.equal(l6, l5)
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
    assert_close(host(o6), ro, "na3d plan 6 large scores out")
    np.testing.assert_allclose(host(l6), rl, atol=LSE_ATOL, rtol=0, err_msg="na3d plan 6 large scores lse")


def test_na3d_e5m2_window_near_its_range_limit():
    # raw scores above 1e8, within a factor ~4 of the 2^30 the E5M2 window is exact for, at a
    # scale above its 2^-22 threshold (so plan 6 itself runs): keys outside a row's window still
    # get an exact zero weight and every in-window score is unchanged, i.e. plan 5's bits
    grid, kernel, d = (4, 16, 32), (3, 9, 9), 128
    q, k, v = na_inputs(1, 2, grid, d, seed=53)
    q, k = (q.float() * 1500).bfloat16(), (k.float() * 1500).bfloat16()
    raw = max((q[0, h].float() @ k[0, h].float().T).abs().max().item() for h in range(2))
    assert 1e8 < raw < 2.0 ** 30, raw
    scale = 2.0 ** -21
    assert scale * math.log2(math.e) >= 2.0 ** -22
    o6, l6 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=6)
    o5, l5 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=5)
    torch.cuda.synchronize()
    assert torch.equal(o6, o5) and torch.equal(l6, l5)
    # peaked softmax: the bf16 bound of the peaked-scores case; the lse within the fp32 accumulation
    # error of raw scores this large (128 products: ~128 * 2^-24 relative, ~1.2e-3 on logits up to 155)
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
    bound = 2.0 ** -8 * (np.abs(ro).max() + np.abs(host(v)).max()) + 1e-3
    assert np.abs(host(o6) - ro).max() <= bound
    np.testing.assert_allclose(host(l6), rl, rtol=0, atol=4e-3, err_msg="na3d plan 6 near range lse")


def test_na3d_e5m2_window_small_scale_falls_back():
    # below scale * log2(e) = 2^-22 the E5M2 bias no longer zeroes a key's weight for certain:
    # the library runs plan 5 (bf16 window) instead, below 2^-80 the one-brick CTAs
    grid, kernel = (3, 13, 21), (3, 5, 7)
    q, k, v = na_inputs(1, 2, grid, 128, seed=47)
    for scale, fallback in [(2.0 ** -30, 5), (2.0 ** -90, 3)]:
        o6, l6 = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=6)
        of, lf = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=3, pair_axis=fallback)
        torch.cuda.synchronize()
        assert torch.equal(o6, of) and torch.equal(l6, lf), scale
        ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
        assert_close(host(o6), ro, f"na3d plan 6 scale {scale} out")
        assert_close(host(l6), rl, f"na3d plan 6 scale {scale} lse")


def test_na3d_e5m2_window_output_16_byte_aligned():
    # plan 6 through the 16-byte store path: the same bits as through the 32-byte one
    grid, kernel, H, d = (3, 13, 21), (3, 5, 7), 2, 128
    S = int(np.prod(grid))
    q, k, v = na_inputs(1, H, grid, d, seed=17)
    buf = torch.empty(H * S * d + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(1, H, S, d)
    assert out.data_ptr() % 32 == 16
    vd.attn_na3d_fwd(q, k, v, grid, kernel, brick=3, pair_axis=6, out=out)
    o6, _ = vd.attn_na3d_fwd(q, k, v, grid, kernel, brick=3, pair_axis=6)
    torch.cuda.synchronize()
    assert torch.equal(out, o6)
