"""GPU parity of 3D neighbourhood attention against the fp64 oracle, through the C ABI.

Every output element of small volumes is compared: ragged volumes (bricks cut
by the borders), every brick shape and pair axis (and one brick per CTA), d = 64/128, B > 1, a single
frame, even windows, windows of one token and of the whole volume.
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


def check(B, H, grid, kernel, d, brick=0, pair=-1, seed=7, scale=None):
    q, k, v = na_inputs(B, H, grid, d, seed)
    scale = 1 / math.sqrt(d) if scale is None else scale
    out, lse = vd.attn_na3d_fwd(q, k, v, grid, kernel, scale=scale, brick=brick, pair_axis=pair)
    torch.cuda.synchronize()
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kernel, scale)
    tag = f"grid {grid} window {kernel} d {d} brick {brick} pair {pair}"
    assert_close(host(out), ro, f"na3d out ({tag})")
    assert_close(host(lse), rl, f"na3d lse ({tag})")
    return q, k, v, out, lse


@pytest.mark.parametrize("brick", [1, 2, 3])
@pytest.mark.parametrize("pair", [0, 1, 2, 3])
def test_na3d_every_plan_ragged_volume(brick, pair):
    check(1, 2, (5, 11, 19), (3, 5, 4), 64, brick, pair, seed=brick * 3 + pair)


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


def test_na3d_peaked_scores_rescale():
    # large scores: the running max moves by more than the lazy-rescale threshold between boxes
    check(1, 2, (4, 16, 32), (3, 9, 9), 128, scale=0.6, seed=5)
