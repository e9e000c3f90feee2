"""attn_sparse_route_fwd_noalloc: the allocation-free variant of the block-sparse path.

It serves callers that may not allocate device memory on this path (a host
framework that owns every allocation, or a latency-critical thread that must
not stall on cudaMalloc): the scratch comes from one fixed device array inside
the library.  Checked here through the C ABI against the regular entry point
(caller-provided workspace), bit for bit, on calls in a row of different sizes,
so each call runs on whatever the one before left in the shared scratch.  This
file is collected last on purpose.
"""
import ctypes
import math

import pytest
import torch

import video_diffusion_transformer_block_gb300 as vd
from workloads import Workload, make_qkv

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _regular(lib, q, k, v, beta, block, scale, stream):
    B, H, S, d = q.shape
    nbytes = lib.attn_sparse_workspace_bytes(B, H, S, d, block, block)
    ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    st = lib.attn_sparse_route_fwd(_p(q), _p(k), _p(v), _p(out), _p(lse), B, H, S, d, scale, beta, block, block,
                                   _p(ws), nbytes, None, None, None, None, stream)
    assert st == 0, vd.attn_status_string(st)
    return out, lse


def _noalloc(lib, q, k, v, beta, block, scale, stream):
    B, H, S, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    st = lib.attn_sparse_route_fwd_noalloc(_p(q), _p(k), _p(v), _p(out), _p(lse), B, H, S, d, scale, beta, block,
                                           block, stream)
    assert st == 0, vd.attn_status_string(st)
    return out, lse


def test_noalloc_matches_regular_entry_point_on_two_calls_in_a_row():
    lib = vd.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    large = (Workload("na1", B=1, H=4, Sq=4000, Skv=4000, d=128, seed=61, q_std=0.5, k_std=0.5,
                      grid=(16, 64, 64), audio_per_frame=8, pe=True), 1.0, 128)
    small = (Workload("na2", B=2, H=2, Sq=1024, Skv=1024, d=64, seed=62), 0.5, 64)
    # the calls run back to back on the shared scratch: the small case on what the large one left, then the
    # large case again on what both left.  The kernels are deterministic, so any read of a stale scratch
    # byte would show as a difference from the regular entry point, which gets a fresh workspace.
    for w, beta, block in (large, small, large):
        q, k, v = make_qkv(w, device="cuda")
        scale = 1.0 / math.sqrt(w.d)
        need = lib.attn_sparse_workspace_bytes(w.B, w.H, w.Sq, w.d, block, block)
        assert 0 < need <= vd.NOALLOC_WORKSPACE_BYTES
        ref_out, ref_lse = _regular(lib, q, k, v, beta, block, scale, stream)
        out, lse = _noalloc(lib, q, k, v, beta, block, scale, stream)
        torch.cuda.synchronize()
        assert vd.attn_last_device_status() == 0
        assert torch.equal(out, ref_out), f"{w.name}: out differs from the regular entry point"
        assert torch.equal(lse, ref_lse), f"{w.name}: lse differs from the regular entry point"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = vd.load_library()
    # the full Stage-2 size (H=32, S=65664) needs ~68 MB of scratch: rejected before any launch
    assert lib.attn_sparse_workspace_bytes(1, 32, 65664, 128, 128, 128) > vd.NOALLOC_WORKSPACE_BYTES
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = lib.attn_sparse_route_fwd_noalloc(_p(dummy), _p(dummy), _p(dummy), _p(dummy), None, 1, 32, 65664, 128,
                                           0.088, 1.0, 128, 128, None)
    assert st == 3, vd.attn_status_string(st)
