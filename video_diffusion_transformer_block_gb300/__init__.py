"""GB300 (sm_103a) attention hot path of an LTX-2.5-style video+audio DiT block.

Thin Python binding over the C ABI in ``include/attn_api.h`` (library
``libvdtb_attn.so`` built in-tree by :mod:`.build`).  Every function here has
the name of the C entry point it calls and only marshals arguments: torch
provides device memory and the current CUDA stream, the kernels do all the
work.  There is no fallback: if the library is missing or fails to load,
every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = [
    "AttnError", "load_library", "attn_dense_fwd", "attn_cross_splitkv_fwd", "attn_lse_merge", "attn_block_pool",
    "attn_sparse_workspace_bytes", "attn_sparse_route_fwd", "attn_sparse_route", "attn_sparse_fwd",
    "attn_last_device_status", "attn_status_string", "attn_selftest_wait_timeout", "attn_selftest_wait_timeout_grid",
    "attn_sparse_route_fwd_noalloc", "attn_sparse_fused_fwd", "attn_na3d_fwd", "attn_na3d_plan",
    "fp8_quantize_rows", "fp8_scaled_gemm", "fp8_linear", "attn_cross_fwd", "attn_cross_workspace_bytes",
    "NOALLOC_WORKSPACE_BYTES", "EXPORTED_SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libvdtb_attn.so")
_lock = threading.Lock()
_lib = None

EXPORTED_SYMBOLS = (
    "attn_dense_fwd", "attn_cross_splitkv_fwd", "attn_lse_merge", "attn_block_pool", "attn_sparse_workspace_bytes",
    "attn_sparse_route_fwd", "attn_sparse_route", "attn_sparse_fwd", "attn_last_device_status", "attn_status_string",
    "attn_selftest_wait_timeout", "attn_selftest_wait_timeout_grid", "attn_sparse_route_fwd_noalloc",
    "attn_sparse_fused_fwd", "attn_na3d_fwd", "attn_na3d_plan", "fp8_quantize_rows", "fp8_scaled_gemm",
    "attn_cross_fwd", "attn_cross_workspace_bytes",
)

# Size of the library-owned scratch of attn_sparse_route_fwd_noalloc (ATTN_NOALLOC_WORKSPACE_BYTES).
NOALLOC_WORKSPACE_BYTES = 32 << 20

_STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_WORKSPACE",
           4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_TIMEOUT"}


class AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {_STATUS.get(code, code)}")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libvdtb_attn.so (built by ``build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build the CUDA library first "
                               "(python -m video_diffusion_transformer_block_gb300.build)")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_dense_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        lib.attn_cross_splitkv_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
        lib.attn_lse_merge.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
        lib.attn_block_pool.argtypes = [vp, vp, i, i, i, i, i, vp]
        lib.attn_sparse_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.attn_sparse_workspace_bytes.restype = sz
        lib.attn_sparse_route_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, f, i, i, vp, sz, vp, vp, vp, vp, vp]
        lib.attn_sparse_route.argtypes = [vp, vp, vp, i, i, i, i, f, f, i, i, vp, sz, vp, vp, vp, vp, vp, vp]
        lib.attn_sparse_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, vp, vp, vp, vp, vp]
        lib.attn_sparse_route_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, f, i, i, vp]
        lib.attn_sparse_fused_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, f, i, i, vp, sz, vp, vp, vp, vp, vp]
        lib.attn_na3d_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i, i, vp]
        ip, llp = ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_longlong)
        lib.attn_na3d_plan.argtypes = [i, i, i, i, i, i, ip, ip, llp]
        lib.attn_cross_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.attn_cross_workspace_bytes.restype = sz
        lib.attn_cross_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz, vp]
        lib.fp8_quantize_rows.argtypes = [vp, vp, vp, i, i, vp]
        lib.fp8_scaled_gemm.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
        lib.attn_last_device_status.argtypes = [vp]
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_selftest_wait_timeout.argtypes = [i, vp]
        lib.attn_selftest_wait_timeout_grid.argtypes = [i, i, vp]
        for name in ("attn_dense_fwd", "attn_cross_splitkv_fwd", "attn_lse_merge", "attn_block_pool",
                     "attn_sparse_route_fwd", "attn_sparse_route", "attn_sparse_fwd", "attn_last_device_status",
                     "attn_selftest_wait_timeout", "attn_selftest_wait_timeout_grid", "attn_sparse_route_fwd_noalloc",
                     "attn_sparse_fused_fwd",
                     "attn_na3d_fwd", "attn_na3d_plan", "fp8_quantize_rows", "fp8_scaled_gemm", "attn_cross_fwd"):
            getattr(lib, name).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(fn: str, code: int):
    if code != 0:
        raise AttnError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _bhsd(x: torch.Tensor, name: str):
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 4 or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [B, H, S, d]")
    return x.shape


def attn_status_string(code: int) -> str:
    return load_library().attn_status_string(int(code)).decode()


def attn_dense_fwd(q, k, v, scale=None, out=None, lse=None, stream=None):
    """Dense attention; returns (out bf16 [B,H,Sq,d], lse fp32 [B,H,Sq])."""
    lib = load_library()
    B, H, Sq, d = _bhsd(q, "q")
    Skv = _bhsd(k, "k")[2]
    _bhsd(v, "v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("attn_dense_fwd", lib.attn_dense_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Sq, Skv, d,
                                                scale, _stream(stream)))
    return out, lse


def attn_na3d_plan(grid, kernel, brick=0, pair_axis=-1):
    """Tile plan of attn_na3d_fwd: (brick, pair_axis, key boxes multiplied per head).  Host only."""
    lib = load_library()
    b, pa, nb = ctypes.c_int(int(brick)), ctypes.c_int(int(pair_axis)), ctypes.c_longlong(0)
    T, Y, X = (int(g) for g in grid)
    Kt, Ky, Kx = (int(g) for g in kernel)
    _check("attn_na3d_plan", lib.attn_na3d_plan(T, Y, X, Kt, Ky, Kx, ctypes.byref(b), ctypes.byref(pa),
                                                ctypes.byref(nb)))
    return b.value, pa.value, nb.value


def attn_na3d_fwd(q, k, v, grid, kernel, scale=None, brick=0, pair_axis=-1, out=None, lse=None, stream=None):
    """3D neighbourhood attention over a (T, Y, X) volume of raster-ordered tokens;
    returns (out bf16 [B,H,S,d], lse fp32 [B,H,S]).  brick / pair_axis: 0 / -1 let
    the library choose the tile plan (attn_na3d_plan); pair_axis 4 is the
    persistent one-brick plan, 5 the same with 4x2x16 key boxes (4x4x8 brick
    only), 6 plan 5 with E5M2 window operands (never chosen by the library:
    exact for raw scores |q.k| < 2^30, and run as plan 5 when scale * log2(e)
    < 2^-22), 3 one brick per CTA, 0-2 two neighbouring bricks per CTA."""
    lib = load_library()
    B, H, S, d = _bhsd(q, "q")
    if _bhsd(k, "k") != q.shape or _bhsd(v, "v") != q.shape:
        raise ValueError("q, k and v must have the same shape")
    T, Y, X = (int(g) for g in grid)
    Kt, Ky, Kx = (int(g) for g in kernel)
    if T * Y * X != S:
        raise ValueError("grid does not match the sequence length")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("attn_na3d_fwd", lib.attn_na3d_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, T, Y, X, d,
                                              Kt, Ky, Kx, scale, int(brick), int(pair_axis), _stream(stream)))
    return out, lse


def _matrix(x, name, dtype):
    if x.dtype != dtype or not x.is_cuda or x.dim() != 2 or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} matrix")
    return x.shape


def fp8_quantize_rows(x, q=None, scale=None, stream=None):
    """Per-row E4M3 quantisation of a bf16 matrix [M, K]: (codes uint8 [M, K], scale fp32 [M])."""
    lib = load_library()
    M, K = _matrix(x, "x", torch.bfloat16)
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
    scale = torch.empty(M, dtype=torch.float32, device=x.device) if scale is None else scale
    _check("fp8_quantize_rows", lib.fp8_quantize_rows(_ptr(x), _ptr(q), _ptr(scale), M, K, _stream(stream)))
    return q, scale


def fp8_scaled_gemm(aq, a_scale, wq, w_scale, y=None, stream=None):
    """y [M, N] bf16 = diag(a_scale) (aq wq^T) diag(w_scale); aq [M, K], wq [N, K] E4M3 codes (uint8)."""
    lib = load_library()
    M, K = _matrix(aq, "aq", torch.uint8)
    N, K2 = _matrix(wq, "wq", torch.uint8)
    if K2 != K or a_scale.shape != (M,) or w_scale.shape != (N,):
        raise ValueError("shape mismatch")
    if a_scale.dtype != torch.float32 or w_scale.dtype != torch.float32:
        raise ValueError("scales must be float32")
    y = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device) if y is None else y
    _check("fp8_scaled_gemm", lib.fp8_scaled_gemm(_ptr(aq), _ptr(a_scale), _ptr(wq), _ptr(w_scale), _ptr(y), M, N, K,
                                                  _stream(stream)))
    return y


def fp8_linear(x, wq, w_scale, stream=None):
    """y = x W^T with W held in FP8 (wq, w_scale) and x quantised per row on the fly."""
    aq, sa = fp8_quantize_rows(x, stream=stream)
    return fp8_scaled_gemm(aq, sa, wq, w_scale, stream=stream)


def attn_cross_splitkv_fwd(q, k, v, n_split, scale=None, out_part=None, lse_part=None, stream=None):
    """Split-KV partials; returns (out_part fp32 [n,B,H,Sq,d], lse_part fp32 [n,B,H,Sq])."""
    lib = load_library()
    B, H, Sq, d = _bhsd(q, "q")
    Skv = _bhsd(k, "k")[2]
    _bhsd(v, "v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out_part is None:
        out_part = torch.empty((n_split, B, H, Sq, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((n_split, B, H, Sq), dtype=torch.float32, device=q.device)
    _check("attn_cross_splitkv_fwd",
           lib.attn_cross_splitkv_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out_part), _ptr(lse_part), B, H, Sq, Skv, d,
                                      int(n_split), scale, _stream(stream)))
    return out_part, lse_part


def attn_cross_workspace_bytes(B, H, Sq, d, n_split) -> int:
    return int(load_library().attn_cross_workspace_bytes(B, H, Sq, d, n_split))


def attn_cross_fwd(q, k, v, n_split, scale=None, out=None, lse=None, workspace=None, stream=None):
    """Split-KV attention with the exact merge fused into the split kernel's tail (one launch);
    returns (out bf16 [B,H,Sq,d], lse fp32 [B,H,Sq]).  ``workspace``: a uint8 device tensor of at
    least attn_cross_workspace_bytes, zero-filled before its first use (a fresh zeroed one is made
    when omitted); calls leave it ready for the next call."""
    lib = load_library()
    B, H, Sq, d = _bhsd(q, "q")
    Skv = _bhsd(k, "k")[2]
    _bhsd(v, "v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    need = attn_cross_workspace_bytes(B, H, Sq, d, n_split)
    workspace = torch.zeros(max(need, 1), dtype=torch.uint8, device=q.device) if workspace is None else workspace
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("attn_cross_fwd", lib.attn_cross_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Sq, Skv, d,
                                                int(n_split), scale, _ptr(workspace),
                                                workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def attn_lse_merge(out_part, lse_part, out=None, lse=None, stream=None):
    """Merge partials; returns (out bf16 [B,H,Sq,d], lse fp32 [B,H,Sq])."""
    lib = load_library()
    n, B, H, Sq, d = out_part.shape
    if out is None:
        out = torch.empty((B, H, Sq, d), dtype=torch.bfloat16, device=out_part.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=out_part.device)
    _check("attn_lse_merge", lib.attn_lse_merge(_ptr(out_part), _ptr(lse_part), _ptr(out), _ptr(lse), n, B, H, Sq, d,
                                                _stream(stream)))
    return out, lse


def attn_block_pool(x, block, x_pool=None, stream=None):
    """Block mean-pool; returns fp32 [B,H,ceil(S/block),d]."""
    lib = load_library()
    B, H, S, d = _bhsd(x, "x")
    nb = (S + block - 1) // block
    if x_pool is None:
        x_pool = torch.empty((B, H, nb, d), dtype=torch.float32, device=x.device)
    _check("attn_block_pool", lib.attn_block_pool(_ptr(x), _ptr(x_pool), B, H, S, d, int(block), _stream(stream)))
    return x_pool


def attn_sparse_workspace_bytes(B, H, S, d, block_q, block_k) -> int:
    return int(load_library().attn_sparse_workspace_bytes(B, H, S, d, block_q, block_k))


def attn_sparse_route_fwd(q, k, v, beta, block=128, scale=None, out=None, lse=None, workspace=None, route=False,
                          stream=None):
    """Sol-Attn block-sparse attention (pool + route + sparse forward).

    Returns (out, lse) or, with route=True, (out, lse, dict(sel_idx, sel_cnt,
    stats, taylor_t)) with the routing results as device tensors."""
    lib = load_library()
    B, H, S, d = _bhsd(q, "q")
    _bhsd(k, "k")
    _bhsd(v, "v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = attn_sparse_workspace_bytes(B, H, S, d, block, block)
    if nbytes == 0:
        raise AttnError("attn_sparse_workspace_bytes", 2)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    extra = sparse_route_buffers(B, H, S, d, block, q.device) if route else {}
    _check("attn_sparse_route_fwd",
           lib.attn_sparse_route_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S, d, scale, float(beta),
                                     block, block, _ptr(workspace), workspace.numel(), _ptr(extra.get("sel_idx")),
                                     _ptr(extra.get("sel_cnt")), _ptr(extra.get("stats")),
                                     _ptr(extra.get("taylor_t")), _stream(stream)))
    return (out, lse, extra) if route else (out, lse)


def sparse_route_buffers(B, H, S, d, block, device, order=False):
    """Allocates (with torch) the routing outputs of attn_sparse_route for these sizes (with
    ``order`` and 128-token blocks also the query-block order the forward pairs its tiles by,
    which only attn_sparse_route writes: leave it out of a routing built by other means)."""
    nq = (S + block - 1) // block
    bufs = dict(sel_idx=torch.empty((B, H, nq, nq), dtype=torch.int32, device=device),
                sel_cnt=torch.empty((B, H, nq), dtype=torch.int32, device=device),
                stats=torch.empty((B, H, nq, 4), dtype=torch.float32, device=device),
                taylor_t=torch.empty((B, H, nq, d), dtype=torch.float32, device=device))
    if order and block == 128:
        bufs["qb_order"] = torch.empty((B, H, nq), dtype=torch.int32, device=device)
    return bufs


def attn_sparse_route(q, k, v, beta, block=128, scale=None, route=None, workspace=None, stream=None):
    """Pool + route only; returns the routing dict (sel_idx, sel_cnt, stats, taylor_t and, with
    128-token blocks, qb_order)."""
    lib = load_library()
    B, H, S, d = _bhsd(q, "q")
    _bhsd(k, "k")
    _bhsd(v, "v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    route = sparse_route_buffers(B, H, S, d, block, q.device, order=True) if route is None else route
    nbytes = attn_sparse_workspace_bytes(B, H, S, d, block, block)
    if nbytes == 0:
        raise AttnError("attn_sparse_workspace_bytes", 2)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check("attn_sparse_route",
           lib.attn_sparse_route(_ptr(q), _ptr(k), _ptr(v), B, H, S, d, scale, float(beta), block, block,
                                 _ptr(workspace), workspace.numel(), _ptr(route["sel_idx"]), _ptr(route["sel_cnt"]),
                                 _ptr(route["stats"]), _ptr(route["taylor_t"]), _ptr(route.get("qb_order")),
                                 _stream(stream)))
    return route


def attn_sparse_fwd(q, k, v, route, block=128, scale=None, out=None, lse=None, stream=None):
    """Block-sparse forward for a given routing; returns (out, lse)."""
    lib = load_library()
    B, H, S, d = _bhsd(q, "q")
    _bhsd(k, "k")
    _bhsd(v, "v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("attn_sparse_fwd",
           lib.attn_sparse_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S, d, scale, block, block,
                               _ptr(route["sel_idx"]), _ptr(route["sel_cnt"]), _ptr(route["stats"]),
                               _ptr(route["taylor_t"]), _ptr(route.get("qb_order")), _stream(stream)))
    return out, lse


def attn_sparse_fused_fwd(q, k, v, beta, block=128, scale=None, out=None, lse=None, workspace=None, route=False,
                          stream=None):
    """Sol-Attn block-sparse attention with the routing folded into the forward kernel.

    Same results as attn_sparse_route_fwd; with route=True the routing the
    kernel computed on chip is also copied out (dict as attn_sparse_route)."""
    lib = load_library()
    B, H, S, d = _bhsd(q, "q")
    _bhsd(k, "k")
    _bhsd(v, "v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = attn_sparse_workspace_bytes(B, H, S, d, block, block)
    if nbytes == 0:
        raise AttnError("attn_sparse_workspace_bytes", 2)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    extra = sparse_route_buffers(B, H, S, d, block, q.device) if route else {}
    _check("attn_sparse_fused_fwd",
           lib.attn_sparse_fused_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S, d, scale, float(beta),
                                     block, block, _ptr(workspace), workspace.numel(), _ptr(extra.get("sel_idx")),
                                     _ptr(extra.get("sel_cnt")), _ptr(extra.get("stats")),
                                     _ptr(extra.get("taylor_t")), _stream(stream)))
    return (out, lse, extra) if route else (out, lse)


def attn_sparse_route_fwd_noalloc(q, k, v, beta, block=128, scale=None, out=None, lse=None, stream=None):
    """attn_sparse_route_fwd with the library's own fixed device scratch, for callers that may
    not allocate device memory on this path (a host framework owning every allocation, or a
    latency-critical thread that must not stall on cudaMalloc).  Sizes needing more than
    NOALLOC_WORKSPACE_BYTES of scratch are rejected; calls that overlap on the GPU share the
    scratch and must be serialised by the caller.  (Outputs may still be allocated here by
    torch when not passed in; pass ``out``/``lse`` to allocate nothing at all.)"""
    lib = load_library()
    B, H, S, d = _bhsd(q, "q")
    _bhsd(k, "k")
    _bhsd(v, "v")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("attn_sparse_route_fwd_noalloc",
           lib.attn_sparse_route_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S, d, scale,
                                             float(beta), block, block, _stream(stream)))
    return out, lse


def attn_last_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(load_library().attn_last_device_status(_stream(stream)))


def attn_selftest_wait_timeout(limit_us: int, stream=None):
    _check("attn_selftest_wait_timeout", load_library().attn_selftest_wait_timeout(int(limit_us), _stream(stream)))


def attn_selftest_wait_timeout_grid(limit_us: int, n_ctas: int, stream=None):
    _check("attn_selftest_wait_timeout_grid",
           load_library().attn_selftest_wait_timeout_grid(int(limit_us), int(n_ctas), _stream(stream)))
