"""fp64 CPU oracle for the LTX-2.5 attention hot path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never calls it and the
two share no code.  The arithmetic lives in ``oracle.c`` (plain C, double
precision); this module compiles it with gcc, loads it with ctypes and
marshals numpy arrays.  See the header of ``oracle.c`` for the definitions
and the sources they follow.

Parity status: dense attention, split-KV partials, the LSE merge, pooling,
proxy scores, mu/sigma/tau and the selection are pinned by closed forms,
library routines and invariants in ``tests/test_oracle_pins.py``.  The Taylor
aggregates (W, T) and the Taylor-corrected sparse output follow a reading
of the Sol-Attn page (first order about the row-mean proxy score,
applied per block with pooled V); they are pinned against exact softmax
attention in the small-deviation limit (the error must shrink as the square of
the score spread) and against a hand-derived closed form of that reading; the
pages' own block-level form is not printed, so parity is unpinned with respect
to the pages.  3D neighbourhood attention follows the published definition of
neighbourhood attention (the pages name the kernel but do not define it) and
is pinned by closed forms, an independent brute force and a mirror symmetry.
The FP8 (E4M3) codec, the per-row activation quantiser and the scaled FP8
product are pinned by torch's float8_e4m3fn conversion, a nearest-value search,
exact rational arithmetic (Python fractions) for the quantiser's codes, and
numpy's matmul.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into _oracle.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    lib.oracle_attend_rows.argtypes = [_D, _D, _D, _i64, _i64, _i64, _i64, ctypes.c_double, _I64, _i64, _D, _D]
    lib.oracle_split_partials.argtypes = [_D, _D, _D, _i64, _i64, _i64, _i64, ctypes.c_double, _i64, _D, _D]
    lib.oracle_lse_merge.argtypes = [_D, _D, _i64, _i64, _i64, _D, _D]
    lib.oracle_block_pool.argtypes = [_D, _i64, _i64, _i64, _i64, _D]
    lib.oracle_route.argtypes = [_D, _D, _D, _i64, _i64, _i64, _i64, _I64, ctypes.c_double, ctypes.c_double,
                                 ctypes.c_int, _U8, _D, _U8, _I64, _D, _D, _D, _D, _D, _I64]
    lib.oracle_sparse_rows.argtypes = [_D, _D, _D, _i64, _i64, _i64, _i64, _i64, _U8, _D, _D, _D,
                                       ctypes.c_double, _I64, _i64, _D, _D]
    lib.oracle_na3d_rows.argtypes = [_D, _D, _D, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_double,
                                     _I64, _i64, _D, _D]
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    _F = ctypes.POINTER(ctypes.c_float)
    lib.oracle_fp8_quantize_rows.argtypes = [_F, _i64, _i64, _U8, _F]
    lib.oracle_fp8_gemm.argtypes = [_U8, _F, _U8, _F, _i64, _i64, _i64, _D, _D]
    for f in (lib.oracle_attend_rows, lib.oracle_split_partials, lib.oracle_lse_merge, lib.oracle_block_pool,
              lib.oracle_route, lib.oracle_sparse_rows, lib.oracle_na3d_rows, lib.oracle_fp8_quantize_rows,
              lib.oracle_fp8_gemm):
        f.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


def _swap_library(path):
    """Test hook: route every oracle call through another build of oracle.c
    (used by the mutation tests, which plant mistakes in a copy).  Returns the
    previous library; pass None to restore the default build."""
    global _lib
    with _lock:
        prev = _lib
        _lib = None if path is None else _configure(ctypes.CDLL(path))
        return prev


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _bhsd(x):
    x = _f64(x)
    if x.ndim != 4:
        raise ValueError("expected a [B, H, S, d] array")
    return x


def attention(q, k, v, scale: float, rows=None):
    """Dense softmax attention.  q: [B,H,Sq,d], k/v: [B,H,Skv,d].

    rows=None evaluates every row and returns (out [B,H,Sq,d], lse [B,H,Sq]);
    otherwise ``rows`` holds flat row indices (b*H + h)*Sq + i and the result
    is (out [n, d], lse [n])."""
    q, k, v = _bhsd(q), _bhsd(k), _bhsd(v)
    B, H, Sq, d = q.shape
    Skv = k.shape[2]
    full = rows is None
    r = np.arange(B * H * Sq, dtype=np.int64) if full else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((r.size, d))
    lse = np.empty(r.size)
    _load().oracle_attend_rows(_p(q, _D), _p(k, _D), _p(v, _D), B * H, Sq, Skv, d, float(scale), _p(r, _I64),
                               r.size, _p(out, _D), _p(lse, _D))
    if full:
        return out.reshape(B, H, Sq, d), lse.reshape(B, H, Sq)
    return out, lse


def split_partials(q, k, v, scale: float, n_split: int):
    """Per-chunk partial answers: (o_part [n,B,H,Sq,d], lse_part [n,B,H,Sq])."""
    q, k, v = _bhsd(q), _bhsd(k), _bhsd(v)
    B, H, Sq, d = q.shape
    Skv = k.shape[2]
    o = np.empty((n_split, B, H, Sq, d))
    lse = np.empty((n_split, B, H, Sq))
    _load().oracle_split_partials(_p(q, _D), _p(k, _D), _p(v, _D), B * H, Sq, Skv, d, float(scale), n_split,
                                  _p(o, _D), _p(lse, _D))
    return o, lse


def lse_merge(o_part, lse_part):
    """Exact merge of partials: o_part [n,...,d], lse_part [n,...] -> (out, lse)."""
    o_part, lse_part = _f64(o_part), _f64(lse_part)
    n = o_part.shape[0]
    d = o_part.shape[-1]
    rows = int(np.prod(lse_part.shape[1:]))
    out = np.empty(lse_part.shape[1:] + (d,))
    lse = np.empty(lse_part.shape[1:])
    _load().oracle_lse_merge(_p(o_part, _D), _p(lse_part, _D), n, rows, d, _p(out, _D), _p(lse, _D))
    return out, lse


def block_pool(x, block: int):
    """Block mean-pool along S: [B,H,S,d] -> [B,H,ceil(S/block),d]."""
    x = _bhsd(x)
    B, H, S, d = x.shape
    nb = (S + block - 1) // block
    xp = np.empty((B, H, nb, d))
    _load().oracle_block_pool(_p(x, _D), B * H, S, d, block, _p(xp, _D))
    return xp


def route(qp, kp, vp, S: int, block_k: int, scale: float, beta: float, clamp: bool = True, force_sel=None):
    """Sol-Attn routing from pooled tensors qp [B,H,NQB,d], kp/vp [B,H,NKB,d].

    ``force_sel`` (bool [B,H,NQB,NKB]) replaces the threshold rule as the
    selection.  Returns a dict with proxy, sel (bool), sel_cnt, mu, sigma,
    tau, W, T and n_clamped."""
    qp, kp, vp = _bhsd(qp), _bhsd(kp), _bhsd(vp)
    B, H, NQB, d = qp.shape
    NKB = kp.shape[2]
    nk = np.array([min(block_k, S - j * block_k) for j in range(NKB)], dtype=np.int64)
    proxy = np.empty((B, H, NQB, NKB))
    sel = np.empty((B, H, NQB, NKB), dtype=np.uint8)
    cnt = np.empty((B, H, NQB), dtype=np.int64)
    mu, sigma, tau, W = (np.empty((B, H, NQB)) for _ in range(4))
    T = np.empty((B, H, NQB, d))
    ncl = np.zeros(1, dtype=np.int64)
    fs = None
    if force_sel is not None:
        fs = np.ascontiguousarray(force_sel, dtype=np.uint8)
        if fs.shape != (B, H, NQB, NKB):
            raise ValueError("force_sel shape")
    _load().oracle_route(_p(qp, _D), _p(kp, _D), _p(vp, _D), B * H, NQB, NKB, d, _p(nk, _I64), float(scale),
                         float(beta), 1 if clamp else 0, None if fs is None else _p(fs, _U8), _p(proxy, _D),
                         _p(sel, _U8), _p(cnt, _I64), _p(mu, _D),
                         _p(sigma, _D), _p(tau, _D), _p(W, _D), _p(T, _D), _p(ncl, _I64))
    return dict(proxy=proxy, sel=sel.astype(bool), sel_cnt=cnt, mu=mu, sigma=sigma, tau=tau, W=W, T=T,
                n_clamped=int(ncl[0]))


def sparse_attention(q, k, v, block_q: int, block_k: int, sel, mu, W, T, scale: float, rows=None):
    """Block-sparse attention with the Taylor term (self-attention, Sq = Skv = S).

    sel [B,H,NQB,NKB] bool, mu/W [B,H,NQB], T [B,H,NQB,d].  ``rows`` as in
    :func:`attention`."""
    q, k, v = _bhsd(q), _bhsd(k), _bhsd(v)
    B, H, S, d = q.shape
    sel8 = np.ascontiguousarray(sel, dtype=np.uint8)
    mu, W, T = _f64(mu), _f64(W), _f64(T)
    full = rows is None
    r = np.arange(B * H * S, dtype=np.int64) if full else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((r.size, d))
    lse = np.empty(r.size)
    _load().oracle_sparse_rows(_p(q, _D), _p(k, _D), _p(v, _D), B * H, S, d, block_q, block_k, _p(sel8, _U8),
                               _p(mu, _D), _p(W, _D), _p(T, _D), float(scale), _p(r, _I64), r.size, _p(out, _D),
                               _p(lse, _D))
    if full:
        return out.reshape(B, H, S, d), lse.reshape(B, H, S)
    return out, lse


def sparse_route_attention(q, k, v, block_q: int, block_k: int, scale: float, beta: float, rows=None):
    """The whole Sol-Attn path in the oracle: pool, route, sparse attention.

    Returns (out, lse, route_dict, pooled (qp, kp, vp))."""
    q, k, v = _bhsd(q), _bhsd(k), _bhsd(v)
    S = q.shape[2]
    qp, kp, vp = block_pool(q, block_q), block_pool(k, block_k), block_pool(v, block_k)
    rt = route(qp, kp, vp, S, block_k, scale, beta)
    out, lse = sparse_attention(q, k, v, block_q, block_k, rt["sel"], rt["mu"], rt["W"], rt["T"], scale, rows)
    return out, lse, rt, (qp, kp, vp)


def na3d_attention(q, k, v, grid, kernel, scale: float, rows=None):
    """3D neighbourhood attention.  q, k, v: [B,H,S,d] with S = T*Y*X tokens in
    raster order (t, y, x), x fastest; grid = (T, Y, X); kernel = (Kt, Ky, Kx)
    with 1 <= K <= L per axis.

    rows=None evaluates every row and returns (out [B,H,S,d], lse [B,H,S]);
    otherwise ``rows`` holds flat row indices (b*H + h)*S + i and the result is
    (out [n, d], lse [n])."""
    q, k, v = _bhsd(q), _bhsd(k), _bhsd(v)
    B, H, S, d = q.shape
    T, Y, X = (int(g) for g in grid)
    Kt, Ky, Kx = (int(g) for g in kernel)
    if T * Y * X != S or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("grid does not match the tensors")
    if not (1 <= Kt <= T and 1 <= Ky <= Y and 1 <= Kx <= X):
        raise ValueError("window must satisfy 1 <= K <= L on every axis")
    full = rows is None
    r = np.arange(B * H * S, dtype=np.int64) if full else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((r.size, d))
    lse = np.empty(r.size)
    _load().oracle_na3d_rows(_p(q, _D), _p(k, _D), _p(v, _D), B * H, T, Y, X, d, Kt, Ky, Kx, float(scale),
                             _p(r, _I64), r.size, _p(out, _D), _p(lse, _D))
    if full:
        return out.reshape(B, H, S, d), lse.reshape(B, H, S)
    return out, lse


def e4m3_decode(codes):
    """float64 values of E4M3 codes (any integer array of 0..255)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.vectorize(lambda x: lib.oracle_e4m3_decode(int(x)), otypes=[np.float64])(c) if c.size else \
        np.zeros(c.shape)


def e4m3_encode(values):
    """E4M3 codes (uint8) of values (taken as float64): nearest, ties to even, saturating at 448."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.vectorize(lambda x: lib.oracle_e4m3_encode(float(x)), otypes=[np.uint8])(v) if v.size else \
        np.zeros(v.shape, dtype=np.uint8)


def fp8_quantize_rows(x):
    """Per-row E4M3 quantisation of x [M, K] (float32 values): (codes uint8 [M, K], scale float32 [M]).

    scale[m] = amax_m / 448 (nearest float); codes are the E4M3 values nearest to the exact quotient
    x * 448 / amax_m, ties to even; rows whose scale is zero or not a normal float quantise to zeros."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if x.ndim != 2:
        raise ValueError("expected [M, K]")
    M, K = x.shape
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty(M, dtype=np.float32)
    _load().oracle_fp8_quantize_rows(_p(x, ctypes.POINTER(ctypes.c_float)), M, K, _p(q, _U8),
                                     _p(s, ctypes.POINTER(ctypes.c_float)))
    return q, s


def fp8_gemm(aq, sa, wq, sw):
    """y[m, n] = sa[m] sw[n] sum_k dec(aq[m, k]) dec(wq[n, k]) in float64, and the matching
    sum of absolute products (for error bounds).  aq [M, K], wq [N, K] uint8 codes."""
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = aq.shape
    N = wq.shape[0]
    if wq.shape[1] != K or sa.shape != (M,) or sw.shape != (N,):
        raise ValueError("shape mismatch")
    y = np.empty((M, N))
    ya = np.empty((M, N))
    F = ctypes.POINTER(ctypes.c_float)
    _load().oracle_fp8_gemm(_p(aq, _U8), _p(sa, F), _p(wq, _U8), _p(sw, F), M, N, K, _p(y, _D), _p(ya, _D))
    return y, ya
