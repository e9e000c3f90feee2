"""Every store stays inside its buffer.

The tools that would catch an out-of-bounds store on the GPU are closed on this
pool, so two substitutes check it on the ragged shapes where a tail tile could
write past the end of an output:

- guard bands: each output is allocated between two 4 KB bands of a fixed byte
  pattern (the output itself pre-filled with it too); after the call both bands
  must be unchanged, and the outputs must match the oracle (so every element
  was written);
- the bounds-checked build (libvdtb_attn_debug.so, compiled with -DATTN_DEBUG):
  every global store of every kernel checks its index against the buffer's
  extent and reports a store outside it through the status word instead of
  writing; on the same shapes it must report none and give the same bits as
  the regular library.
"""
import ctypes
import math
import os

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_block_gb300 as vd
from workloads import Workload, make_linear, LinearWorkload, make_qkv
from parity_util import Guarded, assert_close, host

pytestmark = pytest.mark.gpu

DEV = "cuda"


def rnd_qkv(B, H, Sq, Skv, d, seed):
    return make_qkv(Workload("g", B=B, H=H, Sq=Sq, Skv=Skv, d=d, seed=seed), device=DEV)


@pytest.fixture(autouse=True)
def _status_clean():
    torch.cuda.synchronize()
    yield
    assert vd.attn_last_device_status() == 0


@pytest.mark.parametrize("B,H,Sq,Skv,d", [(1, 2, 300, 517, 64), (2, 1, 1, 1, 128), (1, 1, 129, 1000, 128),
                                          (1, 3, 513, 255, 64)])
def test_dense_guard_bands(B, H, Sq, Skv, d):
    q, k, v = rnd_qkv(B, H, Sq, Skv, d, seed=Sq + Skv)
    out, lse = Guarded((B, H, Sq, d), torch.bfloat16), Guarded((B, H, Sq), torch.float32)
    vd.attn_dense_fwd(q, k, v, out=out.t, lse=lse.t)
    torch.cuda.synchronize()
    out.check("dense out")
    lse.check("dense lse")
    ro, rl = oracle.attention(host(q), host(k), host(v), 1 / math.sqrt(d))
    assert_close(host(out.t), ro, "dense out")
    assert_close(host(lse.t), rl, "dense lse")


@pytest.mark.parametrize("H,Sq,Skv,d,n", [(2, 130, 2000, 128, 3), (1, 128, 5, 128, 5), (2, 128, 4097, 128, 3),
                                          (1, 100, 1000, 64, 7)])
def test_splitkv_and_merge_guard_bands(H, Sq, Skv, d, n):
    q, k, v = rnd_qkv(1, H, Sq, Skv, d, seed=Sq + n)
    op, lp = Guarded((n, 1, H, Sq, d), torch.float32), Guarded((n, 1, H, Sq), torch.float32)
    out, lse = Guarded((1, H, Sq, d), torch.bfloat16), Guarded((1, H, Sq), torch.float32)
    vd.attn_cross_splitkv_fwd(q, k, v, n, out_part=op.t, lse_part=lp.t)
    vd.attn_lse_merge(op.t, lp.t, out=out.t, lse=lse.t)
    torch.cuda.synchronize()
    for g, what in ((op, "out_part"), (lp, "lse_part"), (out, "merged out"), (lse, "merged lse")):
        g.check(what)
    ro, rl = oracle.attention(host(q), host(k), host(v), 1 / math.sqrt(d))
    assert_close(host(out.t), ro, "merged out")
    assert_close(host(lse.t), rl, "merged lse")


@pytest.mark.parametrize("S,d,block,beta", [(100, 128, 128, 2.0), (1, 64, 64, 0.0), (1000, 64, 64, 0.5),
                                            (8208, 128, 128, 1.0)])
def test_sparse_guard_bands(S, d, block, beta):
    B, H = 1, 2
    q, k, v = rnd_qkv(B, H, S, S, d, seed=S)
    nq = (S + block - 1) // block
    rt = {"sel_idx": Guarded((B, H, nq, nq), torch.int32), "sel_cnt": Guarded((B, H, nq), torch.int32),
          "stats": Guarded((B, H, nq, 4), torch.float32), "taylor_t": Guarded((B, H, nq, d), torch.float32)}
    if block == 128:
        rt["qb_order"] = Guarded((B, H, nq), torch.int32)   # the query-block order the forward pairs tiles by
    ws = Guarded((vd.attn_sparse_workspace_bytes(B, H, S, d, block, block),), torch.uint8)
    out, lse = Guarded((B, H, S, d), torch.bfloat16), Guarded((B, H, S), torch.float32)
    route = {name: g.t for name, g in rt.items()}
    vd.attn_sparse_route(q, k, v, beta, block=block, route=route, workspace=ws.t)
    vd.attn_sparse_fwd(q, k, v, route, block=block, out=out.t, lse=lse.t)
    torch.cuda.synchronize()
    for name, g in rt.items():
        g.check(name)
    ws.check("workspace")
    out.check("sparse out")
    lse.check("sparse lse")
    # every element written: the outputs match the oracle evaluated on the GPU's own selection
    idx, cnt = route["sel_idx"].cpu().numpy(), route["sel_cnt"].cpu().numpy()
    sel = np.zeros(idx.shape, dtype=bool)
    for h in range(H):
        for i in range(nq):
            sel[0, h, i, idx[0, h, i, :cnt[0, h, i]]] = True
    qh, kh, vh = host(q), host(k), host(v)
    qp, kp, vp = (oracle.block_pool(x, block) for x in (qh, kh, vh))
    forced = oracle.route(qp, kp, vp, S, block, 1 / math.sqrt(d), beta, force_sel=sel)
    ro, rl = oracle.sparse_attention(qh, kh, vh, block, block, sel, forced["mu"], forced["W"], forced["T"],
                                     1 / math.sqrt(d))
    assert_close(host(out.t), ro, "sparse out")
    assert_close(host(lse.t), rl, "sparse lse")


@pytest.mark.parametrize("S,d,block,beta", [(1000, 128, 128, 0.5), (1000, 64, 64, 1.0)])
def test_fused_guard_bands(S, d, block, beta):
    B, H = 1, 2
    q, k, v = rnd_qkv(B, H, S, S, d, seed=S + 7)
    out, lse = Guarded((B, H, S, d), torch.bfloat16), Guarded((B, H, S), torch.float32)
    ws = Guarded((vd.attn_sparse_workspace_bytes(B, H, S, d, block, block),), torch.uint8)
    vd.attn_sparse_fused_fwd(q, k, v, beta, block=block, out=out.t, lse=lse.t, workspace=ws.t)
    torch.cuda.synchronize()
    out.check("fused out")
    lse.check("fused lse")
    ws.check("fused workspace")
    assert np.isfinite(host(out.t)).all() and np.abs(host(out.t)).max() < 1e3


@pytest.mark.parametrize("grid,kern", [((3, 13, 21), (3, 5, 7)), ((2, 7, 9), (1, 1, 1)), ((4, 9, 17), (3, 9, 17))])
def test_na3d_guard_bands(grid, kern):
    S = int(np.prod(grid))
    w = Workload("gna", B=1, H=2, Sq=S, Skv=S, d=128, seed=S, grid=grid, pe=True)
    q, k, v = make_qkv(w, device=DEV)
    out, lse = Guarded((1, 2, S, 128), torch.bfloat16), Guarded((1, 2, S), torch.float32)
    vd.attn_na3d_fwd(q, k, v, grid, kern, out=out.t, lse=lse.t)
    torch.cuda.synchronize()
    out.check("na3d out")
    lse.check("na3d lse")
    ro, rl = oracle.na3d_attention(host(q), host(k), host(v), grid, kern, w.scale)
    assert_close(host(out.t), ro, "na3d out")
    assert_close(host(lse.t), rl, "na3d lse")


@pytest.mark.parametrize("M,N,K", [(7, 8, 144), (129, 264, 4112), (1, 8, 16), (257, 512, 144)])
def test_fp8_guard_bands(M, N, K):
    x, W = make_linear(LinearWorkload("g", M=M, K=K, N=N, seed=M + N), device=DEV)
    aq, sa = Guarded((M, K), torch.uint8), Guarded((M,), torch.float32)
    wq, sw = Guarded((N, K), torch.uint8), Guarded((N,), torch.float32)
    y = Guarded((M, N), torch.bfloat16)
    vd.fp8_quantize_rows(x, q=aq.t, scale=sa.t)
    vd.fp8_quantize_rows(W, q=wq.t, scale=sw.t)
    vd.fp8_scaled_gemm(aq.t, sa.t, wq.t, sw.t, y=y.t)
    torch.cuda.synchronize()
    for g, what in ((aq, "codes"), (sa, "scales"), (wq, "weight codes"), (sw, "weight scales"), (y, "y")):
        g.check(what)
    rq, rs = oracle.fp8_quantize_rows(x.float().cpu().numpy())
    np.testing.assert_array_equal(aq.t.cpu().numpy(), rq)
    np.testing.assert_array_equal(sa.t.cpu().numpy(), rs)
    ry, ra = oracle.fp8_gemm(aq.t.cpu().numpy(), sa.t.cpu().numpy(), wq.t.cpu().numpy(), sw.t.cpu().numpy())
    g = y.t.float().cpu().double().numpy()
    assert (np.abs(g - ry) <= 2.0 ** -8 * np.abs(ry) + K * 2.0 ** -24 * ra + 1e-30).all()


# ---------------------------------------------------------------- the bounds-checked build

DEBUG_LIB = os.path.join(os.path.dirname(vd.__file__), "libvdtb_attn_debug.so")


@pytest.fixture(scope="module")
def dbg():
    if not os.path.exists(DEBUG_LIB):
        pytest.fail(f"{DEBUG_LIB} is missing: build() makes it next to the regular library")
    return vd.load_library(DEBUG_LIB)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def fresh(*shape, dtype=torch.float32, device=DEV):
    """An output buffer filled with the byte 0xA5: both libraries get the same
    contents wherever a call writes nothing (the entries of a selected-block
    row past its count, for one)."""
    t = torch.empty(*shape, dtype=dtype, device=device)
    t.view(torch.uint8).fill_(0xA5)
    return t


def test_bounds_checked_build_reports_nothing_and_matches(dbg):
    lib = vd.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def both(fn, make_outputs, make_args):
        """Runs C entry point `fn` of both libraries with fresh outputs; returns the two output lists."""
        res = []
        for L in (lib, dbg):
            outs = make_outputs()
            st = getattr(L, fn)(*[(_p(a) if isinstance(a, torch.Tensor) else a) for a in make_args(outs)], stream)
            assert st == 0, f"{fn}: {vd.attn_status_string(st)}"
            res.append(outs)
        torch.cuda.synchronize()
        assert dbg.attn_last_device_status(stream) == 0, f"{fn}: the bounds-checked build skipped a store"
        for a, b in zip(*res):
            assert torch.equal(a, b), f"{fn}: the bounds-checked build gives other results"
        return res[0]

    # dense, ragged query and key tails
    B, H, Sq, Skv, d = 1, 2, 300, 517, 64
    q, k, v = rnd_qkv(B, H, Sq, Skv, d, seed=5)
    both("attn_dense_fwd", lambda: [fresh(B, H, Sq, d, dtype=torch.bfloat16, device=DEV),
                                    fresh(B, H, Sq, device=DEV)],
         lambda o: [q, k, v, o[0], o[1], B, H, Sq, Skv, d, ctypes.c_float(1 / math.sqrt(d))])
    # split-KV partials of an odd key count, then the merge
    H, Sq, Skv, d, n = 2, 130, 2001, 128, 3
    q, k, v = rnd_qkv(1, H, Sq, Skv, d, seed=6)
    op, lp = both("attn_cross_splitkv_fwd", lambda: [fresh(n, 1, H, Sq, d, device=DEV),
                                                     fresh(n, 1, H, Sq, device=DEV)],
                  lambda o: [q, k, v, o[0], o[1], 1, H, Sq, Skv, d, n, ctypes.c_float(1 / math.sqrt(d))])
    both("attn_lse_merge", lambda: [fresh(1, H, Sq, d, dtype=torch.bfloat16, device=DEV),
                                    fresh(1, H, Sq, device=DEV)],
         lambda o: [op, lp, o[0], o[1], n, 1, H, Sq, d])
    # pool + route + block-sparse forward, ragged last block, with the routing outputs
    B, H, S, d, blk = 1, 2, 1000, 128, 128
    q, k, v = rnd_qkv(B, H, S, S, d, seed=7)
    nq = (S + blk - 1) // blk
    nbytes = lib.attn_sparse_workspace_bytes(B, H, S, d, blk, blk)
    both("attn_sparse_route_fwd",
         lambda: [fresh(B, H, S, d, dtype=torch.bfloat16, device=DEV), fresh(B, H, S, device=DEV),
                  torch.zeros(nbytes, dtype=torch.uint8, device=DEV),
                  fresh(B, H, nq, nq, dtype=torch.int32, device=DEV),
                  fresh(B, H, nq, dtype=torch.int32, device=DEV), fresh(B, H, nq, 4, device=DEV),
                  fresh(B, H, nq, d, device=DEV)],
         lambda o: [q, k, v, o[0], o[1], B, H, S, d, ctypes.c_float(1 / math.sqrt(d)), ctypes.c_float(0.5), blk, blk,
                    o[2], ctypes.c_size_t(nbytes), o[3], o[4], o[5], o[6]])
    # neighbourhood attention on a ragged volume
    T, Y, X = 3, 13, 21
    S = T * Y * X
    q, k, v = make_qkv(Workload("dna", B=1, H=2, Sq=S, Skv=S, d=128, seed=8, grid=(T, Y, X), pe=True), device=DEV)
    both("attn_na3d_fwd", lambda: [fresh(1, 2, S, 128, dtype=torch.bfloat16, device=DEV),
                                   fresh(1, 2, S, device=DEV)],
         lambda o: [q, k, v, o[0], o[1], 1, 2, T, Y, X, 128, 3, 5, 7, ctypes.c_float(1 / math.sqrt(128)), 0, -1])
    # FP8 quantiser and scaled product, ragged M and N, K not a multiple of 128
    M, N, K = 129, 264, 144
    x, W = make_linear(LinearWorkload("dfp8", M=M, K=K, N=N, seed=9), device=DEV)
    aq, sa = both("fp8_quantize_rows", lambda: [fresh(M, K, dtype=torch.uint8, device=DEV),
                                                fresh(M, device=DEV)], lambda o: [x, o[0], o[1], M, K])
    wq, sw = vd.fp8_quantize_rows(W)
    both("fp8_scaled_gemm", lambda: [fresh(M, N, dtype=torch.bfloat16, device=DEV)],
         lambda o: [aq, sa, wq, sw, o[0], M, N, K])
