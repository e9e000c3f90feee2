"""Host-side checks of the C ABI (no GPU): the library loads, exports every
entry point the headers in include/ declare, and rejects invalid arguments
before touching the device."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import video_diffusion_transformer_block_gb300 as vd
from video_diffusion_transformer_block_gb300 import build as vbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    vbuild.build()
    return vd.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b((?:attn|fp8)_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(vd.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {vbuild.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} not exported"


def test_bounds_checked_library_exports_every_declared_symbol(lib):
    # built beside the regular library by build(), from the same sources with -DATTN_DEBUG
    assert os.path.exists(vbuild.DEBUG_LIB_PATH)
    out = os.popen(f"nm -D --defined-only {vbuild.DEBUG_LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} not exported by the bounds-checked build"


def test_status_strings(lib):
    for code, name in [(0, "ATTN_OK"), (1, "ATTN_ERR_INVALID_ARG"), (5, "ATTN_ERR_TIMEOUT"), (99, "ATTN_ERR_UNKNOWN")]:
        assert lib.attn_status_string(code).decode() == name


P = ctypes.c_void_p(0x1000)        # aligned, never dereferenced: validation fails before any device work
MIS = ctypes.c_void_p(0x1008)      # not 16-byte aligned
NULL = None


@pytest.mark.parametrize("args,code", [
    ((NULL, P, P, P, P, 1, 1, 16, 16, 128, 0.1), 1),            # null q
    ((P, P, P, MIS, P, 1, 1, 16, 16, 128, 0.1), 1),             # misaligned out
    ((P, P, P, P, P, 0, 1, 16, 16, 128, 0.1), 1),               # B = 0
    ((P, P, P, P, P, 1, 1, 0, 16, 128, 0.1), 1),                # Sq = 0
    ((P, P, P, P, P, 1, 1, 16, 16, 96, 0.1), 2),                # unsupported d
    ((P, P, P, P, P, 1, 1, 16, 16, 128, math.nan), 1),          # NaN scale
    ((P, P, P, P, P, 1, 1, 16, 16, 128, 0.0), 1),               # non-positive scale
    ((P, P, P, P, P, 1, 1, 16, 16, 128, -0.5), 1),
])
def test_dense_rejects_bad_arguments(lib, args, code):
    assert lib.attn_dense_fwd(*args, None) == code


def test_splitkv_rejects_bad_split(lib):
    assert lib.attn_cross_splitkv_fwd(P, P, P, P, P, 1, 1, 128, 10, 128, 11, 0.1, None) == 1
    assert lib.attn_cross_splitkv_fwd(P, P, P, P, P, 1, 1, 128, 10, 128, 0, 0.1, None) == 1


def test_merge_and_pool_reject(lib):
    assert lib.attn_lse_merge(P, P, P, P, 0, 1, 1, 8, 128, None) == 1
    assert lib.attn_lse_merge(P, P, MIS, P, 2, 1, 1, 8, 128, None) == 1
    assert lib.attn_block_pool(P, P, 1, 1, 100, 128, 96, None) == 2
    assert lib.attn_block_pool(NULL, P, 1, 1, 100, 128, 64, None) == 1


def test_sparse_workspace_and_rejections(lib):
    n = lib.attn_sparse_workspace_bytes(1, 32, 65664, 128, 128, 128)
    nq = 513
    nqp = (nq + 3) // 4 * 4
    # pooled q, k, v; lists; counts + stats; Taylor T; the query-block order; tf32 hi / lo of the pooled
    # keys and of the transposed pooled values (rows padded to a multiple of 4)
    expect_min = (32 * nq * 128 * 4 * 3 + 32 * nq * nq * 4 + 32 * nq * 4 * 5 + 32 * nq * 128 * 4 + 32 * nq * 4
                  + 2 * 32 * nq * 128 * 4 + 2 * 32 * 128 * nqp * 4)
    assert expect_min <= n <= expect_min + 12 * 256
    assert lib.attn_sparse_workspace_bytes(1, 1, 1000, 128, 64, 128) == 0      # block_q != block_k
    assert lib.attn_sparse_workspace_bytes(1, 1, 1000, 96, 64, 64) == 0        # bad d
    ws = ctypes.c_void_p(0x100000)
    args = [P, P, P, P, P, 1, 2, 1024, 64, 0.125, 0.5, 64, 64, ws, 0, None, None, None, None, None]
    assert lib.attn_sparse_route_fwd(*args) == 3                              # workspace too small
    args[10] = math.nan
    assert lib.attn_sparse_route_fwd(*args) == 1                              # NaN beta
    args[10], args[11] = 0.5, 32
    assert lib.attn_sparse_route_fwd(*args) == 2                              # unsupported block


def test_sparse_query_block_order_rejections(lib):
    # the order is for 128-token blocks only, and 4-byte aligned
    odd = ctypes.c_void_p(0x1002)
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 40
    route = [P, P, P, 1, 2, 1024, 64, 0.125, 0.5, 64, 64, ws, big, P, P, P, P]
    assert lib.attn_sparse_route(*route, P, None) == 1                      # order with 64-token blocks
    route[9], route[10] = 128, 128
    assert lib.attn_sparse_route(*route, odd, None) == 1                    # misaligned order
    fwd = [P, P, P, P, P, 1, 2, 1024, 64, 0.125, 64, 64, P, P, P, P]
    assert lib.attn_sparse_fwd(*fwd, P, None) == 1
    fwd[10], fwd[11] = 128, 128
    assert lib.attn_sparse_fwd(*fwd, odd, None) == 1


def test_selftest_rejects_bad_limit(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == 1
    assert lib.attn_selftest_wait_timeout(2_000_000, None) == 1


def test_fused_sparse_rejections(lib):
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 40
    # more than 1024 key blocks: the on-chip routing has no room for them
    assert lib.attn_sparse_fused_fwd(P, P, P, P, P, 1, 1, 1025 * 128, 128, 0.088, 1.0, 128, 128, ws, big,
                                     None, None, None, None, None) == 2
    assert lib.attn_sparse_fused_fwd(P, P, P, P, P, 1, 1, 4096, 128, 0.088, 1.0, 128, 128, ws, 0,
                                     None, None, None, None, None) == 3
    assert lib.attn_sparse_fused_fwd(P, P, P, P, P, 1, 1, 4096, 128, 0.088, math.inf, 128, 128, ws, big,
                                     None, None, None, None, None) == 1


# ---------------------------------------------------------------- 3D neighbourhood attention (host logic)

BRICKS = {1: (1, 8, 16), 2: (2, 8, 8), 3: (4, 4, 8)}
WIDE_KEYS = (4, 2, 16)   # the key boxes of plans 5 and 6 (with the 4x4x8 brick)


def key_box(brick, pair):
    return WIDE_KEYS if pair in (5, 6) else BRICKS[brick]


def na_start(p, K, L):
    return min(max(p - K // 2, 0), L - K)


def na_walk(grid, kernel, brick, pair):
    """Python restatement of the kernel's box walk: yields, per CTA, its query
    bricks (two neighbours along ``pair``, or one when pair is 3 to 6: plans
    4 to 6 run the one-brick tiles on persistent CTAs, plan 4 with the same
    boxes per brick, plans 5 and 6 with 4x2x16 key boxes) and the boxes with
    their tile flags."""
    B = BRICKS[brick]
    KB = key_box(brick, pair)
    nq = [-(-grid[a] // B[a]) for a in range(3)]
    np_ = [(-(-nq[a] // 2) if a == pair else nq[a]) for a in range(3)]
    for it in range(np_[0]):
        for iy in range(np_[1]):
            for ix in range(np_[2]):
                idx = [it, iy, ix]
                tiles = []
                for t in range(2 if pair < 3 else 1):
                    ib = [2 * idx[a] + t if a == pair else idx[a] for a in range(3)]
                    if pair < 3 and ib[pair] >= nq[pair]:
                        continue
                    org = [ib[a] * B[a] for a in range(3)]
                    lo = [na_start(org[a], kernel[a], grid[a]) for a in range(3)]
                    hi = [na_start(min(org[a] + B[a], grid[a]) - 1, kernel[a], grid[a]) + kernel[a] for a in range(3)]
                    tiles.append((org, lo, hi))
                cu = [min(tl[1][a] for tl in tiles) for a in range(3)]
                nk = [-(-(max(tl[2][a] for tl in tiles) - cu[a]) // KB[a]) for a in range(3)]
                boxes = []
                for ut in range(nk[0]):
                    for uy in range(nk[1]):
                        for ux in range(nk[2]):
                            box = [cu[0] + ut * KB[0], cu[1] + uy * KB[1], cu[2] + ux * KB[2]]
                            flags = [all(box[a] < tl[2][a] and box[a] + KB[a] > tl[1][a] for a in range(3))
                                     for tl in tiles]
                            if any(flags):
                                boxes.append((box, flags))
                yield tiles, boxes


@pytest.mark.parametrize("grid,kernel", [((3, 13, 21), (3, 5, 7)), ((5, 11, 19), (3, 5, 4)), ((1, 20, 24), (1, 9, 9)),
                                         ((4, 16, 32), (2, 16, 1)), ((2, 5, 6), (2, 5, 6))])
@pytest.mark.parametrize("brick", [1, 2, 3])
@pytest.mark.parametrize("pair", [0, 1, 2, 3, 4, 5, 6])
def test_na3d_walk_covers_every_window_and_plan_counts_it(lib, grid, kernel, brick, pair):
    if pair in (5, 6) and brick != 3:
        pytest.skip("plans 5 and 6 take the 4x4x8 brick only")
    B = BRICKS[brick]
    KB = key_box(brick, pair)
    work = 0
    for tiles, boxes in na_walk(grid, kernel, brick, pair):
        for t, (org, lo, hi) in enumerate(tiles):
            mine = [box for box, fl in boxes if fl[t]]
            work += len(mine)
            # every key of every query's window lies in a box flagged for this tile
            for dt in range(B[0]):
                for dy in range(B[1]):
                    for dx in range(B[2]):
                        c = (org[0] + dt, org[1] + dy, org[2] + dx)
                        if any(c[a] >= grid[a] for a in range(3)):
                            continue
                        ws = [na_start(c[a], kernel[a], grid[a]) for a in range(3)]
                        for a in range(3):
                            covered = set()
                            for box in mine:
                                covered.update(range(box[a], box[a] + KB[a]))
                            assert set(range(ws[a], ws[a] + kernel[a])) <= covered
                        corners = [(ws[0] + e0 * (kernel[0] - 1), ws[1] + e1 * (kernel[1] - 1), ws[2] + e2 * (kernel[2] - 1))
                                   for e0 in (0, 1) for e1 in (0, 1) for e2 in (0, 1)]
                        for kc in corners:
                            assert any(all(box[a] <= kc[a] < box[a] + KB[a] for a in range(3)) for box in mine)
    b, pa, nb = ctypes.c_int(brick), ctypes.c_int(pair), ctypes.c_longlong(0)
    assert lib.attn_na3d_plan(*grid, *kernel, ctypes.byref(b), ctypes.byref(pa), ctypes.byref(nb)) == 0
    assert (b.value, pa.value) == (brick, pair)
    assert nb.value == work


def test_na3d_plan_picks_the_least_work(lib):
    # an open pair axis means the persistent one-brick tiles (plan 4, or plan 5 with the 4x4x8 brick);
    # an open brick minimises 20 (plan 4, 4x4x8) or 23 (plan 4 with the others, plan 5) per key box +
    # 34 per brick there, 20 per box + 40 per CTA elsewhere
    for grid, kernel in [((4, 128, 128), (3, 7, 7)), ((4, 64, 64), (3, 31, 31)), ((1, 96, 160), (1, 13, 13)),
                         ((5, 11, 19), (3, 5, 4)), ((8, 64, 64), (3, 7, 7))]:
        persistent = {}
        for pair in (3, 4, 5):
            costs = {}
            for brick in (1, 2, 3):
                if pair == 5 and brick != 3:
                    continue
                b, pa, nbox = vd.attn_na3d_plan(grid, kernel, brick, pair)
                assert (b, pa) == (brick, pair)
                ctas = np.prod([-(-grid[a] // BRICKS[brick][a]) for a in range(3)])
                if pair == 3:
                    costs[brick] = 20 * nbox + 40 * ctas
                else:
                    costs[brick] = (20 if (brick == 3 and pair == 4) else 23) * nbox + 34 * ctas
                    persistent[(brick, pair)] = costs[brick]
                assert nbox * 128 * 128 >= np.prod(grid) * np.prod(kernel)   # the boxes hold every window
            b, pa, nb = vd.attn_na3d_plan(grid, kernel, 0, pair)
            assert pa == pair and costs[b] == min(costs.values())
        b, pa, nb = vd.attn_na3d_plan(grid, kernel)
        assert pa in (4, 5) and persistent[(b, pa)] == min(persistent.values())
        assert (b, pa, nb) == vd.attn_na3d_plan(grid, kernel, b, pa)
        # a fixed brick with an open pair axis keeps the brick (plan 5 only with the 4x4x8 brick)
        assert vd.attn_na3d_plan(grid, kernel, 2)[:2] == (2, 4)
        assert vd.attn_na3d_plan(grid, kernel, 3)[1] in (4, 5)
        # plan 6 (E5M2 window operands) is never chosen, only taken when asked for
        assert vd.attn_na3d_plan(grid, kernel, 0, 6)[:2] == (3, 6)
        assert vd.attn_na3d_plan(grid, kernel, 3, 6)[2] == vd.attn_na3d_plan(grid, kernel, 3, 5)[2]
    # the volumes timed on GB300 take their fastest plan
    assert vd.attn_na3d_plan((4, 128, 128), (3, 7, 7))[:2] == (3, 5)
    assert vd.attn_na3d_plan((4, 64, 64), (3, 31, 31))[0] == 3
    assert vd.attn_na3d_plan((1, 96, 160), (1, 13, 13))[0] == 1
    assert vd.attn_na3d_plan((8, 64, 64), (3, 7, 7))[0] == 2


def test_na3d_rejections(lib):
    base = [P, P, P, P, P, 1, 2, 4, 16, 16, 128, 3, 5, 5, 0.088, 0, -1, None]
    for i, bad in [(11, 0), (11, 5), (12, 17), (13, 0), (7, 0), (14, 0.0), (14, math.nan), (15, 4), (15, -1),
                   (16, 7), (16, -2)]:
        args = list(base)
        args[i] = bad
        assert lib.attn_na3d_fwd(*args) == 1, (i, bad)
    for brick in (1, 2):   # plans 5 and 6 take the 4x4x8 brick only
        for pair in (5, 6):
            args = list(base)
            args[15], args[16] = brick, pair
            assert lib.attn_na3d_fwd(*args) == 1, (brick, pair)
            b, pa = ctypes.c_int(brick), ctypes.c_int(pair)
            assert lib.attn_na3d_plan(4, 16, 16, 3, 5, 5, ctypes.byref(b), ctypes.byref(pa), None) == 1
    args = list(base)
    args[10] = 96
    assert lib.attn_na3d_fwd(*args) == 2
    args = list(base)
    args[0] = NULL
    assert lib.attn_na3d_fwd(*args) == 1
    args = list(base)
    args[3] = MIS
    assert lib.attn_na3d_fwd(*args) == 1
    b, pa = ctypes.c_int(0), ctypes.c_int(-1)
    assert lib.attn_na3d_plan(4, 16, 16, 5, 3, 3, ctypes.byref(b), ctypes.byref(pa), None) == 1   # Kt > T


def test_fp8_rejections(lib):
    for args in [(NULL, P, P, 4, 64), (P, MIS, P, 4, 64), (P, P, P, 0, 64), (P, P, P, 4, 8), (P, P, P, 4, 72)]:
        assert lib.fp8_quantize_rows(*args, None) == 1, args
    good = [P, P, P, P, P, 256, 512, 1024]
    for i, bad in [(0, NULL), (2, MIS), (3, MIS), (4, MIS), (5, 0), (6, 4), (6, 12), (7, 8), (7, 40)]:
        args = list(good)
        args[i] = bad
        assert lib.fp8_scaled_gemm(*args, None) == 1, (i, bad)


def test_cross_fused_rejections(lib):
    need = lib.attn_cross_workspace_bytes(1, 32, 128, 128, 8)
    rows = 32 * 128
    assert need >= 8 * rows * 129 * 4 + 32 * 4
    assert lib.attn_cross_workspace_bytes(1, 32, 128, 96, 8) == 0
    ws = ctypes.c_void_p(0x100000)
    base = [P, P, P, P, P, 1, 32, 128, 4096, 128, 8, 0.088, ws, need, None]
    args = list(base); args[13] = need - 1
    assert lib.attn_cross_fwd(*args) == 3                 # workspace too small
    args = list(base); args[12] = None
    assert lib.attn_cross_fwd(*args) == 1                 # no workspace
    args = list(base); args[12] = MIS
    assert lib.attn_cross_fwd(*args) == 1                 # misaligned workspace
    args = list(base); args[10] = 4097
    assert lib.attn_cross_fwd(*args) == 1                 # more chunks than keys
    args = list(base); args[10] = 33; args[13] = 1 << 40
    assert lib.attn_cross_fwd(*args) == 2                 # more chunks than the tail merges
