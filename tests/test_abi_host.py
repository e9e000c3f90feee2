"""Host-side checks of the C ABI (no GPU): the library loads, exports every
entry point include/attn_api.h declares, and rejects invalid arguments before
touching the device."""
import ctypes
import math
import os
import re

import pytest

import video_diffusion_transformer_block_gb300 as vd
from video_diffusion_transformer_block_gb300 import build as vbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_api.h")


@pytest.fixture(scope="module")
def lib():
    vbuild.build()
    return vd.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(vd.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {vbuild.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} not exported"


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
    expect_min = 32 * nq * 128 * 4 * 3 + 32 * nq * nq * 4 + 32 * nq * 4 * 5 + 32 * nq * 128 * 4
    assert expect_min <= n <= expect_min + 7 * 256
    assert lib.attn_sparse_workspace_bytes(1, 1, 1000, 128, 64, 128) == 0      # block_q != block_k
    assert lib.attn_sparse_workspace_bytes(1, 1, 1000, 96, 64, 64) == 0        # bad d
    ws = ctypes.c_void_p(0x100000)
    args = [P, P, P, P, P, 1, 2, 1024, 64, 0.125, 0.5, 64, 64, ws, 0, None, None, None, None, None]
    assert lib.attn_sparse_route_fwd(*args) == 3                              # workspace too small
    args[10] = math.nan
    assert lib.attn_sparse_route_fwd(*args) == 1                              # NaN beta
    args[10], args[11] = 0.5, 32
    assert lib.attn_sparse_route_fwd(*args) == 2                              # unsupported block


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
