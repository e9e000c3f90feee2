"""GPU parity of the FP8 projection path against the oracle, through the C ABI.

The quantiser's codes and scales must be bit-identical to the oracle's, which
takes each code as the E4M3 value nearest to the exact quotient x * 448 / amax.
The kernel decides most codes from the product with a rounded inverse scale and
re-forms the quotient exactly where that product lies next to a rounding
midpoint; rows built to hit exact midpoints (amax with significand 3, 5, 7, ...
and small-integer multiples) exercise that path.  The scaled product is
compared element by element with the bound |y_gpu - y| <= 2^-8 |y| + K 2^-24
sum|terms|: the bf16 rounding of the output plus the worst case of fp32
accumulation over K terms.
"""
import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_block_gb300 as vd
from workloads import LINEAR_WORKLOADS, LinearWorkload, make_linear

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    torch.cuda.synchronize()
    yield
    assert vd.attn_last_device_status() == 0


def f32(x):
    return x.detach().to("cpu", torch.float32).numpy()


def check_gemm(y_gpu, y_ref, y_abs, K, what):
    g = y_gpu.detach().to("cpu", torch.float32).double().numpy()
    assert np.isfinite(g).all(), what
    bound = 2.0 ** -8 * np.abs(y_ref) + K * 2.0 ** -24 * y_abs + 1e-30
    bad = np.abs(g - y_ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside the bound, worst excess " \
                          f"{float(np.max((np.abs(g - y_ref) - bound)[bad])):.3e}"


@pytest.mark.parametrize("M,K", [(1, 16), (7, 144), (300, 4096), (129, 4112), (64, 1024), (33, 2048), (9, 8192), (17, 272)])
def test_quantize_rows_bit_exact(M, K):
    x, _ = make_linear(LinearWorkload("q", M=M, K=K, N=8, seed=M + K), device="cuda")
    x[min(3, M - 1)] = 0                                      # a zero row
    if M > 5:
        x[5] *= 1e-4                                          # tiny values: subnormal codes
    if M > 8:
        x[8:] = midpoint_rows(M - 8, K, seed=M).to(x.device)  # exact E4M3 rounding midpoints
    q, s = vd.fp8_quantize_rows(x)
    torch.cuda.synchronize()
    xh = f32(x)
    rq, rs = oracle.fp8_quantize_rows(xh)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    ties = exact_midpoint_count(xh)
    print(f"quantize {M}x{K}: {ties} elements whose exact quotient is an E4M3 rounding midpoint")
    if M > 8:
        assert ties > 0


def midpoint_rows(n, K, seed):
    """bf16 rows whose row max has significand 3, 5, 7, ... and whose other values are small-integer
    multiples of a power of two: many quotients x * 448 / amax land exactly on E4M3 rounding midpoints,
    where a product with the rounded inverse scale 448 / amax would round the wrong way."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    amax = torch.tensor([3.0, 5.0, 7.0, 11.0, 13.0, 0.375, 1.25, 6.5, 3e-3, 5e4])
    rows = torch.randint(-64, 65, (n, K), generator=g).float()
    rows *= 2.0 ** torch.randint(-9, -1, (n, 1), generator=g).float()
    a = amax[torch.randint(0, amax.numel(), (n,), generator=g)] * 2.0 ** torch.randint(-4, 4, (n,), generator=g)
    rows = torch.maximum(torch.minimum(rows * a[:, None] / 3.0, a[:, None]), -a[:, None])
    rows[:, 0] = a
    return rows.bfloat16()


def exact_midpoint_count(x):
    """Elements of x [M, K] (float32) whose exact quotient x * 448 / amax is an E4M3 rounding midpoint."""
    amax = np.abs(x).max(axis=1, keepdims=True).astype(np.float64)
    v = np.abs(x.astype(np.float64)) * 448.0 / np.where(amax > 0, amax, 1.0)
    pos = np.sort(np.unique(oracle.e4m3_decode(np.arange(0x7f, dtype=np.uint8))))
    mids = (pos[:-1] + pos[1:]) / 2
    return int(np.isin(v, mids).sum())


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 128),     # one tile, one k-block
    (300, 264, 4096),    # ragged M and N, many k-blocks
    (1, 8, 16),          # smallest sizes (K tail inside one block)
    (257, 512, 144),     # K not a multiple of 128
    (1000, 1024, 1024),  # many tiles per CTA
])
def test_scaled_gemm_matches_oracle(M, N, K):
    x, W = make_linear(LinearWorkload("g", M=M, K=K, N=N, seed=3 * M + N), device="cuda")
    aq, sa = vd.fp8_quantize_rows(x)
    wq, sw = vd.fp8_quantize_rows(W)
    y = vd.fp8_scaled_gemm(aq, sa, wq, sw)
    torch.cuda.synchronize()
    ry, ra = oracle.fp8_gemm(aq.cpu().numpy(), sa.cpu().numpy(), wq.cpu().numpy(), sw.cpu().numpy())
    check_gemm(y, ry, ra, K, f"fp8 gemm {M}x{N}x{K}")


def test_scaled_gemm_integer_codes_are_exact():
    # small-integer operands: every product and partial sum is an integer below 2^24, so fp32
    # accumulation is exact and only the bf16 output rounding remains
    M, N, K = 200, 256, 512
    g = torch.Generator(device="cpu").manual_seed(4)
    a = torch.randint(-4, 5, (M, K), generator=g).float()
    w = torch.randint(-3, 4, (N, K), generator=g).float()
    aq = a.to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    wq = w.to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    ones_m, ones_n = torch.ones(M, device="cuda"), torch.ones(N, device="cuda")
    y = vd.fp8_scaled_gemm(aq, ones_m, wq, ones_n)
    torch.cuda.synchronize()
    exact = (a.double() @ w.double().T)
    assert torch.equal(y.cpu(), exact.to(torch.bfloat16))


def test_fp8_linear_full_size_sampled_rows():
    w = LINEAR_WORKLOADS["fp8_proj"]
    x, W = make_linear(w, device="cuda")
    wq, sw = vd.fp8_quantize_rows(W)
    aq, sa = vd.fp8_quantize_rows(x)
    y = vd.fp8_scaled_gemm(aq, sa, wq, sw)
    torch.cuda.synchronize()
    rng = np.random.default_rng(108)
    rows = np.sort(np.concatenate([[0, w.M - 1], rng.choice(np.arange(1, w.M - 1), size=254, replace=False)]))
    xr = f32(x[torch.from_numpy(rows).cuda()])
    rq, rs = oracle.fp8_quantize_rows(xr)
    np.testing.assert_array_equal(aq[torch.from_numpy(rows).cuda()].cpu().numpy(), rq)
    np.testing.assert_array_equal(sa[torch.from_numpy(rows).cuda()].cpu().numpy(), rs)
    rwq, rws = oracle.fp8_quantize_rows(f32(W))
    np.testing.assert_array_equal(wq.cpu().numpy(), rwq)
    ry, ra = oracle.fp8_gemm(rq, rs, rwq, rws)
    check_gemm(y[torch.from_numpy(rows).cuda()], ry, ra, w.K, "fp8_proj sampled rows")
