/*
 * FP8 projection path: per-row E4M3 quantisation of activations and the scaled
 * FP8 matrix product of the transformer block's linear layers.
 *
 * Source: "LTX-2.5 at 4K, in half the time" (doubleai.com), section "Thinner
 * seams": weights are kept in FP8 instead of being widened to BF16 before
 * each product, activations are quantised to FP8 at run time with one scale
 * per row, and the tensor cores accumulate in FP32 at FP8 throughput.  "Optimization Tips" (LTX-2 pipelines
 * documentation), section "FP8 Quantization": FP8 scaled matrix
 * multiplication.
 *
 * FP8 here is E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * subnormals, no infinities, S.1111.111 = NaN, largest finite value 448.
 *
 * Ownership and errors as in attn_api.h: the caller owns every device buffer,
 * the library allocates nothing, every call is asynchronous on `stream`, and
 * argument errors return before any launch.
 */
#ifndef FP8_API_H
#define FP8_API_H

#include "attn_api.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Per-row quantisation.  For row m of x [M][K] (bf16, row-major):
 *   amax_m   = max_k |x[m][k]|
 *   scale[m] = amax_m / 448                     (the nearest fp32 value)
 *   q[m][k]  = the E4M3 value nearest to the exact quotient x[m][k] * 448 / amax_m,
 *              ties to even (bit-exact: the kernel multiplies by the rounded
 *              inverse scale and re-forms the quotient with a correctly rounded
 *              division wherever that product lies next to a rounding midpoint)
 * so the row's largest magnitude maps to +-448 and x ~ scale[m] * q.  A row of
 * zeros, or one whose scale is not a normal float (amax_m / 448 < 2^-126), gets
 * scale 0 and zero codes.  NaN inputs are not supported.
 *   x      device, 16-byte aligned, [M][K] bf16.
 *   q      device, 16-byte aligned, [M][K] E4M3 codes (uint8).
 *   scale  device, [M] fp32.
 *   Errors: ATTN_ERR_INVALID_ARG (null or misaligned pointer, M < 1, K < 16,
 *   K not a multiple of 16), ATTN_ERR_CUDA (launch).
 * Weights use the same routine with one row per output channel.
 */
attn_status_t fp8_quantize_rows(const attn_bf16* x, uint8_t* q, float* scale, int M, int K, cudaStream_t stream);

/*
 * Scaled FP8 matrix product (a linear layer without bias):
 *   y[m][n] = a_scale[m] * w_scale[n] * sum_k dec(aq[m][k]) * dec(wq[n][k])
 * with the sum accumulated in fp32 on the tensor cores and y rounded to bf16
 * (nearest even).
 *   aq       device, 16-byte aligned, [M][K] E4M3 codes (activations).
 *   a_scale  device, [M] fp32 (per-row activation scales).
 *   wq       device, 16-byte aligned, [N][K] E4M3 codes (one output channel
 *            per row, i.e. W of y = x W^T).
 *   w_scale  device, 16-byte aligned, [N] fp32 (per-output-channel weight
 *            scales; a per-tensor scale is the case of equal entries).
 *   y        device, 16-byte aligned, [M][N] bf16 (row-major).
 *   Errors: ATTN_ERR_INVALID_ARG (null or misaligned pointer, M < 1, N < 8 or
 *   not a multiple of 8, K < 16 or not a multiple of 16), ATTN_ERR_CUDA
 *   (descriptor encoding or launch); a device wait past its bound sets the
 *   status word read by attn_last_device_status (ATTN_ERR_TIMEOUT).
 */
attn_status_t fp8_scaled_gemm(const uint8_t* aq, const float* a_scale, const uint8_t* wq, const float* w_scale,
                              attn_bf16* y, int M, int N, int K, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8_API_H */
