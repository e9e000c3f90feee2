// FP8 (E4M3) projection path for sm_103a: per-row activation quantisation and
// the scaled FP8 matrix product y = diag(sa) (Aq Wq^T) diag(sw), accumulated
// in fp32 on the tensor cores (tcgen05 kind::f8f6f4) and written as bf16.
//
// GEMM CTA (persistent, one per SM): warp 0 = TMA producer, warp 1 = MMA
// issuer (one thread), warps 2..9 = epilogue: two warps per TMEM lane quarter
// (a warp may only read its own quarter of the lanes), each taking 128 of the
// tile's 256 columns for its 32 rows.  Output tiles are 128 x 256; K advances in
// blocks of 128 bytes (one 128-byte swizzle atom, four MMAs of K = 32) through a
// ring of kStages shared-memory slots.  The two halves of TMEM (2 x 256
// columns) hold the accumulators of consecutive tiles, so the epilogue of tile
// i overlaps the MMAs of tile i + 1.
#include <cuda_fp8.h>

#include "launch.h"
#include "ptx.cuh"

namespace vdtb {
namespace {

// ---------------------------------------------------------------- quantiser

constexpr int kQuantThreads = 256;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
    f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}

// Row scales from the row's amax: the dequantisation scale s = amax / 448 and
// the inverse 448 / amax (fp32 divisions, once per row).  A row whose scale is
// zero or not a normal float (amax / 448 < 2^-126) quantises to zeros with
// scale 0; otherwise the inverse is at most 2^126 and finite.
__device__ __forceinline__ void row_scales(float amax, float& s, float& inv) {
  s = __fdiv_rn(amax, 448.0f);
  if (!(s >= 0x1p-126f)) {
    s = 0.f;
    inv = 0.f;
  } else {
    inv = __fdiv_rn(448.0f, amax);
  }
}

// The code of a bf16 value x is the E4M3 value nearest to the exact quotient
// x * 448 / amax (ties to even).  The product v = x * inv with the rounded
// inverse scale inv lies within two float steps of that quotient, so it decides
// the same code unless it sits next to an E4M3 rounding midpoint.  Where it
// might, the quotient is formed again with one correctly rounded division,
// which for bf16 operands decides exactly: x * 0.875 is exact, and a quotient of bf16
// values either is a midpoint (returned exactly by the division) or lies at
// least 2^-13 of its size away from every midpoint.  Tiny rows are scaled by
// 2^64 first so that no operand of the division is subnormal.
__device__ __forceinline__ float exact_quotient(float x, float amax) {
  if (amax < 0x1p-60f) {
    x *= 0x1p64f;
    amax *= 0x1p64f;
  }
  return __fmul_rn(__fdiv_rn(__fmul_rn(x, 0.875f), amax), 512.0f);
}

// Whether the product with the rounded inverse scale may decide a code other
// than the exact quotient for some value of the row in the normal E4M3 range
// (|v| >= 2^-6).  There the decision depends only on the value's bf16
// significand, so thread t (0..127) tries the significand 1 + t/128 at the
// row's scale (x = (1 + t/128) * 2^(E-1) with amax in [2^E, 2^(E+1)), so that
// x * 448 / amax lies in (112, 448)) both ways: the product and the exact
// division.  The row is flagged when any significand's codes differ (about
// 2% of random rows); flagged rows take every code from the division.
__device__ __forceinline__ bool row_product_differs(float amax, float inv, int t) {
  const uint32_t e = __float_as_uint(amax) >> 23;   // biased exponent of amax (> 8 for a non-flushed row)
  const float x = __uint_as_float(((e - 1u) << 23) | ((uint32_t)(t & 127) << 16));
  const uint32_t fast = (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(x, inv), __NV_SATFINITE, __NV_E4M3);
  const uint32_t exact = (uint32_t)__nv_cvt_float_to_fp8(exact_quotient(x, amax), __NV_SATFINITE, __NV_E4M3);
  return fast != exact;
}

// Two codes in one conversion (round to nearest even, saturating at +-448):
// `lo` in the low byte, `hi` in the high byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Codes of 8 values: from the products, except values on the E4M3 subnormal
// grid (0 < |v| < 2^-6, where the grid is not scale-free) and every value of a
// flagged row, which take the exact division.
__device__ __forceinline__ uint2 quantize8(const uint4& v, float inv, float amax, bool row_exact) {
  float f[8], t[8];
  unpack8(v, f);
  bool sub = false;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    t[e] = __fmul_rn(f[e], inv);
    sub |= fabsf(t[e]) < 0x1p-6f && t[e] != 0.f;
  }
  if (sub || row_exact) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (row_exact || (fabsf(t[e]) < 0x1p-6f && t[e] != 0.f)) t[e] = exact_quotient(f[e], amax);
  }
  const uint32_t lo = e4m3x2(t[0], t[1]) | (e4m3x2(t[2], t[3]) << 16);
  const uint32_t hi = e4m3x2(t[4], t[5]) | (e4m3x2(t[6], t[7]) << 16);
  return make_uint2(lo, hi);
}

// One CTA per row (rows longer than the register-resident kernel takes): amax
// over the row, then the codes.  The second pass re-reads the row, which the
// first pass has just brought into L1.
__global__ void __launch_bounds__(kQuantThreads) fp8_quantize_rows_kernel(const uint16_t* __restrict__ x,
                                                                          uint8_t* __restrict__ q,
                                                                          float* __restrict__ scale, int K,
                                                                          int* status) {
  const long long row = blockIdx.x;
  const uint16_t* xr = x + row * K;
  uint8_t* qr = q + row * K;
  float amax = 0.f;
  for (int i = threadIdx.x * 8; i < K; i += kQuantThreads * 8) {
    float f[8];
    unpack8(*reinterpret_cast<const uint4*>(xr + i), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[kQuantThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  float s, inv;
  row_scales(amax, s, inv);
  const bool row_exact = __syncthreads_or(inv != 0.f && row_product_differs(amax, inv, threadIdx.x));
  [[maybe_unused]] const long long M = gridDim.x;
  if (threadIdx.x == 0 && ATTN_CHECKED(row, 1, M, status)) scale[row] = s;
  for (int i = threadIdx.x * 8; i < K; i += kQuantThreads * 8)
    if (ATTN_CHECKED(row * K + i, 8, M * K, status))
      *reinterpret_cast<uint2*>(qr + i) = quantize8(*reinterpret_cast<const uint4*>(xr + i), inv, amax, row_exact);
}

// One CTA of 128 threads per row for rows of up to NV * 1024 elements: each
// thread keeps its NV 16-byte vectors in registers between the amax and the
// quantisation, so HBM is read once and every load is issued up front.
template <int NV>
__global__ void __launch_bounds__(128) fp8_quantize_rows_reg_kernel(const uint16_t* __restrict__ x,
                                                                    uint8_t* __restrict__ q,
                                                                    float* __restrict__ scale, int K, int* status) {
  const long long row = blockIdx.x;
  const uint16_t* xr = x + row * K;
  uint8_t* qr = q + row * K;
  uint4 v[NV];
#pragma unroll
  for (int c = 0; c < NV; ++c) {
    const int i = (c * 128 + threadIdx.x) * 8;
    v[c] = i < K ? __ldcs(reinterpret_cast<const uint4*>(xr + i)) : make_uint4(0, 0, 0, 0);
  }
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < NV; ++c) {
    float f[8];
    unpack8(v[c], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[4];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  float s, inv;
  row_scales(amax, s, inv);
  const bool row_exact = __syncthreads_or(inv != 0.f && row_product_differs(amax, inv, threadIdx.x));
  [[maybe_unused]] const long long M = gridDim.x;
  if (threadIdx.x == 0 && ATTN_CHECKED(row, 1, M, status)) scale[row] = s;
#pragma unroll
  for (int c = 0; c < NV; ++c) {
    const int i = (c * 128 + threadIdx.x) * 8;
    if (i < K && ATTN_CHECKED(row * K + i, 8, M * K, status))
      __stcs(reinterpret_cast<uint2*>(qr + i), quantize8(v[c], inv, amax, row_exact));
  }
}

// ---------------------------------------------------------------- GEMM

constexpr int kBM = 128, kBN = 256, kBK = 128, kStages = 4;
constexpr int kGemmThreads = 320;
constexpr int kEpilogueThreads = 256;
constexpr int kStageA = kBM * kBK, kStageB = kBN * kBK, kStageBytes = kStageA + kStageB;
constexpr int kGemmSmem = 1024 + kStages * kStageBytes;
constexpr uint32_t kTmemCols = 512;
// instruction descriptor, kind::f8f6f4: fp32 accumulator (bit 4), A and B
// E4M3 (type code 0 in bits 7-9 and 10-12), both K-major, N >> 3 at bit 17,
// M >> 4 at bit 24
constexpr uint32_t kIdescF8 = (1u << 4) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accum));
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"((uint64_t)m), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const float* __restrict__ sa, const float* __restrict__ sw, uint16_t* __restrict__ y, int M, int N,
                    int K, int* status, unsigned launch_id) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages], bar_acc_full[2], bar_acc_empty[2], bar_mma_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ WaitState wstate;
  __shared__ int skip_cta;   // the launch had already aborted when this CTA started
  WaitState* const wc = &wstate;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_nb = (N + kBN - 1) / kBN;
  const int tiles = ((M + kBM - 1) / kBM) * n_nb;
  const int nk = (K + kBK - 1) / kBK;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_acc_full[b], 1);
      mbar_init(&bar_acc_empty[b], kEpilogueThreads);
    }
    mbar_init(&bar_mma_done, 1);
    skip_cta = wait_state_init(wstate, status, launch_id);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (!skip_cta) {

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
        const int mb = tile / n_nb, nb = tile % n_nb;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int slot = it % kStages;
          if (it >= kStages && !bounded_wait(&bar_empty[slot], ((it / kStages) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + slot * kStageBytes;
          mbar_expect_tx(&bar_full[slot], kStageBytes);
          tma_load_2d(sA, &tm_a, &bar_full[slot], kb * kBK, mb * kBM);
          tma_load_2d(sA + kStageA, &tm_b, &bar_full[slot], kb * kBK, nb * kBN);
        }
      }
      // drain: no copy may still be landing when the CTA exits
      for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
        drain_wait(&bar_full[j % kStages], (j / kStages) & 1, wc);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t base = smem_u32(smem);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x, ++tcount) {
        const int buf = tcount & 1, use = tcount >> 1;
        if (use > 0 && !bounded_wait(&bar_acc_empty[buf], (use - 1) & 1, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * kBN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int slot = it % kStages;
          if (!bounded_wait(&bar_full[slot], (it / kStages) & 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = base + slot * kStageBytes;
          const uint32_t b_addr = a_addr + kStageA;
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_f8(d, smem_desc_sw128(a_addr + kk * 32, 16, 1024), smem_desc_sw128(b_addr + kk * 32, 16, 1024),
                   kIdescF8, (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar_empty[slot]);
        }
        if (ok) mma_commit(&bar_acc_full[buf]);
      }
      // every MMA issued by this thread has completed before TMEM is released
      mma_commit(&bar_mma_done);
      drain_wait(&bar_mma_done, 0, wc);
    }
  } else {
    // ======================= epilogue =======================
    const int quarter = warp & 3;                 // TMEM lanes [32 quarter, 32 quarter + 32)
    const int half = (warp - 2) >> 2;             // columns [128 half, 128 half + 128)
    const int r = quarter * 32 + lane;
    int tcount = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++tcount) {
      const int buf = tcount & 1, use = tcount >> 1;
      if (!__all_sync(0xffffffffu, bounded_wait(&bar_acc_full[buf], use & 1, wc))) break;
      tc_fence_after();
      const int mb = tile / n_nb, nb = tile % n_nb;
      const long long grow = (long long)mb * kBM + r;
      const bool row_ok = grow < M;
      const float s_row = row_ok ? __ldg(sa + grow) : 0.f;
      uint16_t* dst = y + grow * N;
      const uint32_t t_addr = tmem + ((uint32_t)(quarter * 32) << 16) + buf * kBN;
#pragma unroll 1
      for (int c0 = half * (kBN / 2); c0 < (half + 1) * (kBN / 2); c0 += 32) {
        uint32_t acc[32];
        tmem_ld32(t_addr + c0, acc);
        tmem_ld_wait();
        tmem_reg_fence(acc);
        const int col0 = nb * kBN + c0;
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            const int col = col0 + j;
            if (col + 8 <= N) {
              // column scales: the same 8 floats for every lane (broadcast loads)
              const float4 w0 = __ldg(reinterpret_cast<const float4*>(sw + col));
              const float4 w1 = __ldg(reinterpret_cast<const float4*>(sw + col + 4));
              const float ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
              float o[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(acc[j + e]) * s_row * ws[e];
              uint4 pk;
              pk.x = pack_bf16x2(o[0], o[1]);
              pk.y = pack_bf16x2(o[2], o[3]);
              pk.z = pack_bf16x2(o[4], o[5]);
              pk.w = pack_bf16x2(o[6], o[7]);
              if (ATTN_CHECKED(grow * N + col, 8, (long long)M * N, status)) *reinterpret_cast<uint4*>(dst + col) = pk;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_acc_empty[buf]);
    }
  }
  }   // !skip_cta

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fp8_quantize_rows(const uint16_t* x, uint8_t* q, float* scale, int M, int K, int* status,
                                     cudaStream_t stream) {
  if (K <= 1024)
    fp8_quantize_rows_reg_kernel<1><<<M, 128, 0, stream>>>(x, q, scale, K, status);
  else if (K <= 2048)
    fp8_quantize_rows_reg_kernel<2><<<M, 128, 0, stream>>>(x, q, scale, K, status);
  else if (K <= 4096)
    fp8_quantize_rows_reg_kernel<4><<<M, 128, 0, stream>>>(x, q, scale, K, status);
  else
    fp8_quantize_rows_kernel<<<M, kQuantThreads, 0, stream>>>(x, q, scale, K, status);
  return cudaGetLastError();
}

cudaError_t launch_fp8_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const float* sa, const float* sw,
                            uint16_t* y, int M, int N, int K, int* status, unsigned launch_id,
                            cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long tiles = (long long)((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  const int grid = (int)(tiles < sms ? tiles : sms);
  fp8_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, stream>>>(ta, tb, sa, sw, y, M, N, K, status, launch_id);
  return cudaGetLastError();
}

}  // namespace vdtb
