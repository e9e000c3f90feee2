// Bandwidth-bound kernels of the hot path: block mean-pool and the exact
// log-sum-exp merge of split-KV partials (the routing is in route_tc.cu).
#include <math.h>
#include <stdint.h>

#include "launch.h"

namespace vdtb {

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ============================================================ block mean-pool
// One CTA per (tensor, head, block).  Thread = (16-byte column chunk, row
// group); each thread streams rows of its chunk with 128-bit non-caching
// loads, then the row groups are summed through shared memory.  For the
// tensor-core routing the pooled keys (tensor 1) are also written as tf32
// hi / lo pairs ([BH][NB][D]) and the pooled values (tensor 2) as transposed
// hi / lo pairs ([BH][D][NBp]): hi = the mean with its 13 low mantissa bits
// cleared, lo = mean - hi.
// Source: "Accelerating LTX-2.5 with Sol Engine", Sol-Attn bullet
// "On-the-fly routing" (pooled keys).
template <int D>
__global__ void __launch_bounds__(256) pool_kernel(const uint16_t* __restrict__ x0, const uint16_t* __restrict__ x1,
                                                   const uint16_t* __restrict__ x2, float* __restrict__ p0,
                                                   float* __restrict__ p1, float* __restrict__ p2, int S, int block,
                                                   int NB, const PoolSplit split, int* status) {
  constexpr int CH = D / 8;        // 16-byte chunks per row
  constexpr int RG = 256 / CH;     // row groups
  __shared__ float red[RG][D + 1];
  const uint16_t* x = blockIdx.y == 0 ? x0 : (blockIdx.y == 1 ? x1 : x2);
  float* xp = blockIdx.y == 0 ? p0 : (blockIdx.y == 1 ? p1 : p2);
  const long long bh = blockIdx.x / NB;
  const int i = blockIdx.x % NB;
  const int lo = i * block;
  const int hi = min(lo + block, S);
  const int c = threadIdx.x % CH, g = threadIdx.x / CH;
  const uint16_t* base = x + (bh * S) * D + c * 8;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  int r = lo + g;
  for (; r + 3 * RG < hi; r += 4 * RG) {
    uint4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) w[u] = ld_stream_u4(base + (long long)(r + u * RG) * D);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc[0] += bf16lo(w[u].x); acc[1] += bf16hi(w[u].x);
      acc[2] += bf16lo(w[u].y); acc[3] += bf16hi(w[u].y);
      acc[4] += bf16lo(w[u].z); acc[5] += bf16hi(w[u].z);
      acc[6] += bf16lo(w[u].w); acc[7] += bf16hi(w[u].w);
    }
  }
  for (; r < hi; r += RG) {
    uint4 w = ld_stream_u4(base + (long long)r * D);
    acc[0] += bf16lo(w.x); acc[1] += bf16hi(w.x);
    acc[2] += bf16lo(w.y); acc[3] += bf16hi(w.y);
    acc[4] += bf16lo(w.z); acc[5] += bf16hi(w.z);
    acc[6] += bf16lo(w.w); acc[7] += bf16hi(w.w);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[g][c * 8 + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll 8
    for (int gg = 0; gg < RG; ++gg) s += red[gg][threadIdx.x];
    const float m = s / (float)(hi - lo);
    if (ATTN_CHECKED((bh * NB + i) * D + threadIdx.x, 1, (long long)gridDim.x * D, status))
      xp[(bh * NB + i) * D + threadIdx.x] = m;
    const float mh = __uint_as_float(__float_as_uint(m) & 0xFFFFE000u);
    if (blockIdx.y == 1 && split.kh != nullptr &&
        ATTN_CHECKED((bh * NB + i) * D + threadIdx.x, 1, (long long)gridDim.x * D, status)) {
      split.kh[(bh * NB + i) * D + threadIdx.x] = mh;
      split.kl[(bh * NB + i) * D + threadIdx.x] = m - mh;
    }
    if (blockIdx.y == 2 && split.vth != nullptr &&
        ATTN_CHECKED((bh * D + threadIdx.x) * split.NBp + i, 1, (long long)(gridDim.x / NB) * D * split.NBp, status)) {
      split.vth[(bh * D + threadIdx.x) * split.NBp + i] = mh;
      split.vtl[(bh * D + threadIdx.x) * split.NBp + i] = m - mh;
    }
  }
}

cudaError_t launch_pool(const uint16_t* x0, const uint16_t* x1, const uint16_t* x2, float* p0, float* p1, float* p2,
                        int ntensors, int BH, int S, int D, int block, const PoolSplit& split, int* status,
                        cudaStream_t stream) {
  const int NB = (S + block - 1) / block;
  long long nblk = (long long)BH * NB;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)nblk, ntensors);
  if (D == 128)
    pool_kernel<128><<<grid, 256, 0, stream>>>(x0, x1, x2, p0, p1, p2, S, block, NB, split, status);
  else
    pool_kernel<64><<<grid, 256, 0, stream>>>(x0, x1, x2, p0, p1, p2, S, block, NB, split, status);
  return cudaGetLastError();
}

// ============================================================ LSE merge
// One warp per query row; lane l owns D/32 consecutive columns (float4 or
// float2), so each partial row is one coalesced 512/256-byte read.
//   L = M + log sum_c exp(lse_c - M),  o = sum_c exp(lse_c - L) o_c
// Source: "LTX-2.5 at 4K, in half the time", section "Attention across two GPUs".
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const float* __restrict__ o_part,
                                                        const float* __restrict__ lse_part, uint16_t* __restrict__ out,
                                                        float* __restrict__ lse, int n, long long rows, int* status) {
  constexpr int PER = D / 32;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float M = -INFINITY;
  for (int c = 0; c < n; ++c) M = fmaxf(M, __ldg(lse_part + (long long)c * rows + row));
  float o[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) o[e] = 0.f;
  float L = -INFINITY;
  if (M != -INFINITY) {
    float ssum = 0.f;
    for (int c = 0; c < n; ++c) ssum += expf(__ldg(lse_part + (long long)c * rows + row) - M);
    L = M + logf(ssum);
    int c = 0;
    for (; c + 1 < n; c += 2) {
      const float w0 = expf(__ldg(lse_part + (long long)c * rows + row) - L);
      const float w1 = expf(__ldg(lse_part + (long long)(c + 1) * rows + row) - L);
      const float* s0 = o_part + ((long long)c * rows + row) * D + lane * PER;
      const float* s1 = s0 + rows * D;
      float a0[PER], a1[PER];
      if constexpr (PER == 4) {
        const float4 v0 = __ldcs(reinterpret_cast<const float4*>(s0));
        const float4 v1 = __ldcs(reinterpret_cast<const float4*>(s1));
        a0[0] = v0.x; a0[1] = v0.y; a0[2] = v0.z; a0[3] = v0.w;
        a1[0] = v1.x; a1[1] = v1.y; a1[2] = v1.z; a1[3] = v1.w;
      } else {
        const float2 v0 = __ldcs(reinterpret_cast<const float2*>(s0));
        const float2 v1 = __ldcs(reinterpret_cast<const float2*>(s1));
        a0[0] = v0.x; a0[1] = v0.y;
        a1[0] = v1.x; a1[1] = v1.y;
      }
#pragma unroll
      for (int e = 0; e < PER; ++e) o[e] = fmaf(w1, a1[e], fmaf(w0, a0[e], o[e]));
    }
    for (; c < n; ++c) {
      const float w0 = expf(__ldg(lse_part + (long long)c * rows + row) - L);
      const float* s0 = o_part + ((long long)c * rows + row) * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[e] = fmaf(w0, __ldcs(s0 + e), o[e]);
    }
  }
  uint16_t* dst = out + row * D + lane * PER;
  if (ATTN_CHECKED(row * D + lane * PER, PER, rows * D, status)) {
    if constexpr (PER == 4) {
      uint2 pk;
      pk.x = pack_bf16x2(o[0], o[1]);
      pk.y = pack_bf16x2(o[2], o[3]);
      *reinterpret_cast<uint2*>(dst) = pk;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[0], o[1]);
    }
  }
  if (lse != nullptr && lane == 0 && ATTN_CHECKED(row, 1, rows, status)) lse[row] = L;
}

// Same merge with every load of a row issued before any arithmetic (rows with
// n <= NMAX partials): the n lse values (one broadcast load each) and the
// n slices of the partial outputs go into registers at once, so a row costs one
// memory round trip instead of three dependent ones.  The arithmetic and its
// order are those of lse_merge_kernel, so the results are bit-identical.
template <int D, int NMAX>
__global__ void __launch_bounds__(256) lse_merge_reg_kernel(const float* __restrict__ o_part,
                                                            const float* __restrict__ lse_part,
                                                            uint16_t* __restrict__ out, float* __restrict__ lse, int n,
                                                            long long rows, int* status) {
  constexpr int PER = D / 32;
  // programmatic dependent launch: let the next kernel in the stream start its
  // launch now, and wait until the kernel before this one (which may have
  // produced the partials) has completed and its writes are visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Meanwhile thread c asks L2 for this block's 8 rows of partial c and their
  // lse values, so that the loads after the wait find them there instead of
  // waiting on DRAM.  A prefetch returns no data and L2 is where every write
  // of the kernel before lands, so a line it is still writing cannot be read
  // stale: the loads come after the wait.
  {
    const long long row0 = (long long)blockIdx.x * 8;
    const int c = threadIdx.x;
    if (c < n && row0 < rows) {
      const long long nr = rows - row0 < 8 ? rows - row0 : 8;
      const float* src = o_part + ((long long)c * rows + row0) * D;   // 16-byte aligned, nr * D * 4 bytes
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"((unsigned)(nr * D * 4)) : "memory");
      asm volatile("prefetch.global.L2 [%0];" ::"l"(lse_part + (long long)c * rows + row0) : "memory");
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float ls[NMAX];
  float a[NMAX][PER];
#pragma unroll
  for (int c = 0; c < NMAX; ++c) {
    if (c < n) {
      ls[c] = __ldg(lse_part + (long long)c * rows + row);
      const float* src = o_part + ((long long)c * rows + row) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(src));
        a[c][0] = v.x; a[c][1] = v.y; a[c][2] = v.z; a[c][3] = v.w;
      } else {
        const float2 v = __ldcs(reinterpret_cast<const float2*>(src));
        a[c][0] = v.x; a[c][1] = v.y;
      }
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int c = 0; c < NMAX; ++c)
    if (c < n) M = fmaxf(M, ls[c]);
  float o[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) o[e] = 0.f;
  float L = -INFINITY;
  if (M != -INFINITY) {
    float ssum = 0.f;
#pragma unroll
    for (int c = 0; c < NMAX; ++c)
      if (c < n) ssum += expf(ls[c] - M);
    L = M + logf(ssum);
#pragma unroll
    for (int c = 0; c + 1 < NMAX; c += 2) {
      if (c + 1 < n) {
        const float w0 = expf(ls[c] - L);
        const float w1 = expf(ls[c + 1] - L);
#pragma unroll
        for (int e = 0; e < PER; ++e) o[e] = fmaf(w1, a[c + 1][e], fmaf(w0, a[c][e], o[e]));
      } else if (c < n) {   // odd n: the last partial alone
        const float w0 = expf(ls[c] - L);
#pragma unroll
        for (int e = 0; e < PER; ++e) o[e] = fmaf(w0, a[c][e], o[e]);
      }
    }
  }
  uint16_t* dst = out + row * D + lane * PER;
  if (ATTN_CHECKED(row * D + lane * PER, PER, rows * D, status)) {
    if constexpr (PER == 4) {
      uint2 pk;
      pk.x = pack_bf16x2(o[0], o[1]);
      pk.y = pack_bf16x2(o[2], o[3]);
      *reinterpret_cast<uint2*>(dst) = pk;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[0], o[1]);
    }
  }
  if (lse != nullptr && lane == 0 && ATTN_CHECKED(row, 1, rows, status)) lse[row] = L;
}

cudaError_t launch_merge(const float* o_part, const float* lse_part, uint16_t* out, float* lse, int n, long long rows,
                         int D, int* status, cudaStream_t stream) {
  long long grid = (rows + 7) / 8;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned g = (unsigned)grid;
  // the register kernels are launched with programmatic stream serialisation
  // (they wait for their predecessor themselves, see griddepcontrol above)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128) {
    if (n <= 8) return cudaLaunchKernelEx(&cfg, lse_merge_reg_kernel<128, 8>, o_part, lse_part, out, lse, n, rows, status);
    if (n <= 16) return cudaLaunchKernelEx(&cfg, lse_merge_reg_kernel<128, 16>, o_part, lse_part, out, lse, n, rows, status);
    lse_merge_kernel<128><<<g, 256, 0, stream>>>(o_part, lse_part, out, lse, n, rows, status);
  } else {
    if (n <= 8) return cudaLaunchKernelEx(&cfg, lse_merge_reg_kernel<64, 8>, o_part, lse_part, out, lse, n, rows, status);
    if (n <= 16) return cudaLaunchKernelEx(&cfg, lse_merge_reg_kernel<64, 16>, o_part, lse_part, out, lse, n, rows, status);
    lse_merge_kernel<64><<<g, 256, 0, stream>>>(o_part, lse_part, out, lse, n, rows, status);
  }
  return cudaGetLastError();
}

// ============================================================ bounded-wait self-test
// Every CTA's thread 0 waits on a barrier that nothing arrives on; the first
// wait to give up after limit_us records the timeout and aborts the launch,
// so the CTAs still waiting give up too and the CTAs that start afterwards
// return at once (the launch-wide abort of bounded_wait).
__global__ void wait_selftest_kernel(int* status, unsigned launch_id, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ WaitState wstate;
  __shared__ int skip_cta;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    skip_cta = wait_state_init(wstate, status, launch_id);
    fence_barrier_init();
  }
  __syncthreads();
  if (skip_cta) return;
  if (threadIdx.x == 0) bounded_wait(&bar, 0, &wstate, limit_ns);
}

cudaError_t launch_wait_selftest(int limit_us, int n_ctas, int smem_bytes, int* status, unsigned launch_id,
                                 cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(wait_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  wait_selftest_kernel<<<n_ctas, 32, smem_bytes, stream>>>(status, launch_id, (unsigned long long)limit_us * 1000ull);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- query-block order
// Per head and chunk of 128 query blocks, the blocks sorted by their selected-
// block count, longest first (ties: lower index first), written to order[bh][...]
// at the chunk's positions.  The sparse forward pairs the blocks in slots 2s
// and 2s + 1 in one CTA, whose time is that of the longer list: neighbours in
// this order have nearly equal lists.  A chunk keeps the blocks of 128
// consecutive query positions together (their keys overlap, as in the order
// of positions).  One CTA of 128 threads per (head, chunk); a count outside
// [0, NKB] sorts as its clamp.
__global__ void __launch_bounds__(128) qb_order_kernel(const int32_t* __restrict__ sel_cnt,
                                                       int32_t* __restrict__ order, int NQB, int NKB) {
  __shared__ uint32_t key[128];
  const int i = threadIdx.x;
  const int base = blockIdx.y * 128;
  const long long row = (long long)blockIdx.x * NQB;
  const int n = min(128, NQB - base);
  // key: (count + 1) above the local index's complement, so that a descending
  // sort puts longer lists first and, among equal ones, lower indices first;
  // padding (past the last block) gets 0 and sorts last
  uint32_t k = 0;
  if (i < n) {
    int c = __ldg(sel_cnt + row + base + i);
    c = c < 0 ? 0 : (c > NKB ? NKB : c);
    k = ((uint32_t)(c + 1) << 8) | (uint32_t)(127 - i);
  }
  key[i] = k;
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= 128; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int j = i ^ stride;
      if (j > i) {
        const uint32_t a = key[i], b = key[j];
        const bool desc = (i & size) == 0;
        if (desc ? a < b : a > b) {
          key[i] = b;
          key[j] = a;
        }
      }
      __syncthreads();
    }
  }
  if (i < n) order[row + base + i] = base + (127 - (int)(key[i] & 0xFFu));
}

cudaError_t launch_qb_order(const int32_t* sel_cnt, int32_t* order, int BH, int NQB, int NKB, cudaStream_t stream) {
  if (BH <= 0 || NQB <= 0 || (NQB + 127) / 128 > 65535 || NKB >= (1 << 23)) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)BH, (unsigned)((NQB + 127) / 128));
  qb_order_kernel<<<grid, 128, 0, stream>>>(sel_cnt, order, NQB, NKB);
  return cudaGetLastError();
}

}  // namespace vdtb
