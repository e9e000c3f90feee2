// Bandwidth/ALU-bound kernels of the hot path: block mean-pool, Sol-Attn
// routing (proxy scores, Welford statistics, threshold, ballot/popc
// compaction, Taylor aggregates) and the exact log-sum-exp merge of split-KV
// partials.
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
// loads, then the row groups are summed through shared memory.
// Source: "Accelerating LTX-2.5 with Sol Engine", Sol-Attn bullet
// "On-the-fly routing" (pooled keys).
template <int D>
__global__ void __launch_bounds__(256) pool_kernel(const uint16_t* __restrict__ x0, const uint16_t* __restrict__ x1,
                                                   const uint16_t* __restrict__ x2, float* __restrict__ p0,
                                                   float* __restrict__ p1, float* __restrict__ p2, int S, int block,
                                                   int NB) {
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
    xp[(bh * NB + i) * D + threadIdx.x] = s / (float)(hi - lo);
  }
}

cudaError_t launch_pool(const uint16_t* x0, const uint16_t* x1, const uint16_t* x2, float* p0, float* p1, float* p2,
                        int ntensors, int BH, int S, int D, int block, cudaStream_t stream) {
  const int NB = (S + block - 1) / block;
  long long nblk = (long long)BH * NB;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)nblk, ntensors);
  if (D == 128)
    pool_kernel<128><<<grid, 256, 0, stream>>>(x0, x1, x2, p0, p1, p2, S, block, NB);
  else
    pool_kernel<64><<<grid, 256, 0, stream>>>(x0, x1, x2, p0, p1, p2, S, block, NB);
  return cudaGetLastError();
}

// ============================================================ routing
// One CTA per (head, 32 query blocks); 256 threads.  Pooled keys stream
// through shared memory in chunks of 32 key blocks, twice:
//   pass 1: proxy scores s_ij = scale * Qbar_i . Kbar_j, per-thread Welford
//           mean/M2 and argmax, merged across the 16 threads of a row group
//           (Chan's pairwise update) -> mu_i, sigma_i, tau_i = mu_i + beta sigma_i
//   pass 2: the same scores recomputed bit-for-bit, selection
//           s_ij >= tau_i or j = argmax, compaction of the selected j into an
//           ascending list with ballot/popc, and the Taylor weights
//           w_ij = n_j max(0, 1 + s_ij - mu_i) of rejected blocks folded into
//           W_i and T_i = sum w_ij Vbar_j.
// The proxy row is never written to memory.
// Source: "Accelerating LTX-2.5 with Sol Engine", section "Stage 2
// Optimization - Core Technology: Sol-Attn".
constexpr int kRouteRows = 32;   // query blocks per CTA
constexpr int kRouteChunk = 32;  // key blocks per streamed chunk

template <int D>
struct RouteSmem {
  static constexpr int LD = D + 4;  // padded row stride (floats): conflict-free float4 column reads
  float q[kRouteRows][LD];
  float k[kRouteChunk][LD];
  float v[kRouteChunk][LD];
  float w[kRouteRows][kRouteChunk + 1];
  float mu[kRouteRows], tau[kRouteRows];
  int amax[kRouteRows];
};

template <int D>
__device__ __forceinline__ void route_scores(const RouteSmem<D>& sm, int ti, int tj, float scale, float (&s)[2][2]) {
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 8
  for (int c = 0; c < D; c += 4) {
    const float4 q0 = *reinterpret_cast<const float4*>(&sm.q[ti][c]);
    const float4 q1 = *reinterpret_cast<const float4*>(&sm.q[ti + 16][c]);
    const float4 k0 = *reinterpret_cast<const float4*>(&sm.k[tj][c]);
    const float4 k1 = *reinterpret_cast<const float4*>(&sm.k[tj + 16][c]);
    acc[0][0] = fmaf(q0.x, k0.x, fmaf(q0.y, k0.y, fmaf(q0.z, k0.z, fmaf(q0.w, k0.w, acc[0][0]))));
    acc[0][1] = fmaf(q0.x, k1.x, fmaf(q0.y, k1.y, fmaf(q0.z, k1.z, fmaf(q0.w, k1.w, acc[0][1]))));
    acc[1][0] = fmaf(q1.x, k0.x, fmaf(q1.y, k0.y, fmaf(q1.z, k0.z, fmaf(q1.w, k0.w, acc[1][0]))));
    acc[1][1] = fmaf(q1.x, k1.x, fmaf(q1.y, k1.y, fmaf(q1.z, k1.z, fmaf(q1.w, k1.w, acc[1][1]))));
  }
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 2; ++b) s[a][b] = scale * acc[a][b];
}

template <int D>
__device__ __forceinline__ void route_load_rows(float (*dst)[D + 4], const float* __restrict__ src, int row0,
                                                int nrows_total, int nrows) {
  // nrows rows of D floats starting at src row row0 (rows >= nrows_total are zero)
  constexpr int F4 = D / 4;
  for (int e = threadIdx.x; e < nrows * F4; e += blockDim.x) {
    const int r = e / F4, c = (e % F4) * 4;
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + r < nrows_total) val = __ldg(reinterpret_cast<const float4*>(src + (long long)(row0 + r) * D + c));
    *reinterpret_cast<float4*>(&dst[r][c]) = val;
  }
}

// One chunk of pooled rows held in registers (D/32 float4 per thread of 256):
// the next chunk is fetched while the current one is being used from shared
// memory, so the L2 latency of the stream overlaps the arithmetic.
template <int D>
struct ChunkRegs {
  float4 v[D / 32];
  __device__ __forceinline__ void load(const float* __restrict__ src, int row0, int nrows_total) {
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      const int e = threadIdx.x + k * 256;
      const int r = e / (D / 4), c = (e % (D / 4)) * 4;
      v[k] = (row0 + r < nrows_total) ? __ldg(reinterpret_cast<const float4*>(src + (long long)(row0 + r) * D + c))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __device__ __forceinline__ void store(float (*dst)[D + 4]) const {
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      const int e = threadIdx.x + k * 256;
      *reinterpret_cast<float4*>(&dst[e / (D / 4)][(e % (D / 4)) * 4]) = v[k];
    }
  }
};

template <int D>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ qp, const float* __restrict__ kp,
                                                    const float* __restrict__ vp, int NQB, int NKB, int S,
                                                    int block_k, float scale, float beta, int32_t* __restrict__ sel_idx,
                                                    int32_t* __restrict__ sel_cnt, float* __restrict__ stats,
                                                    float* __restrict__ taylor_t) {
  extern __shared__ __align__(16) uint8_t route_smem_raw[];
  RouteSmem<D>& sm = *reinterpret_cast<RouteSmem<D>*>(route_smem_raw);
  const int n_groups = (NQB + kRouteRows - 1) / kRouteRows;
  const long long bh = blockIdx.x / n_groups;
  const int i0 = (blockIdx.x % n_groups) * kRouteRows;
  const int tid = threadIdx.x;
  const int ti = tid >> 4, tj = tid & 15;
  const float* kh = kp + bh * NKB * D;
  const float* vh = vp + bh * NKB * D;

  route_load_rows<D>(sm.q, qp + bh * NQB * D, i0, NQB, kRouteRows);

  // ---------------- pass 1: Welford mean / M2 and argmax per row
  float wn[2] = {0.f, 0.f}, wmean[2] = {0.f, 0.f}, wm2[2] = {0.f, 0.f};
  float bmax[2] = {-INFINITY, -INFINITY};
  int bidx[2] = {INT_MAX, INT_MAX};
  ChunkRegs<D> kreg;
  kreg.load(kh, 0, NKB);
  for (int j0 = 0; j0 < NKB; j0 += kRouteChunk) {
    __syncthreads();
    kreg.store(sm.k);
    if (j0 + kRouteChunk < NKB) kreg.load(kh, j0 + kRouteChunk, NKB);
    __syncthreads();
    float s[2][2];
    route_scores<D>(sm, ti, tj, scale, s);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int j = j0 + tj + 16 * b;
      if (j >= NKB) continue;
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        wn[a] += 1.f;
        const float delta = s[a][b] - wmean[a];
        wmean[a] += delta / wn[a];
        wm2[a] = fmaf(delta, s[a][b] - wmean[a], wm2[a]);
        if (s[a][b] > bmax[a]) {  // j increases within a thread: strict > keeps the lowest j
          bmax[a] = s[a][b];
          bidx[a] = j;
        }
      }
    }
  }
  // merge the 16 partial states of each row (lanes of one half-warp)
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) {
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const float on = __shfl_xor_sync(0xffffffffu, wn[a], off);
      const float om = __shfl_xor_sync(0xffffffffu, wmean[a], off);
      const float o2 = __shfl_xor_sync(0xffffffffu, wm2[a], off);
      const float ob = __shfl_xor_sync(0xffffffffu, bmax[a], off);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx[a], off);
      const float n = wn[a] + on;
      if (n > 0.f) {
        const float delta = om - wmean[a];
        const float nb_n = on / n;
        wmean[a] = fmaf(delta, nb_n, wmean[a]);
        wm2[a] = wm2[a] + o2 + delta * delta * wn[a] * nb_n;
      }
      wn[a] = n;
      if (ob > bmax[a] || (ob == bmax[a] && oi < bidx[a])) {
        bmax[a] = ob;
        bidx[a] = oi;
      }
    }
  }
  if (tj == 0) {
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int row = ti + 16 * a;
      const float mu = wmean[a];
      const float sigma = sqrtf(fmaxf(wm2[a], 0.f) / wn[a]);
      const float tau = (beta == -INFINITY) ? -INFINITY : fmaf(beta, sigma, mu);
      sm.mu[row] = mu;
      sm.tau[row] = tau;
      sm.amax[row] = bidx[a];
      const int i = i0 + row;
      if (i < NQB) {
        float* st = stats + (bh * NQB + i) * 4;
        st[0] = mu;
        st[1] = sigma;
        st[2] = tau;
      }
    }
  }
  __syncthreads();

  // ---------------- pass 2: selection, compaction, Taylor aggregates
  float mu_r[2], tau_r[2];
  int am_r[2];
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    mu_r[a] = sm.mu[ti + 16 * a];
    tau_r[a] = sm.tau[ti + 16 * a];
    am_r[a] = sm.amax[ti + 16 * a];
  }
  int cnt[2] = {0, 0};
  // T accumulation layout: thread -> row tr, columns tc + 32 m
  const int tr = tid >> 3, tc = (tid & 7) * 4;
  float tacc[D / 32][4];
#pragma unroll
  for (int m = 0; m < D / 32; ++m) tacc[m][0] = tacc[m][1] = tacc[m][2] = tacc[m][3] = 0.f;
  float wsum = 0.f;
  ChunkRegs<D> vreg;
  kreg.load(kh, 0, NKB);
  vreg.load(vh, 0, NKB);
  for (int j0 = 0; j0 < NKB; j0 += kRouteChunk) {
    __syncthreads();
    kreg.store(sm.k);
    vreg.store(sm.v);
    if (j0 + kRouteChunk < NKB) {
      kreg.load(kh, j0 + kRouteChunk, NKB);
      vreg.load(vh, j0 + kRouteChunk, NKB);
    }
    __syncthreads();
    float s[2][2];
    route_scores<D>(sm, ti, tj, scale, s);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int row = ti + 16 * a;
      const int i = i0 + row;
      uint32_t bits = 0;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int col = tj + 16 * b;
        const int j = j0 + col;
        float w = 0.f;
        if (j < NKB) {
          const bool keep = (s[a][b] >= tau_r[a]) || (j == am_r[a]);
          if (keep) {
            bits |= 1u << col;
          } else {
            const int nj = min(block_k, S - j * block_k);
            w = (float)nj * fmaxf(0.f, 1.f + s[a][b] - mu_r[a]);
          }
        }
        sm.w[row][col] = w;
      }
      uint32_t mask = bits;  // OR over the 16 lanes of this row group (xor < 16 stays in the half-warp)
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mask |= __shfl_xor_sync(0xffffffffu, mask, off);
      if (i < NQB) {
        int32_t* list = sel_idx + (bh * NQB + i) * NKB;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int col = tj + 16 * b;
          if (bits & (1u << col)) list[cnt[a] + __popc(mask & ((1u << col) - 1u))] = j0 + col;
        }
      }
      cnt[a] += __popc(mask);
    }
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < kRouteChunk; ++jj) {
      const float w = sm.w[tr][jj];
      wsum += w;
#pragma unroll
      for (int m = 0; m < D / 32; ++m) {
        const float4 vv = *reinterpret_cast<const float4*>(&sm.v[jj][tc + 32 * m]);
        tacc[m][0] = fmaf(w, vv.x, tacc[m][0]);
        tacc[m][1] = fmaf(w, vv.y, tacc[m][1]);
        tacc[m][2] = fmaf(w, vv.z, tacc[m][2]);
        tacc[m][3] = fmaf(w, vv.w, tacc[m][3]);
      }
    }
  }
  if (tj == 0) {
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int i = i0 + ti + 16 * a;
      if (i < NQB) sel_cnt[bh * NQB + i] = cnt[a];
    }
  }
  const int i = i0 + tr;
  if (i < NQB) {
    float* dst = taylor_t + (bh * NQB + i) * D;
#pragma unroll
    for (int m = 0; m < D / 32; ++m)
      *reinterpret_cast<float4*>(dst + tc + 32 * m) = make_float4(tacc[m][0], tacc[m][1], tacc[m][2], tacc[m][3]);
    if ((tid & 7) == 0) stats[(bh * NQB + i) * 4 + 3] = wsum;
  }
}

cudaError_t launch_route(const float* qp, const float* kp, const float* vp, int BH, int NQB, int NKB, int S, int D,
                         int block_k, float scale, float beta, int32_t* sel_idx, int32_t* sel_cnt, float* stats,
                         float* taylor_t, cudaStream_t stream) {
  const int n_groups = (NQB + kRouteRows - 1) / kRouteRows;
  long long grid = (long long)BH * n_groups;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  if (D == 128) {
    const int smem = (int)sizeof(RouteSmem<128>);
    e = cudaFuncSetAttribute(route_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    route_kernel<128><<<(unsigned)grid, 256, smem, stream>>>(qp, kp, vp, NQB, NKB, S, block_k, scale, beta, sel_idx,
                                                             sel_cnt, stats, taylor_t);
  } else {
    const int smem = (int)sizeof(RouteSmem<64>);
    e = cudaFuncSetAttribute(route_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    route_kernel<64><<<(unsigned)grid, 256, smem, stream>>>(qp, kp, vp, NQB, NKB, S, block_k, scale, beta, sel_idx,
                                                            sel_cnt, stats, taylor_t);
  }
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
                                                        float* __restrict__ lse, int n, long long rows) {
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
  if constexpr (PER == 4) {
    uint2 pk;
    pk.x = pack_bf16x2(o[0], o[1]);
    pk.y = pack_bf16x2(o[2], o[3]);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[0], o[1]);
  }
  if (lse != nullptr && lane == 0) lse[row] = L;
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
                                                            long long rows) {
  constexpr int PER = D / 32;
  // programmatic dependent launch: let the next kernel in the stream start its
  // launch now, and wait until the kernel before this one (which may have
  // produced the partials) has completed and its writes are visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
  if constexpr (PER == 4) {
    uint2 pk;
    pk.x = pack_bf16x2(o[0], o[1]);
    pk.y = pack_bf16x2(o[2], o[3]);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[0], o[1]);
  }
  if (lse != nullptr && lane == 0) lse[row] = L;
}

cudaError_t launch_merge(const float* o_part, const float* lse_part, uint16_t* out, float* lse, int n, long long rows,
                         int D, cudaStream_t stream) {
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
    if (n <= 8) return cudaLaunchKernelEx(&cfg, lse_merge_reg_kernel<128, 8>, o_part, lse_part, out, lse, n, rows);
    if (n <= 16) return cudaLaunchKernelEx(&cfg, lse_merge_reg_kernel<128, 16>, o_part, lse_part, out, lse, n, rows);
    lse_merge_kernel<128><<<g, 256, 0, stream>>>(o_part, lse_part, out, lse, n, rows);
  } else {
    if (n <= 8) return cudaLaunchKernelEx(&cfg, lse_merge_reg_kernel<64, 8>, o_part, lse_part, out, lse, n, rows);
    if (n <= 16) return cudaLaunchKernelEx(&cfg, lse_merge_reg_kernel<64, 16>, o_part, lse_part, out, lse, n, rows);
    lse_merge_kernel<64><<<g, 256, 0, stream>>>(o_part, lse_part, out, lse, n, rows);
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

}  // namespace vdtb
