// Sol-Attn routing on the tensor cores (tcgen05 kind::tf32): proxy scores,
// row statistics and threshold, selection with ascending compaction, and the
// Taylor aggregates W_i and T_i = sum_j w_ij Vbar_j of the rejected blocks.
//
// Source: "Accelerating LTX-2.5 with Sol Engine", section "Stage 2
// Optimization - Core Technology: Sol-Attn", bullets "Query-dependent
// thresholding" (tau_i = mu_i + beta sigma_i over the block proxy scores of
// query block i), "On-the-fly routing" (pooled keys, no proxy map in memory)
// and "Proxy-score reuse" (the rejected blocks' first-order Taylor term).
//
// CTA = one head and a tile of 128 query blocks; TMEM lane r holds query block
// i0 + r.  (A short last tile of up to 32 blocks goes to the CUDA-core kernel
// at the end of this file instead.)  Both products are tcgen05 GEMMs with fp32-grade accuracy from three
// tf32 products: every operand x is split into hi = x with its 13 low mantissa
// bits cleared (a tf32 value) and lo = x - hi (exact in fp32), and
// X.Y = Xh.Yh + Xh.Yl + Xl.Yh; the dropped Xl.Yl and the tf32 rounding of the
// lo parts are below 2^-20 of |X||Y| per term.
//   proxies  S = (scale Qbar) Kbar^T: A = Qbar hi/lo in TMEM (stored by the row
//            threads), B = pooled-key hi/lo slices from shared memory (TMA),
//            128 key blocks per chunk into 128 TMEM columns
//   Taylor   T = w Vbar: A = the weights' hi/lo slices in shared memory
//            (written by the row threads), B = slices of the transposed pooled
//            values (TMA), accumulated in TMEM over every key block
// The proxy row is never written to memory.  Two passes over the key chunks:
// pass 1 reduces each row's proxies to mean, M2 and argmax (thread r owns row
// r, so no cross-thread reduction); pass 2 recomputes every chunk with the
// same MMA sequence (bit-identical proxies), selects s >= tau or the argmax,
// appends the selected j to the row's list in ascending order, and turns the
// rejected proxies into Taylor weights w = n_j max(0, 1 + s - mu) for the T
// product.
//
// Warps 0-7: row threads, two per query block: warp w reads TMEM lanes
// 32 (w % 4) .. + 32 (its lane = its row) and half h = w / 4 of every chunk's
// 128 columns.  Warp 8, lane 0: TMA producer of the pooled-key ring.  Warp 9,
// lane 0: MMA issuer (and TMEM owner).  Warp 10, lane 0: TMA producer of the
// pooled-value ring (its own thread, so value loads start at once and never
// wait behind a key slot).  TMEM columns: Qbar hi [0, D), Qbar lo [D, 2D), S [256, 384),
// T [384, 384 + D).
#include <math.h>
#include <stdint.h>

#include "launch.h"

namespace vdtb {
namespace {

constexpr int kRtRows = 128;      // query blocks per CTA
constexpr int kRtChunk = 128;     // key blocks per proxy chunk (two halves of 64, one per row thread)
constexpr int kRtKStages = 2;     // pooled-key ring: one 32-wide d-slice of a chunk (hi + lo) per stage
constexpr int kRtVStages = 2;     // transposed pooled-value ring: one 32-wide key slice (hi + lo)
constexpr int kRtThreads = 352;
constexpr int kRtRowThreads = 256;
constexpr uint32_t kRtTmemCols = 512;
constexpr uint32_t kColS = 256, kColT = 384;

template <int D>
struct RtCfg {
  static constexpr int kDS = D / 32;                           // d-slices per chunk
  static constexpr int kKHalf = kRtChunk * 128;                // one slice of 128 keys x 32 fp32
  static constexpr int kKStageBytes = 2 * kKHalf;
  static constexpr int kVHalf = D * 128;                       // D rows x 32 fp32
  static constexpr int kVStageBytes = 2 * kVHalf;
  static constexpr int kWHalf = kRtRows * 128;                 // 128 rows x 32 fp32
  static constexpr int kWBytes = 2 * kWHalf;                   // one Taylor-weight slice, hi + lo
  static constexpr int kSmemBytes = 1024 + kRtKStages * kKStageBytes + kRtVStages * kVStageBytes + 2 * kWBytes;
  static_assert(D == 64 || D == 128, "head dim");
  // with the ~5 KB of static shared memory (barriers, exchange between a row's two threads)
  static_assert(kSmemBytes + 6 * 1024 <= 227 * 1024, "shared memory");
  static_assert(2 * D <= (int)kColS && kColT + D <= kRtTmemCols, "TMEM columns");
};

// The four 32-key slices of a chunk in the order they are multiplied: slice k
// comes from row-thread half k & 1 (which owns keys [64 h, 64 h + 64) of the
// chunk) and covers keys [32 js, 32 js + 32) of the chunk; half h always writes
// weight buffer h.
__host__ __device__ constexpr int rt_slice_js(int k) { return 2 * (k & 1) + (k >> 1); }

// tf32 split: hi keeps the sign, exponent and 10 mantissa bits of x; lo = x - hi exactly.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// One 128-byte row of a 128B-swizzled K-major operand tile (32 fp32 per row):
// row r at r * 128, its 16-byte chunk c at position c ^ (r & 7).
__device__ __forceinline__ void st_sw128_row(uint8_t* tile, int r, const float (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(tile + r * 128 + ((c ^ (r & 7)) << 4)) =
        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

__device__ __forceinline__ void rows_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kRtRowThreads) : "memory"); }

// Per-thread running statistics of its half of a row.
struct RowStats {
  float n, mean, m2, bmax;
  int bidx;
};

// Folds nh proxies x[0..nh) (keys base .. base + nh - 1) into the running
// mean / M2 (exact two-pass sums over the chunk, merged across chunks) and
// argmax (the lowest key on ties).  kFull: nh == 64.
template <bool kFull>
__device__ __forceinline__ void fold_stats(const float (&x)[64], int nh, int base, RowStats& st) {
  if (!kFull && nh <= 0) return;
  float cs[4] = {0.f, 0.f, 0.f, 0.f};
  float cmax = -INFINITY;
#pragma unroll
  for (int jj = 0; jj < 64; ++jj)
    if (kFull || jj < nh) {
      cs[jj & 3] += x[jj];
      cmax = fmaxf(cmax, x[jj]);
    }
  const float cn = kFull ? 64.f : (float)nh;
  const float cm = ((cs[0] + cs[1]) + (cs[2] + cs[3])) / cn;
  float c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int jj = 0; jj < 64; ++jj)
    if (kFull || jj < nh) {
      const float dv = x[jj] - cm;
      c2[jj & 3] = fmaf(dv, dv, c2[jj & 3]);
    }
  if (cmax > st.bmax) {   // strict: an earlier chunk keeps a tie
    st.bmax = cmax;
    bool found = false;
#pragma unroll
    for (int jj = 0; jj < 64; ++jj)
      if ((kFull || jj < nh) && !found && x[jj] == cmax) {
        st.bidx = base + jj;
        found = true;
      }
  }
  const float n = st.n + cn, delta = cm - st.mean;
  st.mean = fmaf(delta, cn / n, st.mean);
  st.m2 = st.m2 + ((c2[0] + c2[1]) + (c2[2] + c2[3])) + delta * delta * st.n * (cn / n);
  st.n = n;
}

// One 32-key slice of a half row in pass 2: selection bits (s >= tau, or the
// argmax at local index am) and Taylor weights w = n_j max(0, 1 + s - mu) of
// the rejected keys, split into tf32 hi / lo.  kFull: all 32 keys exist and
// none is the short last block.
template <bool kFull>
__device__ __forceinline__ uint32_t slice_weights(const float (&x)[64], int g, int nh, int am, int last, float tau,
                                                  float mu, float blk, float nlast, float (&wsum)[4],
                                                  float (&wh)[32], float (&wl)[32]) {
  uint32_t m = 0;
  const float blk1mu = blk * (1.f - mu);
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int jj = 32 * g + e;
    const float s = x[jj];
    bool keep = (s >= tau) || (jj == am);
    float w;
    if (kFull) {
      w = fmaxf(0.f, fmaf(blk, s, blk1mu));
    } else {
      const bool in = jj < nh;
      keep = keep && in;
      const float nb = (jj == last) ? nlast : blk;
      w = in ? nb * fmaxf(0.f, 1.f + s - mu) : 0.f;
    }
    w = keep ? 0.f : w;
    m |= (keep ? 1u : 0u) << e;
    wsum[e & 3] += w;
    wh[e] = tf32_hi(w);
    wl[e] = w - wh[e];
  }
  return m;
}

template <int D>
__global__ void __launch_bounds__(kRtThreads, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tm_kh, const __grid_constant__ CUtensorMap tm_kl,
                    const __grid_constant__ CUtensorMap tm_vh, const __grid_constant__ CUtensorMap tm_vl,
                    const __grid_constant__ CUtensorMap tm_q, int n_tiles, int NQB, int NKB, int S, int block_k,
                    float scale, float beta,
                    int32_t* __restrict__ sel_idx, int32_t* __restrict__ sel_cnt, float* __restrict__ stats,
                    float* __restrict__ taylor_t, int* status, unsigned launch_id) {
  using Cfg = RtCfg<D>;
  constexpr int kDS = Cfg::kDS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sK = smem;
  uint8_t* sV = sK + kRtKStages * Cfg::kKStageBytes;
  uint8_t* sW = sV + kRtVStages * Cfg::kVStageBytes;
  __shared__ uint64_t kfull[kRtKStages], kempty[kRtKStages], vfull[kRtVStages], vempty[kRtVStages];
  __shared__ uint64_t wfull[2], wfree[2];
  __shared__ uint64_t q_ready, q_full, s_full, s_free, t_done, mma_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ WaitState wstate;
  __shared__ int skip_cta;
  // exchange between the two row threads of a query block
  __shared__ float xch_f[4][kRtRows];
  __shared__ int xch_i[kRtRows];
  __shared__ int xch_cnt[2][2][kRtRows];
  WaitState* const wc = &wstate;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long bh = blockIdx.x / n_tiles;   // n_tiles: tiles of this head in the grid
  const int i0 = (blockIdx.x % n_tiles) * kRtRows;
  [[maybe_unused]] const long long nrows = (long long)(gridDim.x / n_tiles) * NQB;   // B * H * NQB
  const int nch = (NKB + kRtChunk - 1) / kRtChunk;

  if (tid == 0) {
    for (int s = 0; s < kRtKStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < kRtVStages; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&wfull[b], kRtRows);
      mbar_init(&wfree[b], 1);
    }
    mbar_init(&q_ready, kRtRowThreads);
    mbar_init(&q_full, 1);
    mbar_init(&s_full, 1);
    mbar_init(&s_free, kRtRowThreads);
    mbar_init(&t_done, 1);
    mbar_init(&mma_done, 1);
    skip_cta = wait_state_init(wstate, status, launch_id);
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(&tmem_base_sh, kRtTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  // a tail-rows kernel launched after this one may start on the SMs this grid leaves idle
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (!skip_cta) {
    if (warp == 8 || warp == 10) {
      // ======================= TMA producers (8: pooled keys, 10: transposed pooled values) =======================
      if (lane == 0 && warp == 8) {
        // the tile's pooled queries (fp32) into the weight buffers, which stay idle until pass 2
        mbar_expect_tx(&q_full, D * kRtRows * 4);
#pragma unroll
        for (int b = 0; b < D / 32; ++b) tma_load_3d(sW + b * (kRtRows * 128), &tm_q, &q_full, 32 * b, i0, (int)bh);
        tma_prefetch_desc(&tm_kh);
        tma_prefetch_desc(&tm_kl);
        int kl = 0;   // loads issued into the ring
        auto load_k = [&](int c) -> bool {
          for (int s = 0; s < kDS; ++s, ++kl) {
            const int st = kl % kRtKStages;
            if (kl >= kRtKStages && !bounded_wait(&kempty[st], ((kl / kRtKStages) - 1) & 1, wc)) return false;
            uint8_t* dst = sK + st * Cfg::kKStageBytes;
            mbar_expect_tx(&kfull[st], Cfg::kKStageBytes);
            tma_load_3d(dst, &tm_kh, &kfull[st], 32 * s, kRtChunk * c, (int)bh);
            tma_load_3d(dst + Cfg::kKHalf, &tm_kl, &kfull[st], 32 * s, kRtChunk * c, (int)bh);
          }
          return true;
        };
        // the order the MMA issuer consumes them: every chunk in pass 1, then again in pass 2
        bool ok = true;
        for (int c = 0; ok && c < nch; ++c) ok = load_k(c);
        for (int c = 0; ok && c < nch; ++c) ok = load_k(c);
        // drain: no copy may still be landing when the CTA exits
        for (int j = (kl > kRtKStages ? kl - kRtKStages : 0); j < kl; ++j)
          drain_wait(&kfull[j % kRtKStages], (j / kRtKStages) & 1, wc);
        drain_wait(&q_full, 0, wc);
      } else if (lane == 0) {
        tma_prefetch_desc(&tm_vh);
        tma_prefetch_desc(&tm_vl);
        int vl = 0;
        bool ok = true;
        for (int c = 0; ok && c < nch; ++c) {
          const int nj = min(kRtChunk, NKB - kRtChunk * c);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int js = rt_slice_js(k);
            if (!ok || 32 * js >= nj) continue;
            const int st = vl % kRtVStages;
            if (vl >= kRtVStages && !bounded_wait(&vempty[st], ((vl / kRtVStages) - 1) & 1, wc)) {
              ok = false;
              continue;
            }
            uint8_t* dst = sV + st * Cfg::kVStageBytes;
            mbar_expect_tx(&vfull[st], Cfg::kVStageBytes);
            tma_load_3d(dst, &tm_vh, &vfull[st], kRtChunk * c + 32 * js, 0, (int)bh);
            tma_load_3d(dst + Cfg::kVHalf, &tm_vl, &vfull[st], kRtChunk * c + 32 * js, 0, (int)bh);
            ++vl;
          }
        }
        for (int j = (vl > kRtVStages ? vl - kRtVStages : 0); j < vl; ++j)
          drain_wait(&vfull[j % kRtVStages], (j / kRtVStages) & 1, wc);
      }
    } else if (warp == 9) {
      // ======================= MMA issuer =======================
      if (lane == 0) {
        int kc = 0, vc = 0, sg = 0;   // key / value stages consumed, S chunks issued
        int wu[2] = {0, 0};           // uses of each weight buffer
        auto mma_s = [&](int c) -> bool {
          const int nj = min(kRtChunk, NKB - kRtChunk * c);
          const uint32_t idesc = idesc_tf32_f32(128, (nj + 15) & ~15);
          if (sg > 0) {   // the row threads have read the previous chunk out of the S columns
            if (!bounded_wait(&s_free, (sg - 1) & 1, wc)) return false;
            tc_fence_after();
          }
          for (int s = 0; s < kDS; ++s, ++kc) {
            const int st = kc % kRtKStages;
            if (!bounded_wait(&kfull[st], (kc / kRtKStages) & 1, wc)) return false;
            tc_fence_after();
            const uint32_t kh = smem_u32(sK + st * Cfg::kKStageBytes), klo = kh + Cfg::kKHalf;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t qcol = 32 * s + 8 * kk;
              const uint64_t bh_desc = smem_desc_sw128(kh + 32 * kk, 16, 1024);
              const uint64_t bl_desc = smem_desc_sw128(klo + 32 * kk, 16, 1024);
              mma_ts_tf32(tmem + kColS, tmem + qcol, bh_desc, idesc, (s > 0 || kk > 0) ? 1u : 0u);
              mma_ts_tf32(tmem + kColS, tmem + qcol, bl_desc, idesc, 1u);
              mma_ts_tf32(tmem + kColS, tmem + D + qcol, bh_desc, idesc, 1u);
            }
            mma_commit(&kempty[st]);
          }
          mma_commit(&s_full);
          ++sg;
          return true;
        };
        bool first_t = true;
        auto mma_t = [&](int c) -> bool {
          const int nj = min(kRtChunk, NKB - kRtChunk * c);
          constexpr uint32_t idesc = idesc_tf32_f32(128, D);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (32 * rt_slice_js(k) >= nj) continue;
            const int b = k & 1, st = vc % kRtVStages;
            if (!bounded_wait(&wfull[b], wu[b] & 1, wc) || !bounded_wait(&vfull[st], (vc / kRtVStages) & 1, wc))
              return false;
            tc_fence_after();
            const uint32_t wh = smem_u32(sW + b * Cfg::kWBytes), wl = wh + Cfg::kWHalf;
            const uint32_t vh = smem_u32(sV + st * Cfg::kVStageBytes), vlo = vh + Cfg::kVHalf;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ah = smem_desc_sw128(wh + 32 * kk, 16, 1024), al = smem_desc_sw128(wl + 32 * kk, 16, 1024);
              const uint64_t bh_desc = smem_desc_sw128(vh + 32 * kk, 16, 1024);
              const uint64_t bl_desc = smem_desc_sw128(vlo + 32 * kk, 16, 1024);
              mma_ss_tf32(tmem + kColT, ah, bh_desc, idesc, (first_t && kk == 0) ? 0u : 1u);
              mma_ss_tf32(tmem + kColT, ah, bl_desc, idesc, 1u);
              mma_ss_tf32(tmem + kColT, al, bh_desc, idesc, 1u);
            }
            first_t = false;
            mma_commit(&wfree[b]);
            mma_commit(&vempty[st]);
            ++wu[b];
            ++vc;
          }
          return true;
        };
        bool ok = bounded_wait(&q_ready, 0, wc);
        tc_fence_after();
        for (int c = 0; ok && c < nch; ++c) ok = mma_s(c);      // pass 1
        if (ok) ok = mma_s(0);                                   // pass 2
        for (int c = 0; ok && c < nch; ++c) {
          if (c + 1 < nch) ok = mma_s(c + 1);                    // the next chunk's proxies under this chunk's weights
          if (ok) ok = mma_t(c);
        }
        mma_commit(&t_done);
        // every MMA this thread issued has completed before TMEM is released
        mma_commit(&mma_done);
        drain_wait(&mma_done, 0, wc);
      }
    } else {
      // ======================= row threads (two per query block) =======================
      const int half = warp >> 2;
      const int r = (warp & 3) * 32 + lane;               // TMEM lane = row of the tile
      const int i = i0 + r;
      const bool valid = i < NQB;
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      // Qbar_i * scale, split into tf32 hi / lo, into this row's TMEM lane: half 0 stores hi, half 1 lo.
      // The tile arrives by TMA (128B-swizzled boxes of 32 columns), so each thread reads its row from
      // shared memory without bank conflicts.
      {
        bool qok = __all_sync(0xffffffffu, bounded_wait(&q_full, 0, wc));
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          const uint8_t* box = sW + (c0 / 32) * (kRtRows * 128) + r * 128;
          uint32_t part[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 v4 = qok ? *reinterpret_cast<const float4*>(box + ((c ^ (r & 7)) << 4))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            const float qs[4] = {v4.x * scale, v4.y * scale, v4.z * scale, v4.w * scale};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float h = tf32_hi(qs[u]);
              part[4 * c + u] = __float_as_uint(half == 0 ? h : qs[u] - h);
            }
          }
          tmem_st32(tmem + lane_base + half * D + c0, part);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&q_ready);
      }

      const uint32_t tS = tmem + lane_base + kColS + 64 * half;
      int sg = 0;
      bool ok = true;
      // Reads this half of the next S chunk (keys [64 half, 64 half + nh) of the chunk) and hands
      // the S columns back to the MMA issuer.  Returns false (having arrived anyway) on an abort.
      auto read_half = [&](int nh, float (&x)[64]) -> bool {
        const bool got = ok && __all_sync(0xffffffffu, bounded_wait(&s_full, sg & 1, wc));
        if (got) {
          tc_fence_after();
          uint32_t rr[2][32];
#pragma unroll
          for (int g = 0; g < 2; ++g)
            if (32 * g < nh) tmem_ld32(tS + 32 * g, rr[g]);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            tmem_reg_fence(rr[g]);
#pragma unroll
            for (int e = 0; e < 32; ++e) x[32 * g + e] = __uint_as_float(rr[g][e]);
          }
          tc_fence_before();
        }
        mbar_arrive(&s_free);
        ++sg;
        return got;
      };

      // ---- pass 1: mean / M2 and argmax of each half row, merged between the halves
      RowStats st{0.f, 0.f, 0.f, -INFINITY, INT_MAX};
      for (int c = 0; ok && c < nch; ++c) {
        const int nj = min(kRtChunk, NKB - kRtChunk * c);
        const int nh = min(64, nj - 64 * half);
        float x[64];
        if (!read_half(nh, x)) {
          ok = false;
          break;
        }
        if (nh == 64)
          fold_stats<true>(x, nh, kRtChunk * c + 64 * half, st);
        else
          fold_stats<false>(x, nh, kRtChunk * c + 64 * half, st);
      }
      if (half == 1) {
        xch_f[0][r] = st.n;
        xch_f[1][r] = st.mean;
        xch_f[2][r] = st.m2;
        xch_f[3][r] = st.bmax;
        xch_i[r] = st.bidx;
      }
      rows_sync();
      float mu, tau;
      int bidx;
      if (half == 0) {
        const float n1 = xch_f[0][r], m1 = xch_f[1][r], q1 = xch_f[2][r], b1 = xch_f[3][r];
        const int i1 = xch_i[r];
        const float n = st.n + n1;
        if (n1 > 0.f) {
          const float delta = m1 - st.mean;
          st.mean = fmaf(delta, n1 / n, st.mean);
          st.m2 = st.m2 + q1 + delta * delta * st.n * (n1 / n);
        }
        st.n = n;
        if (b1 > st.bmax || (b1 == st.bmax && i1 < st.bidx)) st.bidx = i1;
        mu = st.mean;
        const float sigma = sqrtf(fmaxf(st.m2, 0.f) / st.n);
        tau = (beta == -INFINITY) ? -INFINITY : fmaf(beta, sigma, mu);
        bidx = st.bidx;
        if (ok && valid && ATTN_CHECKED((bh * NQB + i) * 4, 3, nrows * 4, status)) {
          float* o = stats + (bh * NQB + i) * 4;
          o[0] = mu;
          o[1] = sigma;
          o[2] = tau;
        }
      }
      rows_sync();
      if (half == 0) {
        xch_f[0][r] = mu;
        xch_f[1][r] = tau;
        xch_i[r] = bidx;
      }
      rows_sync();
      if (half == 1) {
        mu = xch_f[0][r];
        tau = xch_f[1][r];
        bidx = xch_i[r];
      }
      ok = ok && !wstate.abort;

      // ---- pass 2: selection, ascending compaction, Taylor weights.  Every row thread runs
      // every chunk (and its row barrier) even after an abort, so the barrier counts match.
      int32_t* list = sel_idx + (bh * NQB + (valid ? i : 0)) * NKB;
      const float blk = (float)block_k;
      const float nlast = (float)(S - (NKB - 1) * block_k);
      int cnt = 0, wu = 0;
      float wsum[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < nch; ++c) {
        const int nj = min(kRtChunk, NKB - kRtChunk * c);
        const int nh = min(64, nj - 64 * half);
        const int base = kRtChunk * c + 64 * half;
        float x[64];
        const bool got = read_half(nh, x);
        ok = ok && got;
        uint32_t km[2] = {0u, 0u};
        const bool full = nh == 64 && !(c == nch - 1 && nlast != blk);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (!ok || 32 * g >= nh) break;
          if (wu > 0 && !__all_sync(0xffffffffu, bounded_wait(&wfree[half], (wu - 1) & 1, wc))) {
            ok = false;
            break;
          }
          float wh[32], wl[32];
          if (full)
            km[g] = slice_weights<true>(x, g, nh, bidx - base, NKB - 1 - base, tau, mu, blk, nlast, wsum, wh, wl);
          else
            km[g] = slice_weights<false>(x, g, nh, bidx - base, NKB - 1 - base, tau, mu, blk, nlast, wsum, wh, wl);
          uint8_t* wt = sW + half * Cfg::kWBytes;
          st_sw128_row(wt, r, wh);
          st_sw128_row(wt + Cfg::kWHalf, r, wl);
          // generic-proxy stores read by the tensor core (async proxy)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&wfull[half]);
          ++wu;
        }
        // list entries: this half's kept keys follow the other half's of earlier keys
        xch_cnt[c & 1][half][r] = __popc(km[0]) + __popc(km[1]);
        rows_sync();
        const int c0 = xch_cnt[c & 1][0][r], c1 = xch_cnt[c & 1][1][r];
        int pos = cnt + (half == 1 ? c0 : 0);
        cnt += c0 + c1;
        if (ok && valid) {
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t m = km[g];
            while (m != 0u) {
              const int e = __ffs(m) - 1;
              m &= m - 1u;
              if (ATTN_CHECKED((bh * NQB + i) * NKB + pos, 1, nrows * NKB, status)) list[pos] = base + 32 * g + e;
              ++pos;
            }
          }
        }
      }

      // ---- W (both halves' weights), counts, and T out of TMEM
      if (half == 1) xch_f[2][r] = (wsum[0] + wsum[1]) + (wsum[2] + wsum[3]);
      rows_sync();
      if (half == 0 && ok && valid) {
        const float W = ((wsum[0] + wsum[1]) + (wsum[2] + wsum[3])) + xch_f[2][r];
        if (ATTN_CHECKED((bh * NQB + i) * 4 + 3, 1, nrows * 4, status)) stats[(bh * NQB + i) * 4 + 3] = W;
        if (ATTN_CHECKED(bh * NQB + i, 1, nrows, status)) sel_cnt[bh * NQB + i] = cnt;
      }
      // T: out of TMEM into the idle key ring (row r's 16-byte chunk c at position c ^ (r & 31), so
      // that both the row-wise writes and the later chunk-wise reads are free of bank conflicts), then
      // each warp stores whole rows to global memory with coalesced 512-byte writes
      const bool tok = ok && __all_sync(0xffffffffu, bounded_wait(&t_done, 0, wc)) && !wstate.abort;
      constexpr int kChunks = D / 4;   // 16-byte chunks per T row
      float* sT = reinterpret_cast<float*>(sK);
      if (tok) {
        tc_fence_after();
        constexpr int kHalfD = D / 2;
        const uint32_t tT = tmem + lane_base + kColT + half * kHalfD;
#pragma unroll
        for (int c0 = 0; c0 < kHalfD; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tT + c0, rr);
          tmem_ld_wait();
          tmem_reg_fence(rr);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int chunk = (half * kHalfD + c0 + e) / 4;
            *reinterpret_cast<float4*>(sT + r * D + 4 * (chunk ^ (r & (kChunks - 1)))) =
                make_float4(__uint_as_float(rr[e]), __uint_as_float(rr[e + 1]), __uint_as_float(rr[e + 2]),
                            __uint_as_float(rr[e + 3]));
          }
        }
      }
      rows_sync();
      if (tok) {
        for (int row = warp; row < kRtRows; row += 8) {
          const int ig = i0 + row;
          if (ig >= NQB) break;
          for (int chunk = lane; chunk < kChunks; chunk += 32) {
            const float4 v4 = *reinterpret_cast<const float4*>(sT + row * D + 4 * (chunk ^ (row & (kChunks - 1))));
            const long long off = (bh * NQB + ig) * D + 4 * chunk;
            if (ATTN_CHECKED(off, 4, nrows * D, status)) *reinterpret_cast<float4*>(taylor_t + off) = v4;
          }
        }
      }
    }
  }   // !skip_cta

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kRtTmemCols);
  }
}

// ============================================================ tail rows on the CUDA cores
// The tensor-core kernel works on tiles of 128 query blocks, one CTA per SM.
// A head whose query-block count leaves a short last tile (the Stage-2
// sequence: 513 blocks = 4 x 128 + 1) would spend a whole CTA, with all of its
// key and value traffic, on a few rows, and push the grid into a second wave.
// Those rows go to this kernel instead, one CTA per (head, row), which runs
// beside the tensor-core kernel on the SMs it leaves idle (programmatic
// dependent launch).  Same definitions in fp32 on the CUDA cores: the row's
// proxies s_j = (scale Qbar_i) . Kbar_j, one warp per key block (coalesced
// 512-byte row loads, shuffle reduction), are kept in shared memory (so the
// selection pass needs no recomputation); mean, population std and argmax
// (lowest j on ties) by block reductions; selection s_j >= tau or the argmax,
// compacted in ascending j with ballot/popc; Taylor weights w_j = n_j max(0,
// 1 + s_j - mu) of the rejected blocks; W = sum w_j and T = sum w_j Vbar_j with
// every thread holding a float4 of columns for one residue class of j.
constexpr int kTailThreads = 256;
constexpr int kTailWarps = kTailThreads / 32;

__device__ __forceinline__ float tail_block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kTailWarps; ++w) t += red[w];
  return t;
}

template <int D>
__global__ void __launch_bounds__(kTailThreads) route_tail_kernel(
    const float* __restrict__ qp, const float* __restrict__ kp, const float* __restrict__ vp, int NQB, int NKB, int S,
    int block_k, float scale, float beta, int32_t* __restrict__ sel_idx, int32_t* __restrict__ sel_cnt,
    float* __restrict__ stats, float* __restrict__ taylor_t, int row_lo, int* status) {
  extern __shared__ __align__(16) float srow[];   // NKB proxies, then Taylor weights
  __shared__ float qs[D];
  __shared__ float red[kTailWarps];
  __shared__ int redi[kTailWarps];
  __shared__ float tred[kTailThreads / (D / 4)][D];
  const int nrow = NQB - row_lo;
  const long long bh = blockIdx.x / nrow;
  const int i = row_lo + blockIdx.x % nrow;
  [[maybe_unused]] const long long nrows = (long long)(gridDim.x / nrow) * NQB;   // B * H * NQB
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* kh = kp + bh * NKB * D;
  const float* vh = vp + bh * NKB * D;
  if (tid < D) qs[tid] = scale * __ldg(qp + (bh * NQB + i) * D + tid);
  __syncthreads();

  // proxies: warp per key block, lanes across the row (float4 for d = 128, float2 for d = 64)
  constexpr int PER = D / 32;
  float q[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) q[e] = qs[lane * PER + e];
  for (int j0 = warp; j0 < NKB; j0 += 8 * kTailWarps) {
    float part[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * kTailWarps;
      float a = 0.f;
      if (j < NKB) {
        const float* kr = kh + (long long)j * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 k4 = __ldg(reinterpret_cast<const float4*>(kr));
          a = fmaf(q[0], k4.x, fmaf(q[1], k4.y, fmaf(q[2], k4.z, q[3] * k4.w)));
        } else {
          const float2 k2 = __ldg(reinterpret_cast<const float2*>(kr));
          a = fmaf(q[0], k2.x, q[1] * k2.y);
        }
      }
      part[u] = a;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part[u] += __shfl_xor_sync(0xffffffffu, part[u], o);
      const int j = j0 + u * kTailWarps;
      if (lane == 0 && j < NKB) srow[j] = part[u];
    }
  }
  __syncthreads();

  // mean, then the population variance about it (two passes), and the argmax
  float sum = 0.f, best = -INFINITY;
  int bidx = INT_MAX;
  for (int j = tid; j < NKB; j += kTailThreads) {
    const float v = srow[j];
    sum += v;
    if (v > best) {   // j increases within a thread: strict > keeps the lowest j
      best = v;
      bidx = j;
    }
  }
  const float mu = tail_block_sum(sum, red) / (float)NKB;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (ob > best || (ob == best && oi < bidx)) {
      best = ob;
      bidx = oi;
    }
  }
  __syncthreads();
  if (lane == 0) {
    red[warp] = best;
    redi[warp] = bidx;
  }
  __syncthreads();
  best = red[0];
  bidx = redi[0];
#pragma unroll
  for (int w = 1; w < kTailWarps; ++w)
    if (red[w] > best || (red[w] == best && redi[w] < bidx)) {
      best = red[w];
      bidx = redi[w];
    }
  float sq = 0.f;
  for (int j = tid; j < NKB; j += kTailThreads) {
    const float dv = srow[j] - mu;
    sq = fmaf(dv, dv, sq);
  }
  const float sigma = sqrtf(tail_block_sum(sq, red) / (float)NKB);
  const float tau = (beta == -INFINITY) ? -INFINITY : fmaf(beta, sigma, mu);

  // selection in ascending j (ballot / popc within a warp, warp counts through shared memory),
  // Taylor weights over the proxies
  int32_t* list = sel_idx + (bh * NQB + i) * NKB;
  int cnt = 0;
  float wsum = 0.f;
  for (int j0 = 0; j0 < NKB; j0 += kTailThreads) {
    const int j = j0 + tid;
    const bool in = j < NKB;
    const float v = in ? srow[j] : 0.f;
    const bool keep = in && (v >= tau || j == bidx);
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    __syncthreads();
    if (lane == 0) redi[warp] = __popc(m);
    __syncthreads();
    int before = cnt, total = 0;
#pragma unroll
    for (int w = 0; w < kTailWarps; ++w) {
      if (w < warp) before += redi[w];
      total += redi[w];
    }
    const int slot = before + __popc(m & ((1u << lane) - 1u));
    if (keep && ATTN_CHECKED((bh * NQB + i) * NKB + slot, 1, nrows * NKB, status)) list[slot] = j;
    cnt += total;
    if (in) {
      const float w = keep ? 0.f : (float)min(block_k, S - j * block_k) * fmaxf(0.f, 1.f + v - mu);
      srow[j] = w;
      wsum += w;
    }
  }
  const float W = tail_block_sum(wsum, red);

  // T = sum_j w_j Vbar_j: thread = (column quad, residue class of j)
  constexpr int NQ = D / 4, NG = kTailThreads / NQ;
  const int cq = tid % NQ, g = tid / NQ;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int kU = 8;   // loads in flight per thread
  for (int j0 = g; j0 < NKB; j0 += kU * NG) {
    float4 v4[kU];
    float w[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = j0 + u * NG;
      w[u] = j < NKB ? srow[j] : 0.f;
      v4[u] = w[u] != 0.f ? __ldg(reinterpret_cast<const float4*>(vh + (long long)j * D) + cq)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      acc.x = fmaf(w[u], v4[u].x, acc.x);
      acc.y = fmaf(w[u], v4[u].y, acc.y);
      acc.z = fmaf(w[u], v4[u].z, acc.z);
      acc.w = fmaf(w[u], v4[u].w, acc.w);
    }
  }
  *reinterpret_cast<float4*>(&tred[g][4 * cq]) = acc;
  __syncthreads();
  if (tid < D) {
    float t = 0.f;
#pragma unroll
    for (int gg = 0; gg < NG; ++gg) t += tred[gg][tid];
    if (ATTN_CHECKED((bh * NQB + i) * D + tid, 1, nrows * D, status)) taylor_t[(bh * NQB + i) * D + tid] = t;
  }
  if (tid == 0) {
    if (ATTN_CHECKED((bh * NQB + i) * 4, 4, nrows * 4, status)) {
      float* st = stats + (bh * NQB + i) * 4;
      st[0] = mu;
      st[1] = sigma;
      st[2] = tau;
      st[3] = W;
    }
    if (ATTN_CHECKED(bh * NQB + i, 1, nrows, status)) sel_cnt[bh * NQB + i] = cnt;
  }
  // launched beside the tensor-core kernel (programmatic dependent launch): do not complete before it
  // has, so that work queued after this kernel sees both kernels' results
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

// Largest short last tile (query blocks) that goes to the CUDA-core kernel.
constexpr int kTailRowsMax = 32;

cudaError_t launch_route_tc(const CUtensorMap& tkh, const CUtensorMap& tkl, const CUtensorMap& tvh,
                            const CUtensorMap& tvl, const CUtensorMap& tq, const float* qp, const float* kp,
                            const float* vp, int BH, int NQB, int NKB, int S, int D, int block_k, float scale,
                            float beta, int32_t* sel_idx, int32_t* sel_cnt, float* stats, float* taylor_t, int* status,
                            unsigned launch_id, cudaStream_t stream) {
  const int rem = NQB % kRtRows;
  const bool tail = rem != 0 && rem <= kTailRowsMax;
  const int tc_tiles = tail ? NQB / kRtRows : (NQB + kRtRows - 1) / kRtRows;
  const long long grid = (long long)BH * tc_tiles;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  if (grid > 0) {
    if (D == 128) {
      e = cudaFuncSetAttribute(route_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               RtCfg<128>::kSmemBytes);
      if (e != cudaSuccess) return e;
      route_tc_kernel<128><<<(unsigned)grid, kRtThreads, RtCfg<128>::kSmemBytes, stream>>>(
          tkh, tkl, tvh, tvl, tq, tc_tiles, NQB, NKB, S, block_k, scale, beta, sel_idx, sel_cnt, stats, taylor_t,
          status, launch_id);
    } else {
      e = cudaFuncSetAttribute(route_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               RtCfg<64>::kSmemBytes);
      if (e != cudaSuccess) return e;
      route_tc_kernel<64><<<(unsigned)grid, kRtThreads, RtCfg<64>::kSmemBytes, stream>>>(
          tkh, tkl, tvh, tvl, tq, tc_tiles, NQB, NKB, S, block_k, scale, beta, sel_idx, sel_cnt, stats, taylor_t,
          status, launch_id);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (!tail) return cudaSuccess;
  const int row_lo = tc_tiles * kRtRows;
  const long long tgrid = (long long)BH * (NQB - row_lo);
  if (tgrid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tgrid);
  cfg.blockDim = dim3(kTailThreads);
  cfg.dynamicSmemBytes = (size_t)NKB * 4;   // NKB <= 8192: at most 32 KB
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = grid > 0 ? 1 : 0;
  if (D == 128)
    return cudaLaunchKernelEx(&cfg, route_tail_kernel<128>, qp, kp, vp, NQB, NKB, S, block_k, scale, beta, sel_idx,
                              sel_cnt, stats, taylor_t, row_lo, status);
  return cudaLaunchKernelEx(&cfg, route_tail_kernel<64>, qp, kp, vp, NQB, NKB, S, block_k, scale, beta, sel_idx,
                            sel_cnt, stats, taylor_t, row_lo, status);
}

}  // namespace vdtb
