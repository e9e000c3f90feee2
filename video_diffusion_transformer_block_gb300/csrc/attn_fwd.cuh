// tcgen05 attention forward for sm_103a: dense, block-sparse (selected-block
// lists + Taylor term) and split-KV (chunk partials) share one main loop.
//
// CTA = NQT query tiles of 128 rows.  Three layouts:
//  - two-issuer CTA (dense and sparse, NQT = 2, one CTA per SM): the two tiles
//    run like two one-tile CTAs, each with its own list walk, its own two K/V
//    slots, its own TMA producer warp and MMA-issuing warp; the issuers take a
//    shared-memory lock around each step's MMA batch.  Two one-tile CTAs on an
//    SM were measured to fall into step with each other (both issuing MMAs,
//    then both in softmax, with the tensor pipe idle); the lock makes one
//    tile's batch run while the other tile's softmax does.  Per tile and step
//    one full barrier (K of key tile s with V of key tile s-1) and one commit
//    (S ready, both slots free): each barrier operation of an issuer costs
//    100-200 clocks while the score MMAs keep shared memory busy.
//  - one-tile CTA, two per SM: split-KV (the same per-tile roles) and the
//    one-brick neighbourhood plans (one producer, one issuer, a full/empty
//    barrier pair per slot).
//  - shared-walk two-tile CTA (fused routing, paired neighbourhood plans):
//    one producer and one issuer walk the union of the tiles' lists and every
//    K/V load serves both tiles.
//   warps 0..4*NQT-1 : softmax/epilogue, one warpgroup per query tile; thread
//                      r of the warpgroup owns query row r = TMEM lane r
//   warp  4*NQT      : TMA producer (Q once, then K_s, V_s for every step s
//                      into the K/V slots)
//   warp  4*NQT+1    : tcgen05 MMA issuer (one thread); allocates TMEM
//   (two-issuer CTA: warps 8, 9 are tile 0's producer and issuer, 10, 11 tile 1's)
// TMEM, per query tile t: S_t at columns [256t, 256t+BK) in fp32; P_t (bf16
// pairs) overwrites the first BK/2 columns of S_t; O_t at [256t+128, +D).
// Per step s: S_t = Q_t K_s^T (SS MMA, both K-major, 128B swizzle), softmax
// writes P_t, O_t += P_t V_s (TS MMA, P from TMEM, V MN-major).  An issuer
// issues PV_t(s-1) immediately before S_t(s) (which overwrites P_t), so the
// tensor pipe works on one tile while the other tile's softmax runs.
// Online softmax in base 2 with a lazy rescale: the running max is only
// moved (and O_t rescaled in TMEM) when a tile's max exceeds it by more than
// kRescaleLog2, so P stays <= 2^kRescaleLog2 and the final normalisation by
// the same stale max is exact.
//
// 3D neighbourhood attention (modes kModeNA*) runs on the same loop: a query
// tile is a brick of 128 tokens (bt x by x bx) of the (T, Y, X) volume, loaded
// by a 5-D TMA box straight from the raster layout; a paired CTA's two bricks
// are neighbours along one axis.  The key tiles are boxes of the same shape
// laid on a grid that starts at the corner of the union of the bricks' windows;
// every role walks that grid in the same order, and each query row masks the
// keys outside its own window.
#pragma once
#include <float.h>
#include <limits.h>
#include "ptx.cuh"

namespace vdtb {

enum FwdMode {
  kModeDense = 0,
  kModeSparse = 1,
  kModeSplit = 2,
  kModeSparseFused = 3,
  // 3D neighbourhood attention; the suffix is the brick (frames x rows x columns)
  kModeNA1x8x16 = 4,
  kModeNA2x8x8 = 5,
  kModeNA4x4x8 = 6,
};

__host__ __device__ constexpr bool is_na_mode(int m) { return m >= kModeNA1x8x16 && m <= kModeNA4x4x8; }
__host__ __device__ constexpr int na_brick_t(int m) { return m == kModeNA4x4x8 ? 4 : (m == kModeNA2x8x8 ? 2 : 1); }
__host__ __device__ constexpr int na_brick_y(int m) { return m == kModeNA4x4x8 ? 4 : 8; }
__host__ __device__ constexpr int na_brick_x(int m) { return m == kModeNA1x8x16 ? 16 : 8; }
// Key boxes of the persistent neighbourhood kernel: kNAKeysBrick takes the
// brick's own shape, kNAKeysWide 4 x 2 x 16 (which covers the window union of a
// 4 x 4 x 8 brick under small windows with fewer boxes); kNAKeysWideF8 the same
// boxes with the window operand in E5M2 instead of bf16 (half the bytes, so two
// window buffers per tile fit at d = 128; exact for a narrower score range).
constexpr int kNAKeysBrick = 0, kNAKeysWide = 1, kNAKeysWideF8 = 2;
__host__ __device__ constexpr int na_keys_t(int m, int keys) { return keys != kNAKeysBrick ? 4 : na_brick_t(m); }
__host__ __device__ constexpr int na_keys_y(int m, int keys) { return keys != kNAKeysBrick ? 2 : na_brick_y(m); }
__host__ __device__ constexpr int na_keys_x(int m, int keys) { return keys != kNAKeysBrick ? 16 : na_brick_x(m); }
// How a key tile's scores mark keys outside the row's window: not at all (the
// caller masks them), or by a bias the tensor core added (NABiasLayout): -2^120
// per missed coordinate with a bf16 window operand, -57344^2 = -49 * 2^26 with an
// E5M2 one.  kWinMaskBelow: a tile maximum below it means no key of the tile is
// in the window (with |raw score| < 2^96, resp. 2^30, every biased score lies
// below it and every other above).
constexpr int kWinNone = 0, kWinBf16 = 1, kWinF8 = 2;
__host__ __device__ constexpr float win_mask_below(int win) { return win == kWinF8 ? -0x1p31f : -0x1p119f; }

constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// largest chunk count the split-KV kernel merges in its tail
constexpr int kMergeMaxSplit = 32;

struct FwdParams {
  int BH;             // B * H
  int Sq, Skv;        // query rows, key rows (per head)
  int n_qg;           // CTA query groups per head = ceil(Sq / (128 * NQT))
  float scale_log2;   // softmax scale * log2(e)
  uint16_t* out;      // dense/sparse: [BH][Sq][D] bf16
  float* lse;         // dense/sparse: [BH][Sq] (nullable)
  float* out_part;    // split: [n_split][BH][Sq][D]
  float* lse_part;    // split: [n_split][BH][Sq]
  int n_split;
  const int32_t* sel_idx;  // sparse: [BH][NQB][NKB]
  const int32_t* sel_cnt;  // sparse: [BH][NQB]
  const float* stats;      // sparse: [BH][NQB][4] = mu, sigma, tau, W
  const float* taylor_t;   // sparse: [BH][NQB][D]
  // sparse with 128-row blocks, nullable: [BH][NQB], per head a permutation of
  // the query blocks; the two tiles of CTA qg take blocks qb_order[2qg] and
  // qb_order[2qg + 1] (null: blocks 2qg and 2qg + 1)
  const int32_t* qb_order;
  int NQB, NKB;
  int* status;             // device status words (status bits, id of the last launch that timed out)
  unsigned launch_id;      // this launch (never 0)
  // fused routing (kModeSparseFused): pooled inputs, routing constants and
  // optional copies of the routing the kernel computed on chip
  const float* qbar;       // [BH][NQB][D]
  const float* kbar;       // [BH][NKB][D]
  const float* vbar;       // [BH][NKB][D]
  float scale;             // softmax scale (natural units)
  float beta;
  int block_k;
  int32_t* out_sel_idx;    // nullable, [BH][NQB][NKB]
  int32_t* out_sel_cnt;    // nullable, [BH][NQB]
  float* out_stats;        // nullable, [BH][NQB][4]
  float* out_taylor;       // nullable, [BH][NQB][D]
  // 3D neighbourhood attention: volume (T, Y, X), window (Kt, Ky, Kx), query
  // bricks per axis, CTA grid per axis (the pair axis holds ceil(nq / 2))
  int na_L[3];
  int na_K[3];
  int na_nq[3];
  int na_np[3];
  int na_pair_axis;        // 0 = frames, 1 = rows, 2 = columns, 3 = one brick per CTA
  // split-KV with the merge in the tail (nullable): one arrival counter per
  // (head, query tile), zero between calls; the last chunk's CTA merges the
  // partials of its rows into out (bf16) and lse
  int* merge_count;
};

// Window start along one axis: centred on p, moved inward at the borders
// (1 <= K <= L).
__device__ __forceinline__ int na_window_start(int p, int K, int L) {
  int s = p - K / 2;
  s = s < 0 ? 0 : s;
  return s > L - K ? L - K : s;
}

// The key boxes of one neighbourhood-attention CTA, in the order every role
// visits them.  Box u has origin cu + (ut, uy, ux) * brick (x fastest); bit t
// of its flags is set when it overlaps query tile t's window union.
template <int BT, int BY, int BX>
struct NAWalk {
  int org[2][3];   // query brick origins
  int lo[2][3];    // per tile: union of its rows' windows, [lo, hi) per axis
  int hi[2][3];
  int cu[3];       // origin of the box grid
  int nk[3];       // boxes per axis
  int ntiles;
  int u, nb;

  // paired: the CTA owns two bricks that are neighbours along p.na_pair_axis
  // (the CTA grid holds pairs on that axis); otherwise one brick per CTA.
  __device__ __forceinline__ void init(const FwdParams& p, int qg, bool paired) {
    const int B[3] = {BT, BY, BX};
    int idx[3];
    idx[2] = qg % p.na_np[2];
    const int r = qg / p.na_np[2];
    idx[1] = r % p.na_np[1];
    idx[0] = r / p.na_np[1];
    ntiles = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      int ib[3];
#pragma unroll
      for (int a = 0; a < 3; ++a) ib[a] = (paired && a == p.na_pair_axis) ? 2 * idx[a] + t : idx[a];
      const int pa = p.na_pair_axis;
      const bool valid = paired ? (pa == 0 ? ib[0] : pa == 1 ? ib[1] : ib[2]) <
                                      (pa == 0 ? p.na_nq[0] : pa == 1 ? p.na_nq[1] : p.na_nq[2])
                                : t == 0;
      if (valid) ntiles = t + 1;
#pragma unroll
      for (int a = 0; a < 3; ++a) {
        org[t][a] = ib[a] * B[a];
        const int last = min(org[t][a] + B[a], p.na_L[a]) - 1;
        lo[t][a] = na_window_start(min(org[t][a], p.na_L[a] - 1), p.na_K[a], p.na_L[a]);
        hi[t][a] = na_window_start(last, p.na_K[a], p.na_L[a]) + p.na_K[a];
        if (!valid) {   // an absent second tile adds nothing to the union
          lo[t][a] = lo[0][a];
          hi[t][a] = hi[0][a];
        }
      }
    }
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      cu[a] = min(lo[0][a], lo[1][a]);
      nk[a] = (max(hi[0][a], hi[1][a]) - cu[a] + B[a] - 1) / B[a];
    }
    nb = nk[0] * nk[1] * nk[2];
    u = 0;
  }
  // Next box overlapping at least one tile: its index, origin and flags; -1 at the end.
  __device__ __forceinline__ int next(uint32_t& flags, int (&box)[3]) {
    const int B[3] = {BT, BY, BX};
    while (u < nb) {
      const int uu = u++;
      const int ux = uu % nk[2];
      const int r = uu / nk[2];
      box[2] = cu[2] + ux * BX;
      box[1] = cu[1] + (r % nk[1]) * BY;
      box[0] = cu[0] + (r / nk[1]) * BT;
      flags = 0;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        bool ov = t < ntiles;
#pragma unroll
        for (int a = 0; a < 3; ++a) ov = ov && box[a] < hi[t][a] && box[a] + B[a] > lo[t][a];
        if (ov) flags |= 1u << t;
      }
      if (flags) return uu;
    }
    return -1;
  }
};

// Walks the ascending union of up to NL tile lists (one per query block the
// CTA owns; NL is fixed at compile time so that a one-list CTA carries one
// list's state).  Each step yields the kv tile index and a bit per list that
// contains it.  Dense/split lists are implicit ranges [0, n).
template <int NL>
struct TileMerge {
  const int32_t* ptr[NL];
  const uint16_t* sptr[NL];   // lists in shared memory (fused routing)
  bool smem_lists;
  int n[NL];
  int pos[NL];
  int nlists;
  int limit;      // valid tile indices are [0, limit)
  bool implicit;
  int* status;

  __device__ __forceinline__ int head(int l) const {
    if (implicit) return pos[l];
    if (smem_lists) return sptr[l][pos[l]];
    int v = __ldg(ptr[l] + pos[l]);
    if ((unsigned)v >= (unsigned)limit) {
      atomicOr(status, ATTN_DEVICE_BAD_LIST);
      v = v < 0 ? 0 : limit - 1;
    }
    return v;
  }
  // Returns the next tile index, or -1 when every list is exhausted.
  __device__ __forceinline__ int next(uint32_t& flags) {
    int u = INT_MAX;
    int h[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      h[l] = INT_MAX;
      if (l < nlists && pos[l] < n[l]) h[l] = head(l);
      u = min(u, h[l]);
    }
    if (u == INT_MAX) return -1;
    flags = 0;
#pragma unroll
    for (int l = 0; l < NL; ++l)
      if (h[l] == u) {
        flags |= 1u << l;
        ++pos[l];
      }
    return u;
  }
};

template <int D, int BK, int MODE, int NQT, int NSTAGE>
struct FwdCfg {
  static constexpr bool kSparseLike = MODE == kModeSparse || MODE == kModeSparseFused;
  static constexpr bool kFused = MODE == kModeSparseFused;
  static constexpr bool kNA = is_na_mode(MODE);
  // two independent query tiles per CTA (dense / sparse with NQT = 2): each
  // tile has its own list walk, its own two K/V slots, its own TMA producer
  // warp and its own MMA-issuing warp, like two one-tile CTAs; the two issuers
  // take a shared-memory lock around each step's MMA batch (PV of the previous
  // key tile, S of the current one).  Per tile and step one barrier pair:
  // K of key tile g and V of key tile g-1 land together on the tile's full
  // barrier, and one commit after the batch frees both slots.
  static constexpr bool kDual = NQT == 2 && (MODE == kModeDense || MODE == kModeSparse);
  // per-tile roles (the two-issuer CTA and the one-tile split-KV / dense / sparse CTAs): tile t
  // has its own producer and issuer warps and K/V slots 2t, 2t+1 with one full barrier per step.
  // The neighbourhood CTAs and the shared-walk two-tile CTA (fused routing) keep one producer
  // and one issuer with a barrier per slot (for the one-brick neighbourhood CTA the per-tile
  // roles measured no faster: its control warps spill the walk's box state).
  static constexpr bool kPerTile = kDual || (NQT == 1 && !kNA);
  static constexpr int kNaT = na_brick_t(MODE), kNaY = na_brick_y(MODE), kNaX = na_brick_x(MODE);
  static constexpr int QB = kSparseLike ? 128 / BK : 1;   // query blocks per 128-row tile
  // fused routing: query blocks per CTA, key-block capacity, staging chunk
  static constexpr int kFusedR = NQT * QB;
  static constexpr int kFusedMaxNKB = 1024;
  static constexpr int kFusedCH = 128;
  static constexpr int kFusedPersistBytes =
      kFused ? ((kFusedR * kFusedMaxNKB * 2 + kFusedR * D * 4 + kFusedR * 16 + 15) / 16) * 16 : 0;
  // NQT softmax warpgroups + one control warpgroup (TMA producer warp, MMA
  // warp, two idle warps): whole warpgroups so that setmaxnreg can move
  // registers from the control warpgroup to the softmax warpgroups.
  static constexpr int kThreads = NQT * 128 + 128;
  static constexpr int kProducerWarp = NQT * 4;
  static constexpr int kMmaWarp = NQT * 4 + 1;
  // (two independent tiles: tile t's producer is warp kProducerWarp + 2t, its MMA issuer the next warp)
  // Registers per thread: at launch (65536 / (threads * CTAs per SM), rounded
  // down to 8), for the control warpgroup after setmaxnreg.dec, and for the
  // softmax warpgroups after setmaxnreg.inc.  The split must add up to the
  // launch allocation: NQT*128*kRegsSoftmax + 128*kRegsControl <= kThreads*kRegsLaunch.
  static constexpr int kRegsLaunch = NQT == 2 ? 168 : 128;
  // (one-tile CTA: 208 / 48 leaves the dense, split and neighbourhood softmax
  // without spills; the sparse walk measured faster with 200 / 56)
  static constexpr int kRegsControl = NQT == 2 ? 64 : (kSparseLike ? 56 : 48);
  static constexpr int kRegsSoftmax = NQT == 2 ? 216 : (kSparseLike ? 200 : 208);
  static_assert(NQT * 128 * kRegsSoftmax + 128 * kRegsControl <= kThreads * kRegsLaunch, "register split");
  static constexpr int kQTileBytes = 128 * D * 2;
  static constexpr int kSlotBytes = BK * D * 2;
  // A two-tile CTA takes all 512 TMEM columns: its shared-memory request is
  // padded past half of the SM's 228 KB so that two such CTAs never share an
  // SM (the second would stall in tcgen05.alloc until the first exits).
  static constexpr int kSmemRaw = 1024 + NQT * kQTileBytes + NSTAGE * kSlotBytes + kFusedPersistBytes;
  static constexpr int kSmemBytes = (NQT == 2 && kSmemRaw < 120 * 1024) ? 120 * 1024 : kSmemRaw;
  static constexpr uint32_t kTmemCols = NQT == 2 ? 512 : 256;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, BK, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BK == 64 || BK == 128, "kv tile");
  static_assert(NQT == 1 || NQT == 2, "query tiles per CTA");
  static_assert(NQT * QB <= 4, "lists per CTA");
  static_assert(NSTAGE >= 2, "ring depth");
  static_assert(!kDual || NSTAGE == 4, "two K/V slots per tile");
  static_assert(!kPerTile || NSTAGE >= 2 * NQT, "two K/V slots per tile");
  static_assert(!kFused || kFusedCH * D * 4 + kFusedR * kFusedMaxNKB * 4 + kFusedR * D * 4 <= NSTAGE * kSlotBytes,
                "fused routing scratch must fit in the K/V ring");
  static_assert(!kFused || NQT == 2, "fused routing runs on the two-tile CTA");
  static_assert(!kNA || (BK == 128 && kNaT * kNaY * kNaX == 128), "neighbourhood bricks");
  static_assert(MODE != kModeSplit || NQT == 1, "split-KV CTAs take one query tile (the merge tail assumes it)");
  static_assert(MODE != kModeSplit || 128 * (kMergeMaxSplit + 1) * 4 <= NSTAGE * kSlotBytes,
                "the merge weights live in the idle K/V ring");
};

// Next key tile of a CTA's walk: neighbourhood boxes or the merged lists.
template <bool NA, class Walk, class Merge>
__device__ __forceinline__ int next_tile(Walk& naw, Merge& merge, uint32_t& flags, int (&box)[3]) {
  if constexpr (NA) {
    return naw.next(flags, box);
  } else {
    return merge.next(flags);
  }
}

// The lists of query tile `qtile` (independent tiles): the selected lists of
// its QB query blocks (sparse), or the implicit range of all key tiles (dense;
// empty for a tile past the end of the sequence).
template <int QB, bool SPARSE>
__device__ __forceinline__ void tile_walk_init(TileMerge<QB>& w, const FwdParams& p, int bh, int qtile, bool valid,
                                               int n_kv_tiles) {
  w.status = p.status;
  w.smem_lists = false;
#pragma unroll
  for (int l = 0; l < QB; ++l) {
    w.sptr[l] = nullptr;
    w.pos[l] = 0;
    w.n[l] = 0;
    w.ptr[l] = p.sel_idx;
  }
  if constexpr (SPARSE) {
    w.implicit = false;
    w.nlists = QB;
    w.limit = p.NKB;
#pragma unroll
    for (int l = 0; l < QB; ++l) {
      const long long i = (long long)qtile * QB + l;
      if (valid && i < p.NQB) {
        const long long row = (long long)bh * p.NQB + i;
        const int c = __ldg(p.sel_cnt + row);
        w.n[l] = c < 0 ? 0 : (c > p.NKB ? p.NKB : c);
        w.ptr[l] = p.sel_idx + row * p.NKB;
      }
    }
  } else {
    w.implicit = true;
    w.nlists = 1;
    w.limit = n_kv_tiles;
    w.n[0] = valid ? n_kv_tiles : 0;
  }
}

// Next key tile of a per-tile role: its own tile's walk (two-issuer CTA) or the CTA's walk.
template <bool DUAL, bool NA, class Own, class Walk, class Merge>
__device__ __forceinline__ int next_step(Own& own, Walk& naw, Merge& merge, uint32_t& flags, int (&box)[3]) {
  if constexpr (DUAL) {
    return own.next(flags);
  } else {
    return next_tile<NA>(naw, merge, flags, box);
  }
}

// Spin lock in shared memory with a time limit: on timeout the caller goes on
// without it (the lock only orders MMA issue between the CTA's two tiles; no
// result depends on it).
__device__ __forceinline__ bool issue_lock(int* lock, volatile int* abort_flag) {
  if (atomicCAS(lock, 0, 1) == 0) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (atomicCAS(lock, 0, 1) == 0) return true;
    if (*abort_flag || global_timer_ns() - t0 > 1000000ull) return false;
  }
}
__device__ __forceinline__ void issue_unlock(int* lock) { atomicExch(lock, 0); }

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 3D neighbourhood attention: the scores of one query row against a key box
// (origin `box`, shape BT x BY x BX, x fastest) keep the keys inside the row's
// window (start `ws`, extent K per axis) and become -inf elsewhere.
template <int BT, int BY, int BX, int BK>
__device__ __forceinline__ void na_mask_scores(float (&x)[BK], const int (&ws)[3], const int (&box)[3],
                                               const int (&K)[3]) {
  int lo[3], hi[3];
  const int Bd[3] = {BT, BY, BX};
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    lo[a] = min(max(ws[a] - box[a], 0), Bd[a]);
    hi[a] = min(max(ws[a] + K[a] - box[a], 0), Bd[a]);
  }
  const bool full = lo[0] == 0 && hi[0] == BT && lo[1] == 0 && hi[1] == BY && lo[2] == 0 && hi[2] == BX;
  if (full) return;
  const bool any = lo[0] < hi[0] && lo[1] < hi[1] && lo[2] < hi[2];
  const uint32_t xm = any ? (((1u << hi[2]) - 1u) & ~((1u << lo[2]) - 1u)) : 0u;
  const uint32_t ym = ((1u << hi[1]) - 1u) & ~((1u << lo[1]) - 1u);
  uint32_t lm = 0;   // bit (frame * BY + row) of the box: that line is in the window
#pragma unroll
  for (int ct = 0; ct < BT; ++ct)
    if (ct >= lo[0] && ct < hi[0]) lm |= ym << (ct * BY);
  constexpr int LPW = 32 / BX;   // lines per 32-column word
#pragma unroll
  for (int w = 0; w < BK / 32; ++w) {
    uint32_t wd = 0;
#pragma unroll
    for (int j = 0; j < LPW; ++j)
      if ((lm >> (w * LPW + j)) & 1u) wd |= xm << (j * BX);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (!((wd >> j) & 1u)) x[w * 32 + j] = -INFINITY;
  }
}

// One online-softmax step of the query row a thread owns (TMEM lane), on its
// raw scores x of one key tile: moves the running max (lazily, see
// kRescaleLog2) and rescales O in TMEM at tO when `o_live` (O holds earlier
// steps), then writes P = 2^(x scale_log2 - m) as bf16 pairs over the first
// BK/2 columns of S at tS and adds its row sum to l_run.  Returns after the
// TMEM stores have completed; the caller fences and signals P ready.
//
// kWin (kWinBf16, kWinF8): keys outside the row's window carry a large
// negative bias instead of -inf (the window added by the tensor core, see
// NABiasLayout); a maximum below win_mask_below(kWin) means no key of the tile
// is in the window and counts as -inf, so such a tile moves nothing, as a tile
// of -inf scores would.
template <int BK, int D, int kWin = kWinNone>
__device__ __forceinline__ void softmax_step(float (&x)[BK], float scale_log2, float& m_run, float& l_run, bool o_live,
                                             uint32_t tS, uint32_t tO) {
  // row max: two chains of three-input maxima (max is exact, so the order is free)
  float mx0 = fmaxf(x[0], x[1]), mx1 = fmaxf(x[2], x[3]);
#pragma unroll
  for (int c = 4; c < BK; c += 4) {
    mx0 = fmax3(mx0, x[c], x[c + 1]);
    mx1 = fmax3(mx1, x[c + 2], x[c + 3]);
  }
  float raw = fmaxf(mx0, mx1);
  if constexpr (kWin != kWinNone) raw = raw < win_mask_below(kWin) ? -INFINITY : raw;
  const float mt = raw * scale_log2;
  // lazy rescale of the running max
  float alpha = 1.f;
  bool need = mt > m_run + kRescaleLog2 || (m_run == -INFINITY && mt > -INFINITY);
  if (need) {
    alpha = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - mt);
    l_run *= alpha;
    m_run = mt;
  }
  if (__any_sync(0xffffffffu, need && alpha != 0.f && o_live)) {
    // O holds the sum over earlier steps; rescale it in TMEM.  No wait is
    // needed: the issuer committed the barrier of this step's S after issuing
    // the previous PV of this tile, and a commit tracks every earlier MMA of
    // the issuing thread, so that PV has completed as well.
    const float a = (need && o_live) ? alpha : 1.f;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t rr[32];
      tmem_ld32(tO + c0, rr);
      tmem_ld_wait();
      tmem_reg_fence(rr);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float2 v = __fmul2_rn(make_float2(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1])),
                                    make_float2(a, a));
        rr[j] = __float_as_uint(v.x);
        rr[j + 1] = __float_as_uint(v.y);
      }
      tmem_st32(tO + c0, rr);
    }
  }
  const float nbase = (m_run == -INFINITY) ? 0.f : -m_run;
  // pairs of columns through the packed fp32 pipe: the same fused multiply-add
  // and the same two (even / odd) row-sum chains as scalar code, half the instructions
  const float2 sc2 = make_float2(scale_log2, scale_log2), nb2 = make_float2(nbase, nbase);
  float2 ls = make_float2(0.f, 0.f);
#pragma unroll
  for (int c0 = 0; c0 < BK; c0 += 64) {
    uint32_t pk[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float2 arg = __ffma2_rn(make_float2(x[c0 + 2 * j], x[c0 + 2 * j + 1]), sc2, nb2);
      const float p0 = ex2_approx(arg.x);
      const float p1 = ex2_approx(arg.y);
      ls = __fadd2_rn(ls, make_float2(p0, p1));
      pk[j] = pack_bf16x2(p0, p1);
    }
    tmem_st32(tS + c0 / 2, pk);
  }
  l_run += ls.x + ls.y;
  tmem_st_wait();
}

// softmax_step reading its scores from TMEM twice instead of holding all BK
// of them in registers: pass 1 takes the row maximum 64 columns at a time,
// pass 2 reloads each 64 columns, exponentiates them and writes their P (which
// lands on columns pass 2 has already read).  The same maxima, the same
// fused multiply-adds in the same order and the same row-sum chains as
// softmax_step, so the same bits, with 64 score registers live instead of BK.
// `between()` runs while the first loads are in flight.
template <int BK, int D, int kWin, class Between>
__device__ __forceinline__ void softmax_step_tmem(uint32_t tS, float scale_log2, float& m_run, float& l_run,
                                                  bool o_live, uint32_t tO, Between&& between) {
  static_assert(BK % 64 == 0, "key tile");
  // pass 1: the row max, in softmax_step's two chains of three-input maxima
  float mx0 = 0.f, mx1 = 0.f;
#pragma unroll
  for (int c0 = 0; c0 < BK; c0 += 64) {
    uint32_t ra[32], rb[32];
    tmem_ld32(tS + c0, ra);
    tmem_ld32(tS + c0 + 32, rb);
    if (c0 == 0) between();
    tmem_ld_wait();
    tmem_reg_fence(ra);
    tmem_reg_fence(rb);
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      const uint32_t* r = c < 32 ? ra : rb;
      const int e = c & 31;
      const float x0 = __uint_as_float(r[e]), x1 = __uint_as_float(r[e + 1]);
      const float x2 = __uint_as_float(r[e + 2]), x3 = __uint_as_float(r[e + 3]);
      if (c0 == 0 && c == 0) {
        mx0 = fmaxf(x0, x1);
        mx1 = fmaxf(x2, x3);
      } else {
        mx0 = fmax3(mx0, x0, x1);
        mx1 = fmax3(mx1, x2, x3);
      }
    }
  }
  float raw = fmaxf(mx0, mx1);
  if constexpr (kWin != kWinNone) raw = raw < win_mask_below(kWin) ? -INFINITY : raw;
  const float mt = raw * scale_log2;
  float alpha = 1.f;
  bool need = mt > m_run + kRescaleLog2 || (m_run == -INFINITY && mt > -INFINITY);
  if (need) {
    alpha = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - mt);
    l_run *= alpha;
    m_run = mt;
  }
  if (__any_sync(0xffffffffu, need && alpha != 0.f && o_live)) {
    const float a = (need && o_live) ? alpha : 1.f;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t rr[32];
      tmem_ld32(tO + c0, rr);
      tmem_ld_wait();
      tmem_reg_fence(rr);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float2 v = __fmul2_rn(make_float2(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1])),
                                    make_float2(a, a));
        rr[j] = __float_as_uint(v.x);
        rr[j + 1] = __float_as_uint(v.y);
      }
      tmem_st32(tO + c0, rr);
    }
  }
  // pass 2: P = 2^(x scale_log2 - m), 64 columns at a time, as in softmax_step
  const float nbase = (m_run == -INFINITY) ? 0.f : -m_run;
  const float2 sc2 = make_float2(scale_log2, scale_log2), nb2 = make_float2(nbase, nbase);
  float2 ls = make_float2(0.f, 0.f);
#pragma unroll
  for (int c0 = 0; c0 < BK; c0 += 64) {
    uint32_t ra[32], rb[32];
    tmem_ld32(tS + c0, ra);
    tmem_ld32(tS + c0 + 32, rb);
    tmem_ld_wait();
    tmem_reg_fence(ra);
    tmem_reg_fence(rb);
    uint32_t pk[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t* r = j < 16 ? ra : rb;
      const int e = (2 * j) & 31;
      const float2 arg = __ffma2_rn(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), sc2, nb2);
      const float p0 = ex2_approx(arg.x);
      const float p1 = ex2_approx(arg.y);
      ls = __fadd2_rn(ls, make_float2(p0, p1));
      pk[j] = pack_bf16x2(p0, p1);
    }
    tmem_st32(tS + c0 / 2, pk);
  }
  l_run += ls.x + ls.y;
  tmem_st_wait();
}

// Epilogue of the query row a thread owns: (O + f T) * inv from TMEM at tO
// (zero when !have_o; T optional) as bf16 into dst[0, D), element offset `off`
// of an output of `total` elements (bounds-checked in the debug build).
template <int D>
__device__ __forceinline__ void store_row_bf16(uint32_t tO, bool have_o, float inv, float f, const float* tt,
                                               bool row_valid, uint16_t* dst, [[maybe_unused]] long long off,
                                               [[maybe_unused]] long long total, [[maybe_unused]] int* status) {
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t rr[32];
    if (have_o) {
      tmem_ld32(tO + c0, rr);
      tmem_ld_wait();
      tmem_reg_fence(rr);
    }
    if (row_valid) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        uint4 pk;
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float val = have_o ? __uint_as_float(rr[j + e]) : 0.f;
          if (tt != nullptr) val = fmaf(f, tt[c0 + j + e], val);
          o[e] = val * inv;
        }
        pk.x = pack_bf16x2(o[0], o[1]);
        pk.y = pack_bf16x2(o[2], o[3]);
        pk.z = pack_bf16x2(o[4], o[5]);
        pk.w = pack_bf16x2(o[6], o[7]);
        if (ATTN_CHECKED(off + c0 + j, 8, total, status)) *reinterpret_cast<uint4*>(dst + c0 + j) = pk;
      }
    }
  }
}

// Split-KV tail with the merge fused in (one-tile CTA, run by its 128 softmax
// threads after they stored this chunk's partials): the partials are made
// visible device-wide, the (head, query tile) counter counts this chunk, and
// the CTA of the last chunk to arrive merges every chunk's partials of its
// 128 rows exactly (L = log sum exp lse_c, o = sum exp(lse_c - L) o_c, the
// arithmetic of lse_merge_kernel, so the result is bit-identical to the
// two-launch path) and resets the counter for the next call.  Partials written
// by other CTAs of this launch are read through L2.  To keep the merge off the
// latency path, thread r first loads row r's n lse values at once and leaves
// the weights exp(lse_c - L) in shared memory (`wbuf`, n <= kMergeMaxSplit);
// then each warp merges four rows at a time with all their chunk loads in
// flight.
template <int D>
__device__ __forceinline__ void split_merge_tail(const FwdParams& p, int bh, int qg, int q_row0, int r,
                                                 int& merge_last, volatile int& abort_flag, float* wbuf) {
  __threadfence();
  named_sync(2, 128);
  if (r == 0) {
    int last = 0;
    if (!abort_flag) {   // an aborted CTA (device timeout, reported in the status word) does not count
      int* cnt = p.merge_count + ((long long)bh * p.n_qg + qg);
      const int old = atomicAdd(cnt, 1);
      last = old == p.n_split - 1;
      if (last) atomicExch(cnt, 0);
    }
    merge_last = last;
  }
  named_sync(2, 128);
  if (!merge_last) return;
  __threadfence();
  const int n = p.n_split;
  const long long rows = (long long)p.BH * p.Sq;
  constexpr int WS = kMergeMaxSplit + 1;   // wbuf row: n weights, then L
  // ---- weights of row r
  {
    const int grow = q_row0 + r;
    float ls[kMergeMaxSplit];
    float M = -INFINITY;
    if (grow < p.Sq) {
      const long long row = (long long)bh * p.Sq + grow;
#pragma unroll
      for (int c = 0; c < kMergeMaxSplit; ++c) ls[c] = c < n ? __ldcg(p.lse_part + (long long)c * rows + row) : -INFINITY;
#pragma unroll
      for (int c = 0; c < kMergeMaxSplit; ++c)
        if (c < n) M = fmaxf(M, ls[c]);
    }
    float L = -INFINITY;
    if (M != -INFINITY) {
      float ssum = 0.f;
#pragma unroll
      for (int c = 0; c < kMergeMaxSplit; ++c)
        if (c < n) ssum += expf(ls[c] - M);
      L = M + logf(ssum);
#pragma unroll
      for (int c = 0; c < kMergeMaxSplit; ++c)
        if (c < n) wbuf[r * WS + c] = expf(ls[c] - L);
    }
    wbuf[r * WS + kMergeMaxSplit] = L;
    if (grow < p.Sq && p.lse != nullptr && ATTN_CHECKED((long long)bh * p.Sq + grow, 1, rows, p.status))
      p.lse[(long long)bh * p.Sq + grow] = L;
  }
  named_sync(2, 128);
  // ---- outputs: warp w merges rows w + 4 i, four at a time, lanes across d
  constexpr int PER = D / 32;
  constexpr int RB = 4;
  const int lane = r & 31, w = r >> 5;
  for (int i0 = w; i0 < 128; i0 += 4 * RB) {
    float o[RB][PER];
    bool live[RB];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      const int i = i0 + 4 * b;
      live[b] = i < 128 && q_row0 + i < p.Sq && wbuf[i * WS + kMergeMaxSplit] != -INFINITY;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[b][e] = 0.f;
    }
    int c = 0;
    for (; c + 1 < n; c += 2) {
      float a0[RB][PER], a1[RB][PER];
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        if (!live[b]) continue;
        const long long row = (long long)bh * p.Sq + q_row0 + i0 + 4 * b;
        const float* s0 = p.out_part + ((long long)c * rows + row) * D + lane * PER;
        const float* s1 = s0 + rows * D;
        if constexpr (PER == 4) {
          const float4 v0 = __ldcg(reinterpret_cast<const float4*>(s0));
          const float4 v1 = __ldcg(reinterpret_cast<const float4*>(s1));
          a0[b][0] = v0.x; a0[b][1] = v0.y; a0[b][2] = v0.z; a0[b][3] = v0.w;
          a1[b][0] = v1.x; a1[b][1] = v1.y; a1[b][2] = v1.z; a1[b][3] = v1.w;
        } else {
          const float2 v0 = __ldcg(reinterpret_cast<const float2*>(s0));
          const float2 v1 = __ldcg(reinterpret_cast<const float2*>(s1));
          a0[b][0] = v0.x; a0[b][1] = v0.y;
          a1[b][0] = v1.x; a1[b][1] = v1.y;
        }
      }
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        if (!live[b]) continue;
        const float* wr = wbuf + (i0 + 4 * b) * WS;
        const float w0 = wr[c], w1 = wr[c + 1];
#pragma unroll
        for (int e = 0; e < PER; ++e) o[b][e] = fmaf(w1, a1[b][e], fmaf(w0, a0[b][e], o[b][e]));
      }
    }
    if (c < n) {
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        if (!live[b]) continue;
        const long long row = (long long)bh * p.Sq + q_row0 + i0 + 4 * b;
        const float* s0 = p.out_part + ((long long)c * rows + row) * D + lane * PER;
        const float w0 = wbuf[(i0 + 4 * b) * WS + c];
#pragma unroll
        for (int e = 0; e < PER; ++e) o[b][e] = fmaf(w0, __ldcg(s0 + e), o[b][e]);
      }
    }
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      const int i = i0 + 4 * b;
      if (i >= 128 || q_row0 + i >= p.Sq) continue;
      const long long off = ((long long)bh * p.Sq + q_row0 + i) * D + lane * PER;
      if (!ATTN_CHECKED(off, PER, rows * D, p.status)) continue;
      uint16_t* dst = p.out + off;
      if constexpr (PER == 4) {
        uint2 pk;
        pk.x = pack_bf16x2(o[b][0], o[b][1]);
        pk.y = pack_bf16x2(o[b][2], o[b][3]);
        *reinterpret_cast<uint2*>(dst) = pk;
      } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[b][0], o[b][1]);
      }
    }
  }
}

// Sol-Attn routing of the CTA's R query blocks, computed on chip by the TH
// softmax threads before the main loop (no routing launch, no lists in
// memory).  Same definitions as route_kernel: proxy s_ij = scale Qbar_i.Kbar_j,
// mu/sigma over j (two-pass), tau = mu + beta sigma, selection s >= tau or the
// argmax (lowest j), ascending compaction with ballot/popc, Taylor weights
// w = n_j max(0, 1 + s - mu) of rejected blocks, W = sum w, T = sum w Vbar_j.
// chunk/prow/qs live in the (still idle) K/V ring; lists/cnts/mus/Ws/Ts persist.
template <int D, int R, int CH, int KMAX, int TH>
__device__ __forceinline__ void fused_route(const FwdParams& p, int bh, int qb0, int st, float* chunk, float* prow,
                                            float* qs, uint16_t* lists, int* cnts, float* mus, float* Ws, float* Ts) {
  const int NQB = p.NQB, NKB = p.NKB;
  const int w = st >> 5, lane = st & 31;
  for (int e = st; e < R * D; e += TH) {
    const int r = e / D, c = e % D, i = qb0 + r;
    qs[e] = (i < NQB) ? __ldg(p.qbar + ((long long)bh * NQB + i) * D + c) : 0.f;
  }
  // pass 1: proxy scores of every key block, staged through shared memory
  for (int j0 = 0; j0 < NKB; j0 += CH) {
    named_sync(1, TH);
    for (int e = st; e < CH * (D / 4); e += TH) {
      const int jj = e / (D / 4), c4 = e % (D / 4);
      float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j0 + jj < NKB) v4 = __ldg(reinterpret_cast<const float4*>(p.kbar + ((long long)bh * NKB + j0 + jj) * D) + c4);
      reinterpret_cast<float4*>(chunk)[e] = v4;
    }
    named_sync(1, TH);
    for (int e = st; e < R * CH; e += TH) {
      const int r = e / CH, jj = e % CH, j = j0 + jj;
      if (j >= NKB) continue;
      const float* krow = chunk + jj * D;
      const float* qrow = qs + r * D;
      float acc = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; ++c) {
        const int cc = (c + jj) & (D - 1);   // rotated column: conflict-free across the warp
        acc = fmaf(qrow[cc], krow[cc], acc);
      }
      prow[r * KMAX + j] = p.scale * acc;
    }
  }
  named_sync(1, TH);
  // statistics, selection and Taylor weights: warp w owns row w
  if (w < R) {
    float* row = prow + w * KMAX;
    float sum = 0.f, best = -INFINITY;
    int bidx = INT_MAX;
    for (int j = lane; j < NKB; j += 32) {
      const float v = row[j];
      sum += v;
      if (v > best) {
        best = v;
        bidx = j;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, off);
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, off);
      if (ob > best || (ob == best && oi < bidx)) {
        best = ob;
        bidx = oi;
      }
    }
    const float mu = sum / (float)NKB;
    float sq = 0.f;
    for (int j = lane; j < NKB; j += 32) {
      const float dv = row[j] - mu;
      sq = fmaf(dv, dv, sq);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
    const float sigma = sqrtf(sq / (float)NKB);
    const float tau = (p.beta == -INFINITY) ? -INFINITY : fmaf(p.beta, sigma, mu);
    int cnt = 0;
    float wsum = 0.f;
    for (int j0 = 0; j0 < NKB; j0 += 32) {
      const int j = j0 + lane;
      const bool in = j < NKB;
      const float v = in ? row[j] : 0.f;
      const bool keep = in && (v >= tau || j == bidx);
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      if (keep) lists[w * KMAX + cnt + __popc(m & ((1u << lane) - 1u))] = (uint16_t)j;
      cnt += __popc(m);
      float wt = 0.f;
      if (in && !keep) {
        const int nj = min(p.block_k, p.Skv - j * p.block_k);
        wt = (float)nj * fmaxf(0.f, 1.f + v - mu);
      }
      if (in) row[j] = wt;   // the proxy is no longer needed: keep the Taylor weight
      wsum += wt;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    const int i = qb0 + w;
    if (lane == 0) {
      cnts[w] = (i < NQB) ? cnt : 0;
      mus[w] = mu;
      Ws[w] = wsum;
    }
    if (i < NQB) {
      const long long rrow = (long long)bh * NQB + i;
      [[maybe_unused]] const long long nrows = (long long)p.BH * NQB;
      if (p.out_sel_cnt != nullptr && lane == 0 && ATTN_CHECKED(rrow, 1, nrows, p.status)) p.out_sel_cnt[rrow] = cnt;
      if (p.out_stats != nullptr && lane == 0 && ATTN_CHECKED(rrow * 4, 4, nrows * 4, p.status)) {
        p.out_stats[rrow * 4 + 0] = mu;
        p.out_stats[rrow * 4 + 1] = sigma;
        p.out_stats[rrow * 4 + 2] = tau;
        p.out_stats[rrow * 4 + 3] = wsum;
      }
      if (p.out_sel_idx != nullptr) {
        __syncwarp();
        for (int k = lane; k < cnt; k += 32)
          if (ATTN_CHECKED(rrow * NKB + k, 1, nrows * NKB, p.status)) p.out_sel_idx[rrow * NKB + k] = lists[w * KMAX + k];
      }
    }
  }
  // T = sum_j w_j Vbar_j, V staged through shared memory
  constexpr int PER = (R * D + TH - 1) / TH;
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  for (int j0 = 0; j0 < NKB; j0 += CH) {
    named_sync(1, TH);
    for (int e = st; e < CH * (D / 4); e += TH) {
      const int jj = e / (D / 4), c4 = e % (D / 4);
      float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j0 + jj < NKB) v4 = __ldg(reinterpret_cast<const float4*>(p.vbar + ((long long)bh * NKB + j0 + jj) * D) + c4);
      reinterpret_cast<float4*>(chunk)[e] = v4;
    }
    named_sync(1, TH);
    const int jn = min(CH, NKB - j0);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = st + k * TH;
      if (e < R * D) {
        const int r = e / D, c = e % D;
        const float* wrow = prow + r * KMAX + j0;
        float a = acc[k];
        for (int jj = 0; jj < jn; ++jj) a = fmaf(wrow[jj], chunk[jj * D + c], a);
        acc[k] = a;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int e = st + k * TH;
    if (e < R * D) {
      Ts[e] = acc[k];
      const int r = e / D, i = qb0 + r;
      if (p.out_taylor != nullptr && i < NQB &&
          ATTN_CHECKED(((long long)bh * NQB + i) * D + e % D, 1, (long long)p.BH * NQB * D, p.status))
        p.out_taylor[((long long)bh * NQB + i) * D + e % D] = acc[k];
    }
  }
  // the ring is handed over to TMA (async proxy) after these generic accesses
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  named_sync(1, TH);
}

// store_row_bf16 for an output whose rows start on 32-byte boundaries: each
// lane writes whole 32-byte sectors (256-bit stores), half the store
// instructions and sector writes of 16-byte stores, with two TMEM loads in
// flight.  Same arithmetic per element: (O + f T) * inv, T optional (16-byte
// aligned, in global or shared memory).
template <int D>
__device__ __forceinline__ void store_row_bf16_wide(uint32_t tO, float inv, float f, const float* tt, bool row_valid,
                                                    uint16_t* dst, [[maybe_unused]] long long off,
                                                    [[maybe_unused]] long long total, [[maybe_unused]] int* status) {
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 64) {
    uint32_t rr[2][32];
    tmem_ld32(tO + c0, rr[0]);
    tmem_ld32(tO + c0 + 32, rr[1]);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tmem_reg_fence(rr[h]);
      if (!row_valid) continue;
#pragma unroll
      for (int j = 0; j < 32; j += 16) {
        const int col = c0 + 32 * h + j;
        float o[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = __uint_as_float(rr[h][j + e]);
        if (tt != nullptr) {
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            // a generic load: T lives in global memory or (folded routing) in shared memory
            const float4 t4 = reinterpret_cast<const float4*>(tt + col)[e4];
            o[4 * e4 + 0] = fmaf(f, t4.x, o[4 * e4 + 0]);
            o[4 * e4 + 1] = fmaf(f, t4.y, o[4 * e4 + 1]);
            o[4 * e4 + 2] = fmaf(f, t4.z, o[4 * e4 + 2]);
            o[4 * e4 + 3] = fmaf(f, t4.w, o[4 * e4 + 3]);
          }
        }
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(o[2 * e] * inv, o[2 * e + 1] * inv);
        if (ATTN_CHECKED(off + col, 16, total, status))
          asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + col), "r"(pk[0]),
                       "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7])
                       : "memory");
      }
    }
  }
}

template <int D, int BK, int MODE, int NQT, int NSTAGE>
__global__ void __launch_bounds__(NQT * 128 + 128, (NQT == 1) ? 2 : 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Cfg = FwdCfg<D, BK, MODE, NQT, NSTAGE>;
  constexpr int QB = Cfg::QB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + NQT * Cfg::kQTileBytes;
  // fused routing: persistent lists and aggregates after the ring; the
  // prologue's scratch (chunk, proxy rows, pooled Q) lives in the idle ring
  constexpr int FR = Cfg::kFusedR, FKMAX = Cfg::kFusedMaxNKB;
  uint8_t* sFused = sKV + NSTAGE * Cfg::kSlotBytes;
  uint16_t* f_lists = reinterpret_cast<uint16_t*>(sFused);
  float* f_T = reinterpret_cast<float*>(sFused + FR * FKMAX * 2);
  int* f_cnt = reinterpret_cast<int*>(f_T + FR * D);
  float* f_mu = reinterpret_cast<float*>(f_cnt + FR);
  float* f_W = f_mu + FR;

  __shared__ uint64_t bar_q;
  __shared__ uint64_t bar_full[NSTAGE], bar_empty[NSTAGE];
  __shared__ uint64_t bar_s[NQT], bar_p[NQT], bar_o[NQT];
  __shared__ uint64_t bar_mma_done, bar_route;
  __shared__ uint64_t bar_qt[NQT], bar_done_t[NQT];   // independent tiles: Q landed, tile's MMAs done
  __shared__ int mma_lock;
  __shared__ uint32_t tmem_base_sh;
  __shared__ WaitState wstate;
  __shared__ int merge_last;
  __shared__ int skip_cta;   // the launch had already aborted when this CTA started
  WaitState* const wc = &wstate;
  volatile int& abort_flag = wstate.abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // ---- work item
  int linear = blockIdx.x;
  const int qg = linear % p.n_qg;
  linear /= p.n_qg;
  const int bh = linear % p.BH;
  const int chunk = (MODE == kModeSplit) ? linear / p.BH : 0;
  const int q_row0 = qg * NQT * 128;
  int kv_lo = 0, kv_hi = p.Skv;
  if (MODE == kModeSplit) {
    kv_lo = (int)(((long long)chunk * p.Skv) / p.n_split);
    kv_hi = (int)(((long long)(chunk + 1) * p.Skv) / p.n_split);
  }
  int n_valid_tiles = 0;
#pragma unroll
  for (int t = 0; t < NQT; ++t)
    if (q_row0 + t * 128 < p.Sq) n_valid_tiles = t + 1;
  // The query tile (of 128 rows) that tile t runs: its slot qg * NQT + t, or
  // the block a query-block order puts in that slot (independent sparse tiles
  // of 128-row blocks; an entry outside [0, NQB) is clamped and reported).
  auto tile_of = [&](int t) -> int {
    const int slot = qg * NQT + t;
    if constexpr (MODE == kModeSparse && NQT == 2 && QB == 1) {
      if (p.qb_order != nullptr && slot < p.NQB) {
        int v = __ldg(p.qb_order + (long long)bh * p.NQB + slot);
        if ((unsigned)v >= (unsigned)p.NQB) {
          atomicOr(p.status, ATTN_DEVICE_BAD_LIST);
          v = v < 0 ? 0 : p.NQB - 1;
        }
        return v;
      }
    }
    return slot;
  };
  constexpr bool kNA = Cfg::kNA;
  NAWalk<Cfg::kNaT, Cfg::kNaY, Cfg::kNaX> naw;
  int na_box[3] = {0, 0, 0};
  if constexpr (kNA) {
    naw.init(p, blockIdx.x % p.n_qg, NQT == 2);
    n_valid_tiles = naw.ntiles;
  }

  constexpr int kNL = Cfg::kSparseLike ? NQT * QB : NQT;   // lists this CTA walks at most
  TileMerge<kNL> merge;
  merge.status = p.status;
  merge.smem_lists = false;
#pragma unroll
  for (int l = 0; l < kNL; ++l) merge.sptr[l] = f_lists;
  if (MODE == kModeSparseFused) {
    // counts are filled in once the on-chip routing is done (route_ready)
    merge.implicit = false;
    merge.smem_lists = true;
    merge.nlists = FR;
    merge.limit = p.NKB;
#pragma unroll
    for (int l = 0; l < kNL; ++l) {
      merge.pos[l] = 0;
      merge.n[l] = 0;
      merge.ptr[l] = nullptr;
      merge.sptr[l] = f_lists + (l < FR ? l : 0) * FKMAX;
    }
  } else if (MODE == kModeSparse) {
    merge.implicit = false;
    merge.nlists = NQT * QB;
    merge.limit = p.NKB;
#pragma unroll
    for (int l = 0; l < kNL; ++l) {
      merge.pos[l] = 0;
      merge.n[l] = 0;
      merge.ptr[l] = p.sel_idx;
      if (l < NQT * QB) {
        long long i = (long long)(qg * NQT + l / QB) * QB + (l % QB);
        if (i < p.NQB) {
          long long row = (long long)bh * p.NQB + i;
          int c = __ldg(p.sel_cnt + row);
          merge.n[l] = c < 0 ? 0 : (c > p.NKB ? p.NKB : c);
          merge.ptr[l] = p.sel_idx + row * p.NKB;
        }
      }
    }
  } else {
    merge.implicit = true;
    merge.nlists = n_valid_tiles;
    int nt = (kv_hi - kv_lo + BK - 1) / BK;
    merge.limit = nt;
#pragma unroll
    for (int l = 0; l < kNL; ++l) {
      merge.pos[l] = 0;
      merge.n[l] = nt;
      merge.ptr[l] = nullptr;
    }
  }

  // ---- setup
  if (tid == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 128);
      mbar_init(&bar_o[t], 1);
    }
    mbar_init(&bar_mma_done, 1);
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&bar_qt[t], 1);
      mbar_init(&bar_done_t[t], 1);
    }
    mma_lock = 0;
    mbar_init(&bar_route, 1);
    skip_cta = wait_state_init(wstate, p.status, p.launch_id);
    fence_barrier_init();
  }
  if (warp == Cfg::kMmaWarp) tmem_alloc(&tmem_base_sh, Cfg::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (!skip_cta) {
  // fused routing: lists are ready once the softmax threads arrive on bar_route
  auto take_fused_lists = [&]() {
#pragma unroll
    for (int l = 0; l < kNL; ++l) merge.n[l] = (l < FR) ? f_cnt[l] : 0;
  };

  if (warp >= Cfg::kProducerWarp) {
    setmaxnreg_dec<Cfg::kRegsControl>();
  if constexpr (Cfg::kPerTile) {
    // warps kProducerWarp + {0, 1, 2, 3}: producer of tile 0, issuer of tile 0, producer of tile 1,
    // issuer of tile 1 (a one-tile CTA uses the first two)
    const int role = warp - Cfg::kProducerWarp;
    const int t = role >> 1;
    if (lane == 0 && t < NQT) {
      TileMerge<QB> w;
      const int qtile = tile_of(t);
      if constexpr (Cfg::kDual)
        tile_walk_init<QB, Cfg::kSparseLike>(w, p, bh, qtile, t < n_valid_tiles, (kv_hi - kv_lo + BK - 1) / BK);
      uint32_t fl;
      int u;
      if ((role & 1) == 0) {
        // ---- TMA producer of tile t: Q_t, then per step group the K and V tiles into slots 2t, 2t+1
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        const bool valid = t < n_valid_tiles;
        if (valid) {
          mbar_expect_tx(&bar_qt[t], Cfg::kQTileBytes);
          for (int h = 0; h < D / 64; ++h) {
            if constexpr (kNA)
              tma_load_5d(sQ + h * 16384, &tm_q, &bar_qt[t], h * 64, naw.org[0][2], naw.org[0][1], naw.org[0][0], bh);
            else
              tma_load_3d(sQ + t * Cfg::kQTileBytes + h * 16384, &tm_q, &bar_qt[t], h * 64, qtile * 128, bh);
          }
        }
        // group g: K of key tile g into slot 2t, V of key tile g-1 into slot 2t+1, both on
        // bar_full[2t]; the group is loaded once batch g-1 (PV of g-2, S of g-1) has completed
        const int kslot = 2 * t, vslot = 2 * t + 1;
        int g = 0, prev = -1;
        int pbox[3] = {0, 0, 0};
        bool ok = true;
        while (ok) {
          u = next_step<Cfg::kDual, kNA>(w, naw, merge, fl, na_box);
          if (u < 0 && prev < 0) break;
          if (g >= 1 && !bounded_wait(&bar_s[t], (g - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&bar_full[kslot], ((u >= 0) + (prev >= 0)) * Cfg::kSlotBytes);
          for (int h = 0; h < D / 64; ++h) {
            uint8_t* kd = sKV + kslot * Cfg::kSlotBytes + h * (BK * 128);
            uint8_t* vd = sKV + vslot * Cfg::kSlotBytes + h * (BK * 128);
            if constexpr (kNA) {
              if (u >= 0) tma_load_5d(kd, &tm_k, &bar_full[kslot], h * 64, na_box[2], na_box[1], na_box[0], bh);
              if (prev >= 0) tma_load_5d(vd, &tm_v, &bar_full[kslot], h * 64, pbox[2], pbox[1], pbox[0], bh);
            } else {
              if (u >= 0) tma_load_3d(kd, &tm_k, &bar_full[kslot], h * 64, kv_lo + u * BK, bh);
              if (prev >= 0) tma_load_3d(vd, &tm_v, &bar_full[kslot], h * 64, kv_lo + prev * BK, bh);
            }
          }
          prev = u;
#pragma unroll
          for (int a = 0; a < 3; ++a) pbox[a] = na_box[a];
          ++g;
          if (u < 0) break;
        }
        // drain: no copy may still be landing when the CTA exits
        if (valid) drain_wait(&bar_qt[t], 0, wc);
        if (g >= 1) drain_wait(&bar_full[kslot], (g - 1) & 1, wc);
      } else {
        // ---- MMA issuer of tile t: per group PV_t(g-1) then S_t(g) (two-issuer CTA: under the issue lock)
        bool ok = t < n_valid_tiles && bounded_wait(&bar_qt[t], 0, wc);
        tc_fence_after();
        const uint32_t q_addr = smem_u32(sQ) + t * Cfg::kQTileBytes;
        const uint32_t kv_base = smem_u32(sKV);
        const uint32_t s_tmem = tmem + t * 256, o_tmem = tmem + t * 256 + 128;
        const int kslot = 2 * t, vslot = 2 * t + 1;
        const uint32_t k_addr = kv_base + kslot * Cfg::kSlotBytes, v_addr = kv_base + vslot * Cfg::kSlotBytes;
        int g = 0, pvc = 0;
        bool pending = false;
        while (ok) {
          u = next_step<Cfg::kDual, kNA>(w, naw, merge, fl, na_box);
          if (u < 0 && !pending) break;
          if (!bounded_wait(&bar_full[kslot], g & 1, wc) ||
              (pending && !bounded_wait(&bar_p[t], pvc & 1, wc))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool locked = Cfg::kDual && issue_lock(&mma_lock, &abort_flag);
          if (pending) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              uint64_t bdesc = smem_desc_sw128(v_addr + kk * 16 * 128, BK * 128, 1024);
              mma_ts(o_tmem, s_tmem + kk * 8, bdesc, Cfg::kIdescPV, (pvc > 0 || kk > 0) ? 1u : 0u);
            }
            ++pvc;
          }
          if (u >= 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              uint64_t adesc = smem_desc_sw128(q_addr + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
              uint64_t bdesc = smem_desc_sw128(k_addr + (kk / 4) * (BK * 128) + (kk % 4) * 32, 16, 1024);
              mma_ss(s_tmem, adesc, bdesc, Cfg::kIdescS, kk > 0 ? 1u : 0u);
            }
          }
          if (locked) issue_unlock(&mma_lock);
          // one commit serves the softmax (S ready) and the producer (both slots free)
          mma_commit(&bar_s[t]);
          pending = u >= 0;
          ++g;
          if (u < 0) break;
        }
        // the epilogue waits for the last PV here; a commit tracks every earlier MMA of this thread
        mma_commit(&bar_o[t]);
        // every MMA this thread issued has completed before TMEM is released
        mma_commit(&bar_done_t[t]);
        drain_wait(&bar_done_t[t], 0, wc);
      }
    }
  } else
  if (warp == Cfg::kProducerWarp) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_expect_tx(&bar_q, n_valid_tiles * Cfg::kQTileBytes);
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        if (t >= n_valid_tiles) break;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          if constexpr (kNA)
            tma_load_5d(sQ + t * Cfg::kQTileBytes + h * 16384, &tm_q, &bar_q, h * 64, naw.org[t][2], naw.org[t][1],
                        naw.org[t][0], bh);
          else
            tma_load_3d(sQ + t * Cfg::kQTileBytes + h * 16384, &tm_q, &bar_q, h * 64, q_row0 + t * 128, bh);
        }
      }
      int ld = 0;
      uint32_t flags;
      int u;
      bool ok = true;
      if (MODE == kModeSparseFused) {
        ok = bounded_wait(&bar_route, 0, wc);   // the ring holds routing scratch until then
        take_fused_lists();
      }
      while (ok && (u = next_tile<kNA>(naw, merge, flags, na_box)) >= 0) {
        const int row = kv_lo + u * BK;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const int slot = ld % NSTAGE;
          if (ld >= NSTAGE && !bounded_wait(&bar_empty[slot], ((ld / NSTAGE) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          uint8_t* dst = sKV + slot * Cfg::kSlotBytes;
          mbar_expect_tx(&bar_full[slot], Cfg::kSlotBytes);
          for (int h = 0; h < D / 64; ++h) {
            if constexpr (kNA)
              tma_load_5d(dst + h * (BK * 128), kv == 0 ? &tm_k : &tm_v, &bar_full[slot], h * 64, na_box[2], na_box[1],
                          na_box[0], bh);
            else
              tma_load_3d(dst + h * (BK * 128), kv == 0 ? &tm_k : &tm_v, &bar_full[slot], h * 64, row, bh);
          }
          ++ld;
        }
      }
      // drain: make sure no copy is still landing when the CTA exits
      drain_wait(&bar_q, 0, wc);
      for (int j = (ld > NSTAGE ? ld - NSTAGE : 0); j < ld; ++j) drain_wait(&bar_full[j % NSTAGE], (j / NSTAGE) & 1, wc);
    }
  } else if (warp == Cfg::kMmaWarp) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      bool ok = bounded_wait(&bar_q, 0, wc);
      if (MODE == kModeSparseFused) {
        ok = ok && bounded_wait(&bar_route, 0, wc);
        take_fused_lists();
      }
      tc_fence_after();
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t kv_base = smem_u32(sKV);
      int ld = 0;
      bool pending[NQT];
      int pv_count[NQT];
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        pending[t] = false;
        pv_count[t] = 0;
      }
      int prev_vslot = -1, prev_vpar = 0;
      uint32_t flags;
      int u;
      auto issue_pv = [&](int t, int vslot) {
        const uint32_t v_addr = kv_base + vslot * Cfg::kSlotBytes;
        const uint32_t d_tmem = tmem + t * 256 + 128;
        const uint32_t p_tmem = tmem + t * 256;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          uint64_t bdesc = smem_desc_sw128(v_addr + kk * 16 * 128, BK * 128, 1024);
          mma_ts(d_tmem, p_tmem + kk * 8, bdesc, Cfg::kIdescPV, (pv_count[t] > 0 || kk > 0) ? 1u : 0u);
        }
        ++pv_count[t];
        pending[t] = false;
      };
      while (ok && (u = next_tile<kNA>(naw, merge, flags, na_box)) >= 0) {
        const int kslot = ld % NSTAGE;
        if (!bounded_wait(&bar_full[kslot], (ld / NSTAGE) & 1, wc)) break;
        ++ld;
        const int vslot = ld % NSTAGE;
        const int vpar = (ld / NSTAGE) & 1;
        ++ld;
        tc_fence_after();
        bool prev_v_ready = false, any_pv = false;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (pending[t]) {
            if (!prev_v_ready) {
              if (!bounded_wait(&bar_full[prev_vslot], prev_vpar, wc)) { ok = false; break; }
              prev_v_ready = true;
            }
            if (!bounded_wait(&bar_p[t], pv_count[t] & 1, wc)) { ok = false; break; }
            tc_fence_after();
            issue_pv(t, prev_vslot);
            any_pv = true;
          }
          if ((flags >> (t * QB)) & ((1u << QB) - 1u)) {
            const uint32_t k_addr = kv_base + kslot * Cfg::kSlotBytes;
            const uint32_t qa = q_base + t * Cfg::kQTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              uint64_t adesc = smem_desc_sw128(qa + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
              uint64_t bdesc = smem_desc_sw128(k_addr + (kk / 4) * (BK * 128) + (kk % 4) * 32, 16, 1024);
              mma_ss(tmem + t * 256, adesc, bdesc, Cfg::kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bar_s[t]);
            pending[t] = true;
          }
        }
        if (!ok) break;
        mma_commit(&bar_empty[kslot]);
        if (any_pv) mma_commit(&bar_empty[prev_vslot]);
        prev_vslot = vslot;
        prev_vpar = vpar;
      }
      if (ok) {
        bool any_pv = false, v_ready = false;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (!pending[t]) continue;
          if (!v_ready) {
            if (!bounded_wait(&bar_full[prev_vslot], prev_vpar, wc)) break;
            v_ready = true;
          }
          if (!bounded_wait(&bar_p[t], pv_count[t] & 1, wc)) break;
          tc_fence_after();
          issue_pv(t, prev_vslot);
          any_pv = true;
        }
        if (any_pv) mma_commit(&bar_empty[prev_vslot]);
      }
      // the epilogues wait for the last PVs here (a commit tracks every earlier MMA of this thread)
#pragma unroll
      for (int t = 0; t < NQT; ++t) mma_commit(&bar_o[t]);
      // every MMA issued by this thread has completed before TMEM is released
      mma_commit(&bar_mma_done);
      drain_wait(&bar_mma_done, 0, wc);
    }
  }
  } else {
    setmaxnreg_inc<Cfg::kRegsSoftmax>();
    // ======================= softmax + epilogue =======================
    const int t = warp >> 2;
    const int w4 = warp & 3;
    const int r = w4 * 32 + lane;                  // row within the tile = TMEM lane
    const int qtile = tile_of(t);
    int grow = qtile * 128 + r;                    // row within the head
    bool row_valid = grow < p.Sq;
    int na_ws[3] = {0, 0, 0};                      // this row's window start per axis
    if constexpr (kNA) {
      const bool second = t == 1 && n_valid_tiles == 2;   // warp-uniform
      const int c[3] = {(second ? naw.org[1][0] : naw.org[0][0]) + r / (Cfg::kNaY * Cfg::kNaX),
                        (second ? naw.org[1][1] : naw.org[0][1]) + (r / Cfg::kNaX) % Cfg::kNaY,
                        (second ? naw.org[1][2] : naw.org[0][2]) + r % Cfg::kNaX};
      row_valid = c[0] < p.na_L[0] && c[1] < p.na_L[1] && c[2] < p.na_L[2];
      grow = (c[0] * p.na_L[1] + c[1]) * p.na_L[2] + c[2];
#pragma unroll
      for (int a = 0; a < 3; ++a) na_ws[a] = na_window_start(min(c[a], p.na_L[a] - 1), p.na_K[a], p.na_L[a]);
    }
    const int qb = (QB == 2) ? (w4 >> 1) : 0;      // warp-uniform
    // list bits: of the CTA's merged walk, or (independent tiles) of this tile's own walk
    const uint32_t my_bit = Cfg::kDual ? (1u << qb) : (1u << (t * QB + qb));
    const uint32_t tile_mask = Cfg::kDual ? ((1u << QB) - 1u) : (((1u << QB) - 1u) << (t * QB));
    TileMerge<QB> wk;
    if constexpr (Cfg::kDual)
      tile_walk_init<QB, Cfg::kSparseLike>(wk, p, bh, qtile, t < n_valid_tiles, (kv_hi - kv_lo + BK - 1) / BK);
    const uint32_t lane_base = (uint32_t)(w4 * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 256;
    const uint32_t tO = tS + 128;
    if (MODE == kModeSparseFused) {
      float* chunk = reinterpret_cast<float*>(sKV);
      float* prow = chunk + Cfg::kFusedCH * D;
      float* qs = prow + FR * FKMAX;
      fused_route<D, FR, Cfg::kFusedCH, FKMAX, NQT * 128>(p, bh, qg * NQT * QB, tid, chunk, prow, qs, f_lists, f_cnt,
                                                         f_mu, f_W, f_T);
      if (tid == 0) mbar_arrive(&bar_route);
      take_fused_lists();
    }
    float m_run = -INFINITY;
    float l_run = 0.f;
    int it = 0;
    uint32_t flags;
    int u;
    bool ok = t < n_valid_tiles;
    while (ok && (u = next_step<Cfg::kDual, kNA>(wk, naw, merge, flags, na_box)) >= 0) {
      if (!(flags & tile_mask)) continue;
      if (!__all_sync(0xffffffffu, bounded_wait(&bar_s[t], it & 1, wc))) break;
      tc_fence_after();
      float x[BK];
      {
        uint32_t rr[BK / 32][32];
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) tmem_ld32(tS + c * 32, rr[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) {
          tmem_reg_fence(rr[c]);
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c * 32 + j] = __uint_as_float(rr[c][j]);
        }
      }
      const int n_valid = min(BK, kv_hi - (kv_lo + u * BK));
      const bool mine = (flags & my_bit) != 0;
      // raw scores stay unscaled: the softmax scale is positive, so the max
      // commutes with it and the scaling folds into the exponent's FFMA
      if constexpr (kNA) {
        na_mask_scores<Cfg::kNaT, Cfg::kNaY, Cfg::kNaX, BK>(x, na_ws, na_box, p.na_K);
      } else if (!(mine && n_valid == BK)) {
#pragma unroll
        for (int c = 0; c < BK; ++c)
          if (!mine || c >= n_valid) x[c] = -INFINITY;
      }
      softmax_step<BK, D>(x, p.scale_log2, m_run, l_run, it > 0, tS, tO);
      tc_fence_before();
      mbar_arrive(&bar_p[t]);
      ++it;
    }
    // ---- epilogue
    if (t < n_valid_tiles && !abort_flag) {
      bool have_o = it > 0;
      // (every issuer commits bar_o once, after its last PV)
      if (have_o && !__all_sync(0xffffffffu, bounded_wait(&bar_o[t], 0, wc))) have_o = false;
      tc_fence_after();
      if (MODE == kModeSplit) {
        const bool empty = !have_o || l_run == 0.f;
        const float inv = empty ? 0.f : 1.f / l_run;
        const long long orow = ((long long)chunk * p.BH + bh) * p.Sq + grow;
        float* dst = p.out_part + orow * D;
        // rows of D floats start on 32-byte boundaries when the partials do: whole
        // 32-byte sectors per lane then (half the store instructions)
        const bool wide = ((uintptr_t)p.out_part & 31u) == 0;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          if (have_o) {
            tmem_ld32(tO + c0, rr);
            tmem_ld_wait();
            tmem_reg_fence(rr);
          }
          if (row_valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint32_t o[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] = __float_as_uint(have_o ? __uint_as_float(rr[j + e]) * inv : 0.f);
              if (wide) {
                if (ATTN_CHECKED(orow * D + c0 + j, 8, (long long)p.n_split * p.BH * p.Sq * D, p.status))
                  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + c0 + j),
                               "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                               : "memory");
              } else {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                  if (ATTN_CHECKED(orow * D + c0 + j + 4 * h, 4, (long long)p.n_split * p.BH * p.Sq * D, p.status))
                    *reinterpret_cast<uint4*>(dst + c0 + j + 4 * h) =
                        make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
              }
            }
          }
        }
        if (row_valid && ATTN_CHECKED(orow, 1, (long long)p.n_split * p.BH * p.Sq, p.status))
          p.lse_part[orow] = empty ? -INFINITY : (m_run + __log2f(l_run)) * kLn2;
      } else {
        // Taylor term for the rejected blocks of this row's query block (none
        // when the row met no key: an empty, i.e. corrupt, list; its row becomes zeros)
        float f = 0.f;
        const float* tt = nullptr;
        if (MODE == kModeSparseFused && m_run > -INFINITY) {
          const int l = t * QB + qb;
          if (qg * NQT * QB + l < p.NQB && f_cnt[l] < p.NKB) {
            f = ex2_approx(f_mu[l] * kLog2e - m_run);
            l_run += f * f_W[l];
            tt = f_T + l * D;
          }
        }
        if (MODE == kModeSparse && m_run > -INFINITY) {
          const long long qbi = (long long)qtile * QB + qb;
          if (qbi < p.NQB) {
            const long long srow = (long long)bh * p.NQB + qbi;
            const int cnt = __ldg(p.sel_cnt + srow);
            if (cnt < p.NKB) {
              const float mu = __ldg(p.stats + srow * 4 + 0);
              const float W = __ldg(p.stats + srow * 4 + 3);
              f = ex2_approx(mu * kLog2e - m_run);
              l_run += f * W;
              tt = p.taylor_t + srow * D;
            }
          }
        }
        const bool empty = !have_o || !(l_run > 0.f);
        if (empty && row_valid && it == 0 && Cfg::kSparseLike) atomicOr(p.status, ATTN_DEVICE_BAD_LIST);
        const float inv = empty ? 0.f : 1.f / l_run;
        // rows of D bf16 start on 32-byte boundaries when the output does: whole 32-byte sectors per lane
        if (have_o && ((uintptr_t)p.out & 31u) == 0)
          store_row_bf16_wide<D>(tO, inv, f, tt, row_valid, p.out + ((long long)bh * p.Sq + grow) * D,
                                 ((long long)bh * p.Sq + grow) * D, (long long)p.BH * p.Sq * D, p.status);
        else
          store_row_bf16<D>(tO, have_o, inv, f, tt, row_valid, p.out + ((long long)bh * p.Sq + grow) * D,
                            ((long long)bh * p.Sq + grow) * D, (long long)p.BH * p.Sq * D, p.status);
        if (row_valid && p.lse != nullptr && ATTN_CHECKED((long long)bh * p.Sq + grow, 1, (long long)p.BH * p.Sq, p.status))
          p.lse[(long long)bh * p.Sq + grow] = empty ? -INFINITY : (m_run + __log2f(l_run)) * kLn2;
      }
    }
    // reached by all 128 softmax threads whatever happened above (its barriers have no time limit)
    if constexpr (MODE == kModeSplit) {
      if (p.merge_count != nullptr)
        split_merge_tail<D>(p, bh, qg, q_row0, r, merge_last, abort_flag, reinterpret_cast<float*>(sKV));
    }
  }

  }   // !skip_cta

  tc_fence_before();
  __syncthreads();
  if (warp == Cfg::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace vdtb
