// Persistent tcgen05 kernel for 3D neighbourhood attention: one query brick
// per tile, two tiles per CTA, one CTA per SM, each tile walking its own
// sequence of bricks.
//
// Why: a one-brick CTA multiplies only a handful of key boxes (six for a
// 4x4x8 brick under a 3x7x7 window), so its prologue (barrier setup, TMEM
// allocation, the first Q and K loads) and its epilogue (reading O, storing
// the rows) take a large share of its life, during which its tensor work is
// idle.  Here a CTA is set up once; tile t of CTA c takes the bricks
// c*2 + t, c*2 + t + 2*grid, ... (head-major, bricks x fastest), and its
// roles treat the concatenation of those bricks' key boxes as one stream:
//   - group g of the tile's producer loads the K box of stream element g and
//     the V box of element g-1 (and, when g starts a brick, that brick's Q
//     tile, whose slot the last score MMA of the previous brick has freed);
//   - batch g of the tile's issuer is PV(g-1) then S(g) with the window step
//     (see NABiasLayout), under the issue lock that alternates the two tiles'
//     batches on the tensor pipe, with one commit that tells the softmax (S
//     ready) and the producer (slots free); the first PV of a brick
//     overwrites O;
//   - the tile's softmax warpgroup writes the window rows of element g+1
//     while S(g) is computed, and on the batch that starts a brick first
//     reads the previous brick's O out of TMEM (that batch held its last PV)
//     and stores all but its last 64 columns, then runs the softmax of the
//     new brick's first scores, and stores those 64 columns once it has
//     released P.
// So one tile's epilogue and Q load overlap the other tile's MMAs.  The
// online softmax and normalisation are those of attn_fwd_kernel's
// neighbourhood modes; the key boxes tile the union of the brick's windows
// from its corner, in the brick's own shape (KEYS = kNAKeysBrick: the boxes of
// that kernel's one-brick walk) or as 4 x 2 x 16 boxes (kNAKeysWide, fewer
// boxes per 4 x 4 x 8 brick under small windows; kNAKeysWideF8: the same boxes
// with E5M2 window operands, see NABiasLayout).  The window, added by the
// tensor core instead of masked by the softmax threads, leaves every
// in-window score unchanged, so with the brick-shaped boxes results are
// bit-identical to that kernel's one-brick plan (with the wide boxes, equal
// up to the rounding of another key order; the two encodings of the wide
// boxes' window give the same bits wherever both are exact).
#pragma once
#include "attn_fwd.cuh"

namespace vdtb {

// The bricks of one tile and their key boxes, in visiting order.  Unit w =
// head * bricks per head + brick (bricks x fastest); the tile takes units
// first, first + 2 * grid, ... below BH * bricks per head.  A brick is BT x
// BY x BX queries, a key box KT x KY x KX keys (128 each; the key boxes tile
// the union of the brick's windows from its corner).  Only what the next box
// needs is kept; a brick's head and origin are handed out when it starts (so
// they hold no registers between bricks).  Within a brick the box index steps
// like an odometer (x fastest), without divisions.
template <int BT, int BY, int BX, int KT, int KY, int KX>
struct NABrickStream {
  int w;          // next unit
  int lo[3];      // origin of the current brick's box grid (corner of the union of its rows' windows)
  int nk[3];      // boxes per axis
  int ix[3];      // index of the next box; ix[0] == nk[0]: the brick is done

  __device__ __forceinline__ void init(int first) {
    w = first;
    ix[0] = nk[0] = 0;
    ix[1] = ix[2] = nk[1] = nk[2] = 1;
  }
  // Next key box of the stream: its origin `box` and its index `bi` in the
  // brick's box grid (box = lo + bi * key box).  When it starts a brick,
  // `starts` is set and bh / org / glo receive the brick's head, origin and
  // box-grid origin.  False at the end.
  __device__ __forceinline__ bool next(const FwdParams& p, int (&box)[3], int (&bi)[3], bool& starts, int& bh,
                                       int (&org)[3], int (&glo)[3]) {
    starts = ix[0] >= nk[0];
    if (starts) {
      const int per = p.na_nq[0] * p.na_nq[1] * p.na_nq[2];
      if (w >= p.BH * per) return false;
      bh = w / per;
      int b = w - bh * per;
      int id[3];
      id[2] = b % p.na_nq[2];
      b /= p.na_nq[2];
      id[1] = b % p.na_nq[1];
      id[0] = b / p.na_nq[1];
      const int B[3] = {BT, BY, BX}, KB[3] = {KT, KY, KX};
#pragma unroll
      for (int a = 0; a < 3; ++a) {
        org[a] = id[a] * B[a];
        const int last = min(org[a] + B[a], p.na_L[a]) - 1;
        lo[a] = na_window_start(org[a], p.na_K[a], p.na_L[a]);
        const int hi = na_window_start(last, p.na_K[a], p.na_L[a]) + p.na_K[a];
        nk[a] = (hi - lo[a] + KB[a] - 1) / KB[a];
        glo[a] = lo[a];
        ix[a] = 0;
      }
      w += 2 * (int)gridDim.x;
    }
#pragma unroll
    for (int a = 0; a < 3; ++a) bi[a] = ix[a];
    box[0] = lo[0] + bi[0] * KT;
    box[1] = lo[1] + bi[1] * KY;
    box[2] = lo[2] + bi[2] * KX;
    if (++ix[2] == nk[2]) {
      ix[2] = 0;
      if (++ix[1] == nk[1]) {
        ix[1] = 0;
        ++ix[0];
      }
    }
    return true;
  }
};

// The window of a query row, added to its scores by the tensor core.  The
// window separates over the axes: key j of a box (frame tk, row yk, column xk
// within the box) is in the row's window when each coordinate lies in the
// window's range on its axis.  One extra K-step of the score MMA contracts
//   A = Qm [128 rows][KB]: per row and per axis coordinate, 0 when the
//       coordinate is in the row's window, else -b (written per box), with
//   B = Km [128 keys][KB]: per key, a one-hot of each of its coordinates
//       (value c, constant);
// so a key in the window gets x + 0 = x (its score unchanged, bit for bit)
// and a key outside gets x - b c or less.  bf16 operands: b = 2^120, c = 1,
// which the softmax's exponent turns into an exact 0 whenever scale * log2(e)
// >= 2^-80 (|x| < 2^96 leaves x - 2^120 = -2^120).  E5M2 operands (F8): b = c =
// 57344 (the largest finite E5M2 value), b c = 49 * 2^26 exactly in fp32, so
// with |x| < 2^30 a key outside scores below -2^31 and its exponent is an exact
// 0 whenever scale * log2(e) >= 2^-22; one f8f6f4 MMA of K = 32 takes the
// window (two bf16 ones), in half the shared memory.  Frame one-hots are only
// needed when the brick or the key box has several frames (a one-frame
// brick's one-frame boxes all lie in its frame window).  KT x KY x KX: the key
// box; kFrames: frame one-hots kept.  With E5M2 operands the column
// one-hots start on a 16-byte chunk of their own, so a row whose column
// window did not move between two boxes keeps that chunk (write_window_row;
// measured faster there, slower with the bf16 brick-shaped boxes).
template <int KT, int KY, int KX, bool kFrames, bool F8 = false>
struct NABiasLayout {
  static constexpr int kElem = F8 ? 1 : 2;             // bytes per element
  static constexpr int kKStep = F8 ? 32 : 16;          // K of one MMA
  // no-swizzle K-major layout: core matrices of 8 rows x 16 bytes (128 bytes
  // each, kCore elements per row); the kCols / kCore core matrices of an
  // 8-row group are adjacent; one MMA step spans two of them (256 bytes)
  static constexpr int kCore = 16 / kElem;
  static constexpr int kT0 = 0;                        // first frame column
  static constexpr int kY0 = kFrames ? KT : 0;         // first row column
  static constexpr bool kKeepChunks = F8;              // rows rewrite only the chunks that change
  static constexpr int kX0 = kKeepChunks ? (kY0 + KY + kCore - 1) / kCore * kCore : kY0 + KY;   // first column column
  static constexpr int kUsed = kX0 + KX;
  static constexpr int kCols = (kUsed + kKStep - 1) / kKStep * kKStep;   // K of the bias step
  static constexpr int kBytes = 128 * kCols * kElem;   // one operand (128 rows)
  static constexpr int kChunks = kCols / kCore;        // 16-byte chunks of a row
  static constexpr uint32_t kLBO = 128;
  static constexpr uint32_t kSBO = kCols / kCore * 128;
  static constexpr uint32_t kStepBytes = kKStep / kCore * 128;
  __device__ __forceinline__ static uint32_t offset(int row, int col) {
    return (uint32_t)(((row >> 3) * (kCols / kCore) + col / kCore) * 128 + (row & 7) * 16 + (col % kCore) * kElem);
  }
};

template <int D, int MODE, int KEYS>
struct NAPersistCfg {
  static constexpr int BT = na_brick_t(MODE), BY = na_brick_y(MODE), BX = na_brick_x(MODE);
  static constexpr int KT = na_keys_t(MODE, KEYS), KY = na_keys_y(MODE, KEYS), KX = na_keys_x(MODE, KEYS);
  static constexpr int BK = 128;
  static constexpr bool kFrames = BT > 1 || KT > 1;
  static constexpr bool kF8 = KEYS == kNAKeysWideF8;   // E5M2 window operands
  using Bias = NABiasLayout<KT, KY, KX, kFrames, kF8>;
  static constexpr int kWin = kF8 ? kWinF8 : kWinBf16;
  // two softmax warpgroups (one per tile) + one control warpgroup: warps 8, 9
  // are tile 0's producer and issuer, 10, 11 tile 1's
  static constexpr int kThreads = 384;
  static constexpr int kRegsLaunch = 168;
  static constexpr int kRegsControl = 64;
  static constexpr int kRegsSoftmax = 216;
  static_assert(256 * kRegsSoftmax + 128 * kRegsControl <= kThreads * kRegsLaunch, "register split");
  static constexpr int kQTileBytes = 128 * D * 2;
  static constexpr int kSlotBytes = BK * D * 2;
  // Q tiles, K/V slots, the key one-hots, the two tiles' window rows: two
  // buffers per tile where they fit (the rows of element g+1 are then written
  // while S(g) is computed), else one (written once S(g) is done)
  static constexpr int kOffKm = 2 * kQTileBytes + 4 * kSlotBytes;
  static constexpr int kOffQm = kOffKm + Bias::kBytes;
  static constexpr int kQmBufs = 1024 + kOffQm + 4 * Bias::kBytes <= 227 * 1024 ? 2 : 1;
  // all 512 TMEM columns: the request is padded past half of the SM's shared
  // memory so that two such CTAs never share an SM
  static constexpr int kSmemRaw = 1024 + kOffQm + 2 * kQmBufs * Bias::kBytes;
  static constexpr int kSmemBytes = kSmemRaw < 120 * 1024 ? 120 * 1024 : kSmemRaw;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, BK, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
  static constexpr uint32_t kIdescWin = kF8 ? idesc_e5m2_f32(128, BK) : kIdescS;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!kF8 || MODE == kModeNA4x4x8, "E5M2 window operands with the wide key boxes only");
  static_assert(is_na_mode(MODE) && BT * BY * BX == 128 && KT * KY * KX == BK, "neighbourhood bricks and key boxes");
  static_assert(kSmemRaw <= 227 * 1024, "shared memory");
};

// bf16 and E5M2 bit patterns
constexpr uint16_t kBf16One = 0x3F80;        // 1.0
constexpr uint16_t kBf16MaskBias = 0xFB80;   // -2^120
constexpr uint8_t kE5M2Big = 0x7B;           // 57344
constexpr uint8_t kE5M2MaskBias = 0xFB;      // -57344

// Row `row` of the window operand for one key box (KT x KY x KX, layout L):
// per axis, 0 for the box coordinates inside the window (rel_ws: the window
// start minus the box origin, extent K), -b for the others (-2^120 in bf16,
// -57344 in E5M2); unused columns 0.  `key` describes what the buffer's row
// holds (the rel_ws it was written for, 10 bits per axis; kNoWindowRow:
// nothing yet): with L::kKeepChunks only the 16-byte chunks of axes whose
// rel_ws changed are written (a brick's boxes mostly move along one axis),
// else the whole row.  Returns the new key.
constexpr uint32_t kNoWindowRow = 0xFFFFFFFFu;
template <class L, int KT, int KY, int KX>
__device__ __forceinline__ uint32_t write_window_row(uint8_t* qm, int row, const int (&rel_ws)[3], const int (&K)[3],
                                                     uint32_t key) {
  const uint32_t nkey = ((uint32_t)rel_ws[0] & 0x3FFu) | (((uint32_t)rel_ws[1] & 0x3FFu) << 10) |
                        (((uint32_t)rel_ws[2] & 0x3FFu) << 20);
  // the chunks each axis's columns occupy
  constexpr uint32_t kTMask = L::kY0 > 0 ? ((2u << ((L::kT0 + KT - 1) / L::kCore)) - (1u << (L::kT0 / L::kCore))) : 0u;
  constexpr uint32_t kYMask = (2u << ((L::kY0 + KY - 1) / L::kCore)) - (1u << (L::kY0 / L::kCore));
  constexpr uint32_t kXMask = (2u << ((L::kX0 + KX - 1) / L::kCore)) - (1u << (L::kX0 / L::kCore));
  uint32_t mask = (1u << L::kChunks) - 1u;
  if (L::kKeepChunks && key != kNoWindowRow) {
    mask = 0;
    if (((key ^ nkey) & 0x3FFu) != 0) mask |= kTMask;
    if (((key ^ nkey) & (0x3FFu << 10)) != 0) mask |= kYMask;
    if (((key ^ nkey) & (0x3FFu << 20)) != 0) mask |= kXMask;
  }
#pragma unroll
  for (int ch = 0; ch < L::kChunks; ++ch) {
    if (!((mask >> ch) & 1u)) continue;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < L::kCore; ++j) {
      const int col = ch * L::kCore + j;
      bool used = false, in = true;
      if (L::kY0 > 0 && col >= L::kT0 && col < L::kT0 + KT) {
        used = true;
        in = col - L::kT0 >= rel_ws[0] && col - L::kT0 < rel_ws[0] + K[0];
      } else if (col >= L::kY0 && col < L::kY0 + KY) {
        used = true;
        in = col - L::kY0 >= rel_ws[1] && col - L::kY0 < rel_ws[1] + K[1];
      } else if (col >= L::kX0 && col < L::kX0 + KX) {
        used = true;
        in = col - L::kX0 >= rel_ws[2] && col - L::kX0 < rel_ws[2] + K[2];
      }
      if constexpr (L::kElem == 1)
        w[j >> 2] |= (used && !in ? (uint32_t)kE5M2MaskBias : 0u) << ((j & 3) * 8);
      else
        w[j >> 1] |= (used && !in ? (uint32_t)kBf16MaskBias : 0u) << ((j & 1) * 16);
    }
    *reinterpret_cast<uint4*>(qm + L::offset(row, ch * L::kCore)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return nkey;
}

template <int D, int MODE, int KEYS>
__global__ void __launch_bounds__(384, 1)
    attn_na_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Cfg = NAPersistCfg<D, MODE, KEYS>;
  using Bias = typename Cfg::Bias;
  constexpr int BK = Cfg::BK;
  using Stream = NABrickStream<Cfg::BT, Cfg::BY, Cfg::BX, Cfg::KT, Cfg::KY, Cfg::KX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;                              // tile t's Q at t * kQTileBytes
  uint8_t* sKV = smem + 2 * Cfg::kQTileBytes;      // tile t's K slot 2t, V slot 2t + 1
  uint8_t* sKm = smem + Cfg::kOffKm;               // key one-hots
  uint8_t* sQm = smem + Cfg::kOffQm;               // tile t's window rows, buffer b at (t * kQmBufs + b) * Bias::kBytes

  __shared__ uint64_t bar_full[2], bar_s[2], bar_p[2], bar_done[2];
  __shared__ int mma_lock;
  __shared__ uint32_t tmem_base_sh;
  __shared__ WaitState wstate;
  __shared__ int skip_cta;   // the launch had already aborted when this CTA started
  WaitState* const wc = &wstate;
  volatile int& abort_flag = wstate.abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_full[t], 1);
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 128);
      mbar_init(&bar_done[t], 1);
    }
    mma_lock = 0;
    skip_cta = wait_state_init(wstate, p.status, p.launch_id);
    fence_barrier_init();
  }
  if (tid < 128) {
    // key tid of a box: frame, row, column one-hots
    constexpr int kWords = Bias::kCols * Bias::kElem / 4;
    uint32_t w[kWords];
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = 0;
    const int tk = tid / (Cfg::KY * Cfg::KX), yk = (tid / Cfg::KX) % Cfg::KY, xk = tid % Cfg::KX;
    const int cols[3] = {Cfg::kFrames ? Bias::kT0 + tk : -1, Bias::kY0 + yk, Bias::kX0 + xk};
#pragma unroll
    for (int a = 0; a < 3; ++a)
      if (cols[a] >= 0) {
        if constexpr (Bias::kElem == 1)
          w[cols[a] >> 2] |= (uint32_t)kE5M2Big << ((cols[a] & 3) * 8);
        else
          w[cols[a] >> 1] |= (uint32_t)kBf16One << ((cols[a] & 1) * 16);
      }
#pragma unroll
    for (int c = 0; c < Bias::kCols; c += Bias::kCore)
      *reinterpret_cast<uint4*>(sKm + Bias::offset(tid, c)) =
          make_uint4(w[c / Bias::kCore * 4], w[c / Bias::kCore * 4 + 1], w[c / Bias::kCore * 4 + 2],
                     w[c / Bias::kCore * 4 + 3]);
    // the tensor core reads these through the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 9) tmem_alloc(&tmem_base_sh, Cfg::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (!skip_cta) {
    if (warp >= 8) {
      setmaxnreg_dec<Cfg::kRegsControl>();
      const int role = warp - 8;
      const int t = role >> 1;
      if (lane == 0) {
        Stream st;
        st.init(blockIdx.x * 2 + t);
        int box[3], bi[3], org[3], glo[3], bh = 0;
        bool starts;
        const int kslot = 2 * t, vslot = 2 * t + 1;
        if ((role & 1) == 0) {
          // ---- TMA producer of tile t: group g = K of element g, V of element g-1, and the
          // brick's Q when g starts a brick; loaded once batch g-1 (PV(g-2), S(g-1)) has completed
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_k);
          tma_prefetch_desc(&tm_v);
          int g = 0, pbh = 0;
          int pbox[3] = {0, 0, 0};
          bool have_prev = false;
          while (true) {
            const bool got = st.next(p, box, bi, starts, bh, org, glo);
            if (!got && !have_prev) break;
            if (g >= 1 && !bounded_wait(&bar_s[t], (g - 1) & 1, wc)) break;
            const bool load_q = got && starts;
            mbar_expect_tx(&bar_full[t], (got ? Cfg::kSlotBytes : 0) + (have_prev ? Cfg::kSlotBytes : 0) +
                                             (load_q ? Cfg::kQTileBytes : 0));
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              if (load_q)
                tma_load_5d(sQ + t * Cfg::kQTileBytes + h * 16384, &tm_q, &bar_full[t], h * 64, org[2], org[1], org[0],
                            bh);
              if (got)
                tma_load_5d(sKV + kslot * Cfg::kSlotBytes + h * (BK * 128), &tm_k, &bar_full[t], h * 64, box[2], box[1],
                            box[0], bh);
              if (have_prev)
                tma_load_5d(sKV + vslot * Cfg::kSlotBytes + h * (BK * 128), &tm_v, &bar_full[t], h * 64, pbox[2],
                            pbox[1], pbox[0], pbh);
            }
#pragma unroll
            for (int a = 0; a < 3; ++a) pbox[a] = box[a];
            pbh = bh;
            have_prev = got;
            ++g;
            if (!got) break;
          }
          // drain: no copy may still be landing when the CTA exits
          if (g >= 1) drain_wait(&bar_full[t], (g - 1) & 1, wc);
        } else {
          // ---- MMA issuer of tile t: batch g = PV(g-1) then S(g) with its window step, under the
          // issue lock, once K/V have landed and the softmax has released P(g-1) and written the
          // window rows of element g (phase g of bar_p)
          const uint32_t q_addr = smem_u32(sQ) + t * Cfg::kQTileBytes;
          const uint32_t k_addr = smem_u32(sKV) + kslot * Cfg::kSlotBytes;
          const uint32_t v_addr = smem_u32(sKV) + vslot * Cfg::kSlotBytes;
          const uint32_t qm_base = smem_u32(sQm) + t * Cfg::kQmBufs * Bias::kBytes;
          const uint32_t km_addr = smem_u32(sKm);
          const uint32_t s_tmem = tmem + t * 256, o_tmem = tmem + t * 256 + 128;
          int g = 0;
          bool pending = false, pending_starts = false;
          while (true) {
            const bool got = st.next(p, box, bi, starts, bh, org, glo);
            if (!got && !pending) break;
            if (!bounded_wait(&bar_full[t], g & 1, wc) || !bounded_wait(&bar_p[t], g & 1, wc)) break;
            tc_fence_after();
            const bool locked = issue_lock(&mma_lock, &abort_flag);
            if (pending) {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                uint64_t bdesc = smem_desc_sw128(v_addr + kk * 16 * 128, BK * 128, 1024);
                mma_ts(o_tmem, s_tmem + kk * 8, bdesc, Cfg::kIdescPV, (!pending_starts || kk > 0) ? 1u : 0u);
              }
            }
            if (got) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                uint64_t adesc = smem_desc_sw128(q_addr + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
                uint64_t bdesc = smem_desc_sw128(k_addr + (kk / 4) * (BK * 128) + (kk % 4) * 32, 16, 1024);
                mma_ss(s_tmem, adesc, bdesc, Cfg::kIdescS, kk > 0 ? 1u : 0u);
              }
              // the window: x + 0 inside, x - b c or less outside
#pragma unroll
              for (int kb = 0; kb < Bias::kCols / Bias::kKStep; ++kb) {
                uint64_t adesc = smem_desc_noswz(qm_base + (g % Cfg::kQmBufs) * Bias::kBytes + kb * Bias::kStepBytes,
                                                 Bias::kLBO, Bias::kSBO);
                uint64_t bdesc = smem_desc_noswz(km_addr + kb * Bias::kStepBytes, Bias::kLBO, Bias::kSBO);
                if constexpr (Cfg::kF8)
                  mma_ss_f8(s_tmem, adesc, bdesc, Cfg::kIdescWin, 1u);
                else
                  mma_ss(s_tmem, adesc, bdesc, Cfg::kIdescWin, 1u);
              }
            }
            if (locked) issue_unlock(&mma_lock);
            mma_commit(&bar_s[t]);
            pending = got;
            pending_starts = starts;
            ++g;
            if (!got) break;
          }
          // every MMA this thread issued has completed before TMEM is released
          mma_commit(&bar_done[t]);
          drain_wait(&bar_done[t], 0, wc);
        }
      }
    } else {
      setmaxnreg_inc<Cfg::kRegsSoftmax>();
      // ======================= softmax + epilogue of tile t =======================
      const int t = warp >> 2;
      const int r = (warp & 3) * 32 + lane;   // row of the brick = TMEM lane
      const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16) + t * 256;
      const uint32_t tO = tS + 128;
      uint8_t* const qm = sQm + t * Cfg::kQmBufs * Bias::kBytes;
      int la = 0;              // elements looked ahead at (their window rows written)
      Stream st;
      st.init(blockIdx.x * 2 + t);
      float m_run = -INFINITY, l_run = 0.f;
      int it = 0;              // batches of this tile consumed (> 0: a brick is open)
      long long orow = -1;     // output row of this thread in the open brick (-1: outside the volume)
      long long next_orow = -1;
      // this row's window start relative to the box grid origin of the brick
      // of the latest element looked ahead at, one byte per axis (a row's
      // window starts at most brick - 1 past the brick's first row's, and a
      // brick is at most 16 wide on every axis)
      uint32_t ws_rel = 0;
      // what this row of each window buffer holds (write_window_row)
      uint32_t wkey0 = kNoWindowRow, wkey1 = kNoWindowRow;
      // The finished brick: this row, O / l in bf16, and the lse.  Rows of D bf16
      // start on 32-byte boundaries when the output does: whole 32-byte sectors
      // per lane then (half the store instructions and sector writes).
      const bool out_wide = ((uintptr_t)p.out & 31u) == 0;
      auto store_brick = [&]() {
        const bool empty = !(l_run > 0.f);
        const float inv = empty ? 0.f : 1.f / l_run;
        const bool row_valid = orow >= 0;
        if (out_wide)
          store_row_bf16_wide<D>(tO, inv, 0.f, nullptr, row_valid, p.out + orow * D, orow * D, (long long)p.BH * p.Sq * D, p.status);
        else
          store_row_bf16<D>(tO, true, inv, 0.f, nullptr, row_valid, p.out + orow * D, orow * D,
                            (long long)p.BH * p.Sq * D, p.status);
        if (row_valid && p.lse != nullptr && ATTN_CHECKED(orow, 1, (long long)p.BH * p.Sq, p.status))
          p.lse[orow] = empty ? -INFINITY : (m_run + __log2f(l_run)) * kLn2;
      };
      // A finished brick whose successor starts in the same stream: its rows
      // leave TMEM as soon as the successor's first scores are ready (O is
      // final then, and the successor's first PV, which overwrites it, waits
      // for this tile's P).  The last 64 columns reach global memory only after
      // that P is released, while the tensor core runs the next batch (32
      // packed bf16 pairs per thread in between; holding all of d = 128 made
      // the softmax spill); the columns before them are stored at once.  The
      // same values as store_brick.
      constexpr int kDeferCols = 64;
      uint32_t pko[kDeferCols / 2];
      long long pend_row = -1;
      float pend_lse = 0.f;
      auto put_cols = [&](uint16_t* dst, long long off, const uint32_t* pk, int ncols) {
        [[maybe_unused]] const long long total = (long long)p.BH * p.Sq * D;
        if (out_wide) {
#pragma unroll
          for (int c = 0; c < 64; c += 16)
            if (c < ncols && ATTN_CHECKED(off + c, 16, total, p.status))
              asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + c), "r"(pk[c / 2]),
                           "r"(pk[c / 2 + 1]), "r"(pk[c / 2 + 2]), "r"(pk[c / 2 + 3]), "r"(pk[c / 2 + 4]),
                           "r"(pk[c / 2 + 5]), "r"(pk[c / 2 + 6]), "r"(pk[c / 2 + 7])
                           : "memory");
        } else {
#pragma unroll
          for (int c = 0; c < 64; c += 8)
            if (c < ncols && ATTN_CHECKED(off + c, 8, total, p.status))
              *reinterpret_cast<uint4*>(dst + c) = make_uint4(pk[c / 2], pk[c / 2 + 1], pk[c / 2 + 2], pk[c / 2 + 3]);
        }
      };
      auto read_brick = [&]() {
        const bool empty = !(l_run > 0.f);
        const float inv = empty ? 0.f : 1.f / l_run;
        pend_lse = empty ? -INFINITY : (m_run + __log2f(l_run)) * kLn2;
        pend_row = orow;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t rr[2][32];
          tmem_ld32(tO + c0, rr[0]);
          tmem_ld32(tO + c0 + 32, rr[1]);
          tmem_ld_wait();
          uint32_t pk[32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tmem_reg_fence(rr[h]);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[16 * h + j] = pack_bf16x2(__uint_as_float(rr[h][2 * j]) * inv, __uint_as_float(rr[h][2 * j + 1]) * inv);
          }
          if (c0 + 64 < D) {
            if (pend_row >= 0) put_cols(p.out + pend_row * D + c0, pend_row * D + c0, pk, 64);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) pko[j] = pk[j];
          }
        }
      };
      auto write_brick = [&]() {
        if (pend_row < 0) return;
        put_cols(p.out + pend_row * D + (D - kDeferCols), pend_row * D + (D - kDeferCols), pko, kDeferCols);
        if (p.lse != nullptr && ATTN_CHECKED(pend_row, 1, (long long)p.BH * p.Sq, p.status)) p.lse[pend_row] = pend_lse;
      };
      // Looks at the next element of the stream and writes this row of its
      // window operand (into a buffer the scores in flight do not read).
      auto look_ahead = [&](bool& starts) -> bool {
        int box[3], bi[3], org[3], glo[3], bh;
        if (!st.next(p, box, bi, starts, bh, org, glo)) return false;
        if (starts) {
          const int rc[3] = {org[0] + r / (Cfg::BY * Cfg::BX), org[1] + (r / Cfg::BX) % Cfg::BY,
                             org[2] + r % Cfg::BX};
          const bool row_valid = rc[0] < p.na_L[0] && rc[1] < p.na_L[1] && rc[2] < p.na_L[2];
          next_orow = row_valid ? (long long)bh * p.Sq + (rc[0] * p.na_L[1] + rc[1]) * p.na_L[2] + rc[2] : -1;
          ws_rel = 0;
#pragma unroll
          for (int a = 0; a < 3; ++a)
            ws_rel |= (uint32_t)(na_window_start(min(rc[a], p.na_L[a] - 1), p.na_K[a], p.na_L[a]) - glo[a]) << (8 * a);
        }
        const int rel[3] = {(int)(ws_rel & 0xffu) - bi[0] * Cfg::KT, (int)((ws_rel >> 8) & 0xffu) - bi[1] * Cfg::KY,
                            (int)(ws_rel >> 16) - bi[2] * Cfg::KX};
        const bool odd = Cfg::kQmBufs == 2 && (la & 1);
        const uint32_t nk = write_window_row<Bias, Cfg::KT, Cfg::KY, Cfg::KX>(
            qm + (la % Cfg::kQmBufs) * Bias::kBytes, r, rel, p.na_K, odd ? wkey1 : wkey0);
        if (odd)
          wkey1 = nk;
        else
          wkey0 = nk;
        ++la;
        return true;
      };
      bool cur_starts = false;
      bool have = look_ahead(cur_starts);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&bar_p[t]);   // phase 0: the first element's window rows
      bool ok = true;
      while (have) {
        const long long starts_orow = next_orow;   // this element's brick row (when it starts one)
        bool next_starts = false;
        // two buffers: the next element's window rows while S of this one is computed
        if constexpr (Cfg::kQmBufs == 2) have = look_ahead(next_starts);
        if (!__all_sync(0xffffffffu, bounded_wait(&bar_s[t], it & 1, wc))) {
          ok = false;
          break;
        }
        ++it;
        tc_fence_after();
        const bool pend = cur_starts && it > 1;
        if (cur_starts) {
          // this batch held the previous brick's last PV: its rows leave TMEM before O is reused
          if (pend) read_brick();
          orow = starts_orow;
          m_run = -INFINITY;
          l_run = 0.f;
        }
        // O holds earlier boxes of this brick unless this box starts it.  One
        // buffer: the next element's window rows now that S is done, while the
        // first score loads are in flight
        softmax_step_tmem<BK, D, Cfg::kWin>(tS, p.scale_log2, m_run, l_run, !cur_starts, tO, [&]() {
          if constexpr (Cfg::kQmBufs == 1) have = look_ahead(next_starts);
        });
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        mbar_arrive(&bar_p[t]);
        if (pend) write_brick();
        cur_starts = next_starts;
      }
      // the last batch (the last brick's last PV alone); lane 0's view of the flag decides for the warp
      const bool fin = __shfl_sync(0xffffffffu, (int)(ok && it > 0 && !abort_flag), 0) != 0;
      if (fin && __all_sync(0xffffffffu, bounded_wait(&bar_s[t], it & 1, wc))) {
        tc_fence_after();
        store_brick();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace vdtb
