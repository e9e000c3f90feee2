// C ABI of the attention hot path (declarations and contracts in attn_api.h).
// Host-side validation, TMA descriptor encoding, workspace carving and
// kernel launches.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>
#include <math.h>
#include <atomic>
#include <mutex>
#include <stdint.h>
#include <string.h>

#include "attn_api.h"
#include "fp8_api.h"
#include "launch.h"

namespace vdtb {

// Two status words per device; kernels receive their address: [0] the status
// bits, [1] the id of the last launch in which a wait timed out (see ptx.cuh).
__device__ int g_status_word[2];

namespace {

constexpr int kMaxDevices = 64;
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_status_mutex;
int* g_status_ptr[kMaxDevices] = {nullptr};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// An NVTX range around each C-ABI call, named after the entry point, so that a
// profiler can select one call's kernels (e.g. ncu --nvtx --nvtx-include).
// Without a profiler attached the push/pop are no-ops.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Every launch of a kernel with barrier waits gets its own id (never 0, the
// abort word's initial value), so a timeout aborts only the launch it
// happened in.
std::atomic<unsigned> g_launch_counter{0};
unsigned next_launch_id() {
  unsigned id;
  do {
    id = g_launch_counter.fetch_add(1u) + 1u;
  } while (id == 0u);
  return id;
}

attn_status_t status_ptr(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_status_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_status_ptr[dev] = (int*)p;
  }
  *out = g_status_ptr[dev];
  return ATTN_OK;
}

attn_status_t get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  });
  return g_encode ? ATTN_OK : ATTN_ERR_CUDA;
}

// 3-D map over a [BH][S][D] bf16 tensor: dims (D, S, BH), box (64, rows, 1),
// 128-byte swizzle; rows past S read as zero.
attn_status_t make_map(CUtensorMap* m, const void* ptr, int D, int S, int BH, int box_rows) {
  if (get_encoder() != ATTN_OK) return ATTN_ERR_CUDA;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 5-D map over a [BH][T][Y][X][D] bf16 tensor (raster token order): dims
// (D, X, Y, T, BH), box (64, bx, by, bt, 1), 128-byte swizzle; positions
// outside the volume read as zero.
attn_status_t make_map_5d(CUtensorMap* m, const void* ptr, int D, int T, int Y, int X, int BH, int bt, int by,
                          int bx) {
  if (get_encoder() != ATTN_OK) return ATTN_ERR_CUDA;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)X, (cuuint64_t)Y, (cuuint64_t)T, (cuuint64_t)BH};
  cuuint64_t strides[4] = {(cuuint64_t)D * 2, (cuuint64_t)X * D * 2, (cuuint64_t)Y * X * D * 2,
                           (cuuint64_t)T * Y * X * D * 2};
  cuuint32_t box[5] = {64, (cuuint32_t)bx, (cuuint32_t)by, (cuuint32_t)bt, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 3-D map over an fp32 tensor with dims (d0, d1, d2) (d0 innermost), row
// strides s1, s2 in bytes, box (box0, box1, 1), 128-byte swizzle (box0 * 4 =
// 128 bytes); elements outside read as zero.
attn_status_t make_map_f32(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                           uint64_t s2, uint32_t box0, uint32_t box1) {
  if (get_encoder() != ATTN_OK) return ATTN_ERR_CUDA;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)s1, (cuuint64_t)s2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 2-D map over a [rows][inner] uint8 matrix (row stride = inner bytes), box
// (box_inner, box_rows), 128-byte swizzle; elements outside read as zero.
attn_status_t make_map_2d_u8(CUtensorMap* m, const void* ptr, int inner, int rows, int box_inner, int box_rows) {
  if (get_encoder() != ATTN_OK) return ATTN_ERR_CUDA;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---- 3D neighbourhood-attention planning (host mirror of NAWalk's geometry)
int na_start(int p, int K, int L) {
  int s = p - K / 2;
  s = s < 0 ? 0 : s;
  return s > L - K ? L - K : s;
}
int na_mode_of(int brick) { return brick == 1 ? kModeNA1x8x16 : brick == 2 ? kModeNA2x8x8 : kModeNA4x4x8; }

// The key boxes of a plan: the brick's own shape, or the wide boxes (plan 5;
// plan 6 with E5M2 window operands).
int na_keys_of(int pair) { return pair == 5 ? kNAKeysWide : pair == 6 ? kNAKeysWideF8 : kNAKeysBrick; }

// Key boxes a (brick, pair axis) plan makes the CTAs multiply, summed over
// every query tile of one head, and the number of CTAs per head (for the
// persistent plans 4, 5 and 6, of bricks).  The count separates over the axes:
// along a non-pair axis a tile's boxes depend only on its own coordinate,
// along the pair axis on the pair it belongs to.
void na_plan_cost(const int L[3], const int K[3], int brick, int pair, long long* boxes, long long* ctas) {
  const int mode = na_mode_of(brick), keys = na_keys_of(pair);
  const int B[3] = {na_brick_t(mode), na_brick_y(mode), na_brick_x(mode)};
  const int KB[3] = {na_keys_t(mode, keys), na_keys_y(mode, keys), na_keys_x(mode, keys)};
  long long prod = 1, n = 1;
  for (int a = 0; a < 3; ++a) {
    const int nq = (L[a] + B[a] - 1) / B[a];
    auto lo_of = [&](int i) { return na_start(i * B[a], K[a], L[a]); };
    auto hi_of = [&](int i) { return na_start((i + 1) * B[a] < L[a] ? (i + 1) * B[a] - 1 : L[a] - 1, K[a], L[a]) + K[a]; };
    long long sum = 0;
    if (a != pair) {   // (pairs 3 to 6: no axis is paired)
      for (int i = 0; i < nq; ++i) sum += (hi_of(i) - lo_of(i) + KB[a] - 1) / KB[a];
      n *= nq;
    } else {
      for (int j = 0; 2 * j < nq; ++j) {
        const int cu = lo_of(2 * j);   // lo is non-decreasing in the brick index
        for (int i = 2 * j; i < 2 * j + 2 && i < nq; ++i)
          sum += (hi_of(i) - 1 - cu) / B[a] - (lo_of(i) - cu) / B[a] + 1;
      }
      n *= (nq + 1) / 2;
    }
    prod *= sum;
  }
  *boxes = prod;
  *ctas = n;
}

// Picks the plan left open by the caller (brick 0, pair -1).  An open pair
// axis means the persistent one-brick tiles: plan 4 (key boxes of the brick's
// shape) or, for the 4x4x8 brick, plan 5 (4x2x16 key boxes), the fastest plans
// on GB300 for every volume and window measured.  The choice minimises a cost
// in twentieths of a key box: 20 per box whose window step is 16 columns wide
// (plan 4 with the 4x4x8 brick), 23 where it is 32 (a wider MMA step and, at
// d = 128, one window buffer instead of two), plus 34 per brick (its epilogue);
// for the other plans 20 per box plus 40 per CTA (a CTA's fixed cost counted as
// two boxes).  The weights are fits to GB300 timings.  Plans 5 and 6 exist for
// the 4x4x8 brick only: asked for with another brick, they are refused (false).
// Plan 6 (plan 5's boxes with E5M2 window operands: two window buffers per
// tile, exact for raw scores |q.k| < 2^30) is taken only when asked for.
bool na_choose(const int L[3], const int K[3], int* brick, int* pair, long long* boxes) {
  if ((*pair == 5 || *pair == 6) && *brick != 0 && *brick != 3) return false;
  long long best = -1;
  int bb = 1, bp = *pair;
  long long bboxes = 0;
  for (int b = 1; b <= 3; ++b) {
    if (*brick != 0 && b != *brick) continue;
    // the caller's pair axis, or (left open) the persistent plans 4 and 5
    const int first = *pair >= 0 ? *pair : 4, last = *pair >= 0 ? *pair : 5;
    for (int cand = first; cand <= last; ++cand) {
      if (cand >= 5 && b != 3) continue;
      long long nbox, ncta;
      na_plan_cost(L, K, b, cand, &nbox, &ncta);
      const bool wide_step = cand == 5 || (cand == 4 && b != 3);
      const long long cost = cand >= 4 ? (wide_step ? 23 : 20) * nbox + 34 * ncta : 20 * nbox + 40 * ncta;
      if (best < 0 || cost < best) {
        best = cost;
        bb = b;
        bp = cand;
        bboxes = nbox;
      }
    }
  }
  *brick = bb;
  *pair = bp;
  *boxes = bboxes;
  return true;
}

attn_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

bool valid_d(int d) { return d == 64 || d == 128; }

cudaError_t launch_fwd(int D, int BK, int mode, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t stream) {
  return D == 128 ? launch_attn_fwd_d128(BK, mode, tq, tk, tv, p, stream)
                  : launch_attn_fwd_d64(BK, mode, tq, tk, tv, p, stream);
}

FwdParams base_params(int B, int H, int Sq, int Skv, float scale, int mode, int* status) {
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.BH = B * H;
  p.Sq = Sq;
  p.Skv = Skv;
  const int rows_per_cta = 128 * fwd_query_tiles(mode);
  p.n_qg = (Sq + rows_per_cta - 1) / rows_per_cta;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.launch_id = next_launch_id();
  return p;
}

// Sizes checked once: products that index memory must fit the kernels' ranges.
bool sizes_ok(long long B, long long H, long long S) {
  return B >= 1 && H >= 1 && S >= 1 && B * H <= 0x7fffffffLL && S <= 0x3fffffffLL;
}

bool na_args_ok(int B, int H, int T, int Y, int X, int Kt, int Ky, int Kx) {
  if (T < 1 || Y < 1 || X < 1) return false;
  const long long S = (long long)T * Y * X;
  if (!sizes_ok(B, H, S)) return false;
  return Kt >= 1 && Kt <= T && Ky >= 1 && Ky <= Y && Kx >= 1 && Kx <= X;
}

struct SparseLayout {
  size_t qp, kp, vp, sel_idx, sel_cnt, stats, taylor, order, kh, kl, vth, vtl, total;
  int NKBp;   // row pitch (floats) of the transposed pooled values
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool sparse_layout(int B, int H, int S, int d, int block_q, int block_k, SparseLayout* L) {
  if (!sizes_ok(B, H, S) || !valid_d(d) || block_q != block_k || (block_q != 64 && block_q != 128)) return false;
  const size_t BH = (size_t)B * H;
  const size_t NQB = (S + block_q - 1) / block_q, NKB = (S + block_k - 1) / block_k;
  if (NKB > 8192) return false;
  size_t off = 0;
  L->qp = off;
  off = align256(off + BH * NQB * d * 4);
  L->kp = off;
  off = align256(off + BH * NKB * d * 4);
  L->vp = off;
  off = align256(off + BH * NKB * d * 4);
  L->sel_idx = off;
  off = align256(off + BH * NQB * NKB * 4);
  L->sel_cnt = off;
  off = align256(off + BH * NQB * 4);
  L->stats = off;
  off = align256(off + BH * NQB * 4 * 4);
  L->taylor = off;
  off = align256(off + BH * NQB * d * 4);
  L->order = off;   // the query-block order of the forward (128-row blocks)
  off = align256(off + BH * NQB * 4);
  // tf32 hi / lo copies of the pooled keys and of the transposed pooled values (tensor-core routing)
  L->NKBp = (int)((NKB + 3) & ~(size_t)3);
  L->kh = off;
  off = align256(off + BH * NKB * d * 4);
  L->kl = off;
  off = align256(off + BH * NKB * d * 4);
  L->vth = off;
  off = align256(off + BH * d * L->NKBp * 4);
  L->vtl = off;
  off = align256(off + BH * d * L->NKBp * 4);
  L->total = off;
  return true;
}

}  // namespace
}  // namespace vdtb

using namespace vdtb;

extern "C" {

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
  }
  return "ATTN_ERR_UNKNOWN";
}

attn_status_t attn_dense_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out, float* lse,
                             int B, int H, int Sq, int Skv, int d, float scale, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_dense_fwd");
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (lse && ((uintptr_t)lse & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, Sq) || !sizes_ok(B, H, Skv) || !(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!valid_d(d)) return ATTN_ERR_UNSUPPORTED;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, q, d, Sq, B * H, 128)) != ATTN_OK) return st;
  if ((st = make_map(&tk, k, d, Skv, B * H, 128)) != ATTN_OK) return st;
  if ((st = make_map(&tv, v, d, Skv, B * H, 128)) != ATTN_OK) return st;
  FwdParams p = base_params(B, H, Sq, Skv, scale, kModeDense, status);
  p.out = out;
  p.lse = lse;
  return cuda_status(launch_fwd(d, 128, kModeDense, tq, tk, tv, p, stream));
}

attn_status_t attn_na3d_plan(int T, int Y, int X, int Kt, int Ky, int Kx, int* brick, int* pair_axis,
                             long long* key_boxes) {
  if (!brick || !pair_axis || !na_args_ok(1, 1, T, Y, X, Kt, Ky, Kx)) return ATTN_ERR_INVALID_ARG;
  if (*brick < 0 || *brick > 3 || *pair_axis < -1 || *pair_axis > 6) return ATTN_ERR_INVALID_ARG;
  const int L[3] = {T, Y, X}, K[3] = {Kt, Ky, Kx};
  long long boxes = 0;
  if (!na_choose(L, K, brick, pair_axis, &boxes)) return ATTN_ERR_INVALID_ARG;
  if (key_boxes) *key_boxes = boxes;
  return ATTN_OK;
}

attn_status_t attn_na3d_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out, float* lse,
                            int B, int H, int T, int Y, int X, int d, int Kt, int Ky, int Kx, float scale, int brick,
                            int pair_axis, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_na3d_fwd");
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (lse && ((uintptr_t)lse & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (!na_args_ok(B, H, T, Y, X, Kt, Ky, Kx) || !(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (brick < 0 || brick > 3 || pair_axis < -1 || pair_axis > 6) return ATTN_ERR_INVALID_ARG;
  if (!valid_d(d)) return ATTN_ERR_UNSUPPORTED;
  const int L[3] = {T, Y, X}, K[3] = {Kt, Ky, Kx};
  long long boxes = 0;
  if (!na_choose(L, K, &brick, &pair_axis, &boxes)) return ATTN_ERR_INVALID_ARG;
  // the persistent plans add the window to the scores on the tensor core (-2^120
  // outside it), which an exponent turns into an exact 0 only for scale * log2(e)
  // >= 2^-80; below that the one-brick CTAs (the window applied as -inf by the
  // softmax threads) give the same results as plan 4 (the same boxes and
  // arithmetic) and plan 5's results up to rounding (other key boxes).  Plan 6's
  // E5M2 window (-49 * 2^26 outside) needs scale * log2(e) >= 2^-22; below that
  // plan 5 gives its results.
  if (pair_axis == 6 && !(scale * 1.4426950408889634f >= 0x1p-22f)) pair_axis = 5;
  if (pair_axis >= 4 && !(scale * 1.4426950408889634f >= 0x1p-80f)) pair_axis = 3;
  const int mode = na_mode_of(brick), keys = na_keys_of(pair_axis);
  const int Bv[3] = {na_brick_t(mode), na_brick_y(mode), na_brick_x(mode)};
  const int KBv[3] = {na_keys_t(mode, keys), na_keys_y(mode, keys), na_keys_x(mode, keys)};
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  const int S = T * Y * X;
  CUtensorMap tq, tk, tv;
  if ((st = make_map_5d(&tq, q, d, T, Y, X, B * H, Bv[0], Bv[1], Bv[2])) != ATTN_OK) return st;
  if ((st = make_map_5d(&tk, k, d, T, Y, X, B * H, KBv[0], KBv[1], KBv[2])) != ATTN_OK) return st;
  if ((st = make_map_5d(&tv, v, d, T, Y, X, B * H, KBv[0], KBv[1], KBv[2])) != ATTN_OK) return st;
  FwdParams p = base_params(B, H, S, S, scale, mode, status);
  long long n_qg = 1;
  for (int a = 0; a < 3; ++a) {
    p.na_L[a] = L[a];
    p.na_K[a] = K[a];
    p.na_nq[a] = (L[a] + Bv[a] - 1) / Bv[a];
    p.na_np[a] = a == pair_axis ? (p.na_nq[a] + 1) / 2 : p.na_nq[a];
    n_qg *= p.na_np[a];
  }
  if (n_qg * B * H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  p.n_qg = (int)n_qg;
  p.na_pair_axis = pair_axis;
  p.out = out;
  p.lse = lse;
  if (pair_axis >= 4)
    return cuda_status(d == 128 ? launch_na_persist_d128(mode, keys, tq, tk, tv, p, stream)
                                : launch_na_persist_d64(mode, keys, tq, tk, tv, p, stream));
  return cuda_status(launch_fwd(d, 128, mode, tq, tk, tv, p, stream));
}

attn_status_t fp8_quantize_rows(const attn_bf16* x, uint8_t* q, float* scale, int M, int K, cudaStream_t stream) {
  const NvtxRange nvtx_range("fp8_quantize_rows");
  if (!x || !q || !scale || !aligned16(x) || !aligned16(q) || ((uintptr_t)scale & 3u)) return ATTN_ERR_INVALID_ARG;
  if (M < 1 || K < 16 || K % 16 != 0 || K > (1 << 30)) return ATTN_ERR_INVALID_ARG;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  return cuda_status(launch_fp8_quantize_rows(x, q, scale, M, K, status, stream));
}

attn_status_t fp8_scaled_gemm(const uint8_t* aq, const float* a_scale, const uint8_t* wq, const float* w_scale,
                              attn_bf16* y, int M, int N, int K, cudaStream_t stream) {
  const NvtxRange nvtx_range("fp8_scaled_gemm");
  if (!aq || !a_scale || !wq || !w_scale || !y) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(aq) || !aligned16(wq) || !aligned16(y) || ((uintptr_t)a_scale & 3u) || !aligned16(w_scale))
    return ATTN_ERR_INVALID_ARG;
  if (M < 1 || N < 8 || N % 8 != 0 || K < 16 || K % 16 != 0 || K > (1 << 30)) return ATTN_ERR_INVALID_ARG;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  CUtensorMap ta, tb;
  if ((st = make_map_2d_u8(&ta, aq, K, M, 128, 128)) != ATTN_OK) return st;
  if ((st = make_map_2d_u8(&tb, wq, K, N, 128, 256)) != ATTN_OK) return st;
  return cuda_status(launch_fp8_gemm(ta, tb, a_scale, w_scale, y, M, N, K, status, next_launch_id(), stream));
}

attn_status_t attn_cross_splitkv_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* out_part,
                                     float* lse_part, int B, int H, int Sq, int Skv, int d, int n_split, float scale,
                                     cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_cross_splitkv_fwd");
  if (!q || !k || !v || !out_part || !lse_part) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out_part) || ((uintptr_t)lse_part & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, Sq) || !sizes_ok(B, H, Skv) || !(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (n_split < 1 || n_split > Skv) return ATTN_ERR_INVALID_ARG;
  if (!valid_d(d)) return ATTN_ERR_UNSUPPORTED;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, q, d, Sq, B * H, 128)) != ATTN_OK) return st;
  if ((st = make_map(&tk, k, d, Skv, B * H, 128)) != ATTN_OK) return st;
  if ((st = make_map(&tv, v, d, Skv, B * H, 128)) != ATTN_OK) return st;
  FwdParams p = base_params(B, H, Sq, Skv, scale, kModeSplit, status);
  p.out_part = out_part;
  p.lse_part = lse_part;
  p.n_split = n_split;
  return cuda_status(launch_fwd(d, 128, kModeSplit, tq, tk, tv, p, stream));
}

size_t attn_cross_workspace_bytes(int B, int H, int Sq, int d, int n_split) {
  if (!sizes_ok(B, H, Sq) || !valid_d(d) || n_split < 1) return 0;
  const size_t rows = (size_t)B * H * Sq;
  const size_t tiles = (size_t)B * H * ((Sq + 127) / 128);
  return align256((size_t)n_split * rows * d * 4) + align256((size_t)n_split * rows * 4) + align256(tiles * 4);
}

attn_status_t attn_cross_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out, float* lse,
                             int B, int H, int Sq, int Skv, int d, int n_split, float scale, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_cross_fwd");
  if (!q || !k || !v || !out || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(workspace) ||
      (lse && ((uintptr_t)lse & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, Sq) || !sizes_ok(B, H, Skv) || !(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (n_split < 1 || n_split > Skv) return ATTN_ERR_INVALID_ARG;
  if (!valid_d(d)) return ATTN_ERR_UNSUPPORTED;
  if (n_split > kMergeMaxSplit) return ATTN_ERR_UNSUPPORTED;
  const size_t need = attn_cross_workspace_bytes(B, H, Sq, d, n_split);
  if (workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, q, d, Sq, B * H, 128)) != ATTN_OK) return st;
  if ((st = make_map(&tk, k, d, Skv, B * H, 128)) != ATTN_OK) return st;
  if ((st = make_map(&tv, v, d, Skv, B * H, 128)) != ATTN_OK) return st;
  const size_t rows = (size_t)B * H * Sq;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  FwdParams p = base_params(B, H, Sq, Skv, scale, kModeSplit, status);
  p.out_part = reinterpret_cast<float*>(ws);
  p.lse_part = reinterpret_cast<float*>(ws + align256((size_t)n_split * rows * d * 4));
  p.merge_count = reinterpret_cast<int*>(ws + align256((size_t)n_split * rows * d * 4) +
                                         align256((size_t)n_split * rows * 4));
  p.n_split = n_split;
  p.out = out;
  p.lse = lse;
  return cuda_status(launch_fwd(d, 128, kModeSplit, tq, tk, tv, p, stream));
}

attn_status_t attn_lse_merge(const float* out_part, const float* lse_part, attn_bf16* out, float* lse, int n_split,
                             int B, int H, int Sq, int d, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_lse_merge");
  if (!out_part || !lse_part || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(out_part) || ((uintptr_t)lse_part & 3u) || !aligned16(out) || (lse && ((uintptr_t)lse & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, Sq) || n_split < 1) return ATTN_ERR_INVALID_ARG;
  if (!valid_d(d)) return ATTN_ERR_UNSUPPORTED;
  const long long rows = (long long)B * H * Sq;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  return cuda_status(launch_merge(out_part, lse_part, out, lse, n_split, rows, d, status, stream));
}

attn_status_t attn_block_pool(const attn_bf16* x, float* x_pool, int B, int H, int S, int d, int block,
                              cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_block_pool");
  if (!x || !x_pool || !aligned16(x) || !aligned16(x_pool)) return ATTN_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, S)) return ATTN_ERR_INVALID_ARG;
  if (!valid_d(d) || (block != 64 && block != 128)) return ATTN_ERR_UNSUPPORTED;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  return cuda_status(launch_pool(x, x, x, x_pool, x_pool, x_pool, 1, B * H, S, d, block, PoolSplit{}, status, stream));
}

size_t attn_sparse_workspace_bytes(int B, int H, int S, int d, int block_q, int block_k) {
  SparseLayout L;
  if (!sparse_layout(B, H, S, d, block_q, block_k, &L)) return 0;
  return L.total;
}

namespace {

struct SparseArgs {
  const attn_bf16 *q, *k, *v;
  int B, H, S, d, block_q, block_k;
  float scale;
};

attn_status_t sparse_common_checks(const SparseArgs& a) {
  if (!a.q || !a.k || !a.v) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v)) return ATTN_ERR_INVALID_ARG;
  if (!sizes_ok(a.B, a.H, a.S) || !(isfinite(a.scale) && a.scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!valid_d(a.d) || a.block_q != a.block_k || (a.block_q != 64 && a.block_q != 128)) return ATTN_ERR_UNSUPPORTED;
  SparseLayout L;
  if (!sparse_layout(a.B, a.H, a.S, a.d, a.block_q, a.block_k, &L)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn_status_t run_route(const SparseArgs& a, float beta, void* workspace, size_t workspace_bytes, int32_t* si,
                        int32_t* sc, float* stt, float* tt, int32_t* order, cudaStream_t stream) {
  SparseLayout L;
  if (!sparse_layout(a.B, a.H, a.S, a.d, a.block_q, a.block_k, &L)) return ATTN_ERR_UNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.total) return ATTN_ERR_WORKSPACE;
  uint8_t* ws = (uint8_t*)workspace;
  float* qp = (float*)(ws + L.qp);
  float* kp = (float*)(ws + L.kp);
  float* vp = (float*)(ws + L.vp);
  const int BH = a.B * a.H;
  const int NQB = (a.S + a.block_q - 1) / a.block_q, NKB = (a.S + a.block_k - 1) / a.block_k;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  PoolSplit split;
  split.kh = (float*)(ws + L.kh);
  split.kl = (float*)(ws + L.kl);
  split.vth = (float*)(ws + L.vth);
  split.vtl = (float*)(ws + L.vtl);
  split.NBp = L.NKBp;
  CUtensorMap tkh, tkl, tvh, tvl;
  const uint64_t d = (uint64_t)a.d, nk = (uint64_t)NKB, nkp = (uint64_t)L.NKBp;
  if ((st = make_map_f32(&tkh, split.kh, d, nk, BH, d * 4, nk * d * 4, 32, 128)) != ATTN_OK) return st;
  if ((st = make_map_f32(&tkl, split.kl, d, nk, BH, d * 4, nk * d * 4, 32, 128)) != ATTN_OK) return st;
  if ((st = make_map_f32(&tvh, split.vth, nk, d, BH, nkp * 4, d * nkp * 4, 32, (uint32_t)d)) != ATTN_OK) return st;
  if ((st = make_map_f32(&tvl, split.vtl, nk, d, BH, nkp * 4, d * nkp * 4, 32, (uint32_t)d)) != ATTN_OK) return st;
  CUtensorMap tqp;
  const uint64_t nq = (uint64_t)NQB;
  if ((st = make_map_f32(&tqp, qp, d, nq, BH, d * 4, nq * d * 4, 32, 128)) != ATTN_OK) return st;
  if (launch_pool(a.q, a.k, a.v, qp, kp, vp, 3, BH, a.S, a.d, a.block_q, split, status, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (launch_route_tc(tkh, tkl, tvh, tvl, tqp, qp, kp, vp, BH, NQB, NKB, a.S, a.d, a.block_k, a.scale, beta, si, sc,
                      stt, tt, status, next_launch_id(), stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (order != nullptr && launch_qb_order(sc, order, BH, NQB, NKB, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status_t run_sparse_fwd(const SparseArgs& a, attn_bf16* out, float* lse, const int32_t* si, const int32_t* sc,
                             const float* stt, const float* tt, const int32_t* order, cudaStream_t stream) {
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  const int BH = a.B * a.H;
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, a.q, a.d, a.S, BH, 128)) != ATTN_OK) return st;
  if ((st = make_map(&tk, a.k, a.d, a.S, BH, a.block_k)) != ATTN_OK) return st;
  if ((st = make_map(&tv, a.v, a.d, a.S, BH, a.block_k)) != ATTN_OK) return st;
  FwdParams p = base_params(a.B, a.H, a.S, a.S, a.scale, kModeSparse, status);
  p.out = out;
  p.lse = lse;
  p.sel_idx = si;
  p.sel_cnt = sc;
  p.stats = stt;
  p.taylor_t = tt;
  p.NQB = (a.S + a.block_q - 1) / a.block_q;
  p.NKB = (a.S + a.block_k - 1) / a.block_k;
  p.qb_order = a.block_q == 128 ? order : nullptr;
  return cuda_status(launch_fwd(a.d, a.block_k, kModeSparse, tq, tk, tv, p, stream));
}

// A query-block order is for 128-row blocks only and must be 4-byte aligned.
bool bad_order(const int32_t* order, int block_q) {
  return order != nullptr && (block_q != 128 || ((uintptr_t)order & 3u));
}

bool bad_opt_ptrs(const int32_t* si, const int32_t* sc, const float* stt, const float* tt) {
  return (si && ((uintptr_t)si & 3u)) || (sc && ((uintptr_t)sc & 3u)) || (stt && !aligned16(stt)) ||
         (tt && !aligned16(tt));
}

}  // namespace

attn_status_t attn_sparse_route(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, int B, int H, int S,
                                int d, float scale, float beta, int block_q, int block_k, void* workspace,
                                size_t workspace_bytes, int32_t* sel_idx, int32_t* sel_cnt, float* stats,
                                float* taylor_t, int32_t* qb_order, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_sparse_route");
  SparseArgs a{q, k, v, B, H, S, d, block_q, block_k, scale};
  attn_status_t st = sparse_common_checks(a);
  if (st != ATTN_OK) return st;
  if (!sel_idx || !sel_cnt || !stats || !taylor_t || bad_opt_ptrs(sel_idx, sel_cnt, stats, taylor_t) || isnan(beta) ||
      beta == INFINITY || bad_order(qb_order, block_q))
    return ATTN_ERR_INVALID_ARG;
  return run_route(a, beta, workspace, workspace_bytes, sel_idx, sel_cnt, stats, taylor_t, qb_order, stream);
}

attn_status_t attn_sparse_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out, float* lse,
                              int B, int H, int S, int d, float scale, int block_q, int block_k,
                              const int32_t* sel_idx, const int32_t* sel_cnt, const float* stats,
                              const float* taylor_t, const int32_t* qb_order, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_sparse_fwd");
  SparseArgs a{q, k, v, B, H, S, d, block_q, block_k, scale};
  attn_status_t st = sparse_common_checks(a);
  if (st != ATTN_OK) return st;
  if (!out || !aligned16(out) || (lse && ((uintptr_t)lse & 3u))) return ATTN_ERR_INVALID_ARG;
  if (!sel_idx || !sel_cnt || !stats || !taylor_t || bad_opt_ptrs(sel_idx, sel_cnt, stats, taylor_t) ||
      bad_order(qb_order, block_q))
    return ATTN_ERR_INVALID_ARG;
  return run_sparse_fwd(a, out, lse, sel_idx, sel_cnt, stats, taylor_t, qb_order, stream);
}

attn_status_t attn_sparse_route_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out,
                                    float* lse, int B, int H, int S, int d, float scale, float beta, int block_q,
                                    int block_k, void* workspace, size_t workspace_bytes, int32_t* sel_idx,
                                    int32_t* sel_cnt, float* stats, float* taylor_t, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_sparse_route_fwd");
  SparseArgs a{q, k, v, B, H, S, d, block_q, block_k, scale};
  attn_status_t st = sparse_common_checks(a);
  if (st != ATTN_OK) return st;
  if (!out || !aligned16(out) || (lse && ((uintptr_t)lse & 3u)) || bad_opt_ptrs(sel_idx, sel_cnt, stats, taylor_t))
    return ATTN_ERR_INVALID_ARG;
  if (isnan(beta) || beta == INFINITY) return ATTN_ERR_INVALID_ARG;
  SparseLayout L;
  if (!sparse_layout(B, H, S, d, block_q, block_k, &L)) return ATTN_ERR_UNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.total) return ATTN_ERR_WORKSPACE;
  uint8_t* ws = (uint8_t*)workspace;
  int32_t* si = sel_idx ? sel_idx : (int32_t*)(ws + L.sel_idx);
  int32_t* sc = sel_cnt ? sel_cnt : (int32_t*)(ws + L.sel_cnt);
  float* stt = stats ? stats : (float*)(ws + L.stats);
  float* tt = taylor_t ? taylor_t : (float*)(ws + L.taylor);
  int32_t* order = block_q == 128 ? (int32_t*)(ws + L.order) : nullptr;
  if ((st = run_route(a, beta, workspace, workspace_bytes, si, sc, stt, tt, order, stream)) != ATTN_OK) return st;
  return run_sparse_fwd(a, out, lse, si, sc, stt, tt, order, stream);
}

attn_status_t attn_sparse_fused_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out,
                                    float* lse, int B, int H, int S, int d, float scale, float beta, int block_q,
                                    int block_k, void* workspace, size_t workspace_bytes, int32_t* sel_idx,
                                    int32_t* sel_cnt, float* stats, float* taylor_t, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_sparse_fused_fwd");
  SparseArgs a{q, k, v, B, H, S, d, block_q, block_k, scale};
  attn_status_t st = sparse_common_checks(a);
  if (st != ATTN_OK) return st;
  if (!out || !aligned16(out) || (lse && ((uintptr_t)lse & 3u)) || bad_opt_ptrs(sel_idx, sel_cnt, stats, taylor_t))
    return ATTN_ERR_INVALID_ARG;
  if (isnan(beta) || beta == INFINITY) return ATTN_ERR_INVALID_ARG;
  const int NQB = (S + block_q - 1) / block_q, NKB = (S + block_k - 1) / block_k;
  if (NKB > kFusedMaxNKB) return ATTN_ERR_UNSUPPORTED;
  SparseLayout L;
  if (!sparse_layout(B, H, S, d, block_q, block_k, &L)) return ATTN_ERR_UNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.total) return ATTN_ERR_WORKSPACE;
  int* status = nullptr;
  if ((st = status_ptr(&status)) != ATTN_OK) return st;
  uint8_t* ws = (uint8_t*)workspace;
  float* qp = (float*)(ws + L.qp);
  float* kp = (float*)(ws + L.kp);
  float* vp = (float*)(ws + L.vp);
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, q, d, S, BH, 128)) != ATTN_OK) return st;
  if ((st = make_map(&tk, k, d, S, BH, block_k)) != ATTN_OK) return st;
  if ((st = make_map(&tv, v, d, S, BH, block_k)) != ATTN_OK) return st;
  if (launch_pool(q, k, v, qp, kp, vp, 3, BH, S, d, block_q, PoolSplit{}, status, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  FwdParams p = base_params(B, H, S, S, scale, kModeSparseFused, status);
  p.out = out;
  p.lse = lse;
  p.NQB = NQB;
  p.NKB = NKB;
  p.qbar = qp;
  p.kbar = kp;
  p.vbar = vp;
  p.scale = scale;
  p.beta = beta;
  p.block_k = block_k;
  p.out_sel_idx = sel_idx;
  p.out_sel_cnt = sel_cnt;
  p.out_stats = stats;
  p.out_taylor = taylor_t;
  return cuda_status(launch_fwd(d, block_k, kModeSparseFused, tq, tk, tv, p, stream));
}

// ---------------------------------------------------------------- allocation-free variant
// Scratch of attn_sparse_route_fwd_noalloc for callers that cannot allocate
// device memory themselves (see attn_api.h).  It lives in the library's
// module on each device and is shared by every call on that device.
static __device__ __align__(256) uint8_t g_noalloc_workspace[ATTN_NOALLOC_WORKSPACE_BYTES];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Host code cannot use g_noalloc_workspace's name as a device address; look
// the address up once per device, with that device current.
attn_status_t noalloc_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_OK;
}
}  // namespace

attn_status_t attn_sparse_route_fwd_noalloc(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v,
                                            attn_bf16* out, float* lse, int B, int H, int S, int d, float scale,
                                            float beta, int block_q, int block_k, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_sparse_route_fwd_noalloc");
  const size_t need = attn_sparse_workspace_bytes(B, H, S, d, block_q, block_k);
  if (need > ATTN_NOALLOC_WORKSPACE_BYTES) return ATTN_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    attn_status_t st = noalloc_workspace(&ws);
    if (st != ATTN_OK) return st;
  }
  // need == 0 means unsupported sizes: the checks below report them without launching
  return attn_sparse_route_fwd(q, k, v, out, lse, B, H, S, d, scale, beta, block_q, block_k, ws,
                               ATTN_NOALLOC_WORKSPACE_BYTES, nullptr, nullptr, nullptr, nullptr, stream);
}

attn_status_t attn_last_device_status(cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_last_device_status");
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (word & ATTN_DEVICE_TIMEOUT) return ATTN_ERR_TIMEOUT;
  if (word & (ATTN_DEVICE_BAD_LIST | ATTN_DEVICE_OOB)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status_t attn_selftest_wait_timeout(int limit_us, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_selftest_wait_timeout");
  if (limit_us < 1 || limit_us > 1000000) return ATTN_ERR_INVALID_ARG;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  return cuda_status(launch_wait_selftest(limit_us, 1, 0, status, next_launch_id(), stream));
}

attn_status_t attn_selftest_wait_timeout_grid(int limit_us, int n_ctas, cudaStream_t stream) {
  const NvtxRange nvtx_range("attn_selftest_wait_timeout_grid");
  if (limit_us < 1 || limit_us > 1000000 || n_ctas < 1 || n_ctas > 65536) return ATTN_ERR_INVALID_ARG;
  int* status = nullptr;
  attn_status_t st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  // 160 KB of shared memory per CTA: one CTA per SM, so the grid runs in waves
  return cuda_status(launch_wait_selftest(limit_us, n_ctas, 160 * 1024, status, next_launch_id(), stream));
}

}  // extern "C"
