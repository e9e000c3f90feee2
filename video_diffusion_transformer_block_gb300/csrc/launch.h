// Internal host-side launchers shared by the C ABI translation unit.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_fwd.cuh"

namespace vdtb {

// Optional tf32 hi / lo copies the pool kernel writes for the tensor-core
// routing: pooled keys [BH][NB][D] (kh, kl) and transposed pooled values
// [BH][D][NBp] (vth, vtl; NBp = NB rounded up to a multiple of 4).  Null
// pointers: not written.
struct PoolSplit {
  float* kh = nullptr;
  float* kl = nullptr;
  float* vth = nullptr;
  float* vtl = nullptr;
  int NBp = 0;
};

// Block mean-pool of `ntensors` (1..3) bf16 tensors [BH][S][D] into fp32 [BH][NB][D].
cudaError_t launch_pool(const uint16_t* x0, const uint16_t* x1, const uint16_t* x2, float* p0, float* p1, float* p2,
                        int ntensors, int BH, int S, int D, int block, const PoolSplit& split, int* status,
                        cudaStream_t stream);

// Sol-Attn routing (route_tc.cu): on the tensor cores, one CTA per head and 128
// query blocks, and a short last tile of up to 32 blocks per head on the CUDA
// cores beside it.  tkh / tkl: 3-D fp32 maps of the pooled keys' hi / lo (dims
// D, NKB, BH; box 32 x 128); tvh / tvl: of the transposed pooled values' hi /
// lo (dims NKB, D, BH; box 32 x D); tq: of the pooled queries [BH][NQB][D]
// (dims D, NQB, BH; box 32 x 128); qp / kp / vp: the pooled tensors in fp32.
cudaError_t launch_route_tc(const CUtensorMap& tkh, const CUtensorMap& tkl, const CUtensorMap& tvh,
                            const CUtensorMap& tvl, const CUtensorMap& tq, const float* qp, const float* kp,
                            const float* vp, int BH, int NQB, int NKB, int S, int D, int block_k, float scale,
                            float beta, int32_t* sel_idx, int32_t* sel_cnt, float* stats, float* taylor_t, int* status,
                            unsigned launch_id, cudaStream_t stream);

// Query-block order for the sparse forward (FwdParams::qb_order): per head and
// chunk of 128 query blocks, the blocks sorted by sel_cnt, longest first, into
// order [BH][NQB] (NKB < 2^23).
cudaError_t launch_qb_order(const int32_t* sel_cnt, int32_t* order, int BH, int NQB, int NKB, cudaStream_t stream);

// Exact log-sum-exp merge of n partials, rows = B*H*Sq.
cudaError_t launch_merge(const float* o_part, const float* lse_part, uint16_t* out, float* lse, int n, long long rows,
                         int D, int* status, cudaStream_t stream);

// tcgen05 attention forward.  mode: kModeDense / kModeSparse / kModeSplit.
cudaError_t launch_attn_fwd_d64(int BK, int mode, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, cudaStream_t stream);
cudaError_t launch_attn_fwd_d128(int BK, int mode, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const FwdParams& p, cudaStream_t stream);

// The persistent neighbourhood kernel (na_persist.cuh), mode kModeNA* (the
// query brick) and keys kNAKeysBrick / kNAKeysWide / kNAKeysWideF8 (the key
// box and the window operands' type; the wide boxes with the 4 x 4 x 8 brick
// only): tq, tk, tv are 5-D maps (channels, x, y, t, head) of q, k, v with a
// box of 64 channels and the brick's (tq) or the key box's (tk, tv) shape; the
// grid is one CTA per SM at most.
cudaError_t launch_na_persist_d64(int mode, int keys, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_na_persist_d128(int mode, int keys, const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream);

// Query tiles of 128 rows per CTA for a mode (the grid is BH * ceil(Sq / (128 * tiles)) [* n_split]).
// Dense and sparse CTAs take two tiles, each with its own list walk, K/V ring,
// TMA producer and MMA issuer, and one CTA per SM; the issuers take turns on
// the tensor pipe (see attn_fwd.cuh).  Split CTAs take one tile and run two per
// SM.  The fused-routing CTA routes two tiles' query blocks together and keeps
// two tiles.
inline int fwd_query_tiles(int mode) {
  return (mode == kModeSparseFused || mode == kModeDense || mode == kModeSparse) ? 2 : 1;
}

// Largest key-block count the fused (on-chip routing) forward accepts.
constexpr int kFusedMaxNKB = 1024;

// Per-row E4M3 quantisation of x [M][K] bf16 (K % 8 == 0): codes q [M][K], scale [M].
cudaError_t launch_fp8_quantize_rows(const uint16_t* x, uint8_t* q, float* scale, int M, int K, int* status,
                                     cudaStream_t stream);

// y [M][N] bf16 = diag(sa) (Aq Wq^T) diag(sw); ta / tb: 2-D uint8 maps of Aq [M][K]
// (box 128 x 128) and Wq [N][K] (box 128 x 256), 128-byte swizzle.
cudaError_t launch_fp8_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const float* sa, const float* sw,
                            uint16_t* y, int M, int N, int K, int* status, unsigned launch_id,
                            cudaStream_t stream);

// Bounded-wait self-test: n_ctas CTAs (each with `smem_bytes` of dynamic shared
// memory, which limits how many share an SM) wait on barriers nothing arrives on.
cudaError_t launch_wait_selftest(int limit_us, int n_ctas, int smem_bytes, int* status, unsigned launch_id,
                                 cudaStream_t stream);

}  // namespace vdtb
