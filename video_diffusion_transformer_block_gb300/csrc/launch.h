// Internal host-side launchers shared by the C ABI translation unit.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_fwd.cuh"

namespace vdtb {

// Block mean-pool of `ntensors` (1..3) bf16 tensors [BH][S][D] into fp32 [BH][NB][D].
cudaError_t launch_pool(const uint16_t* x0, const uint16_t* x1, const uint16_t* x2, float* p0, float* p1, float* p2,
                        int ntensors, int BH, int S, int D, int block, cudaStream_t stream);

// Sol-Attn routing from pooled tensors (one CTA per head and 32 query blocks).
cudaError_t launch_route(const float* qp, const float* kp, const float* vp, int BH, int NQB, int NKB, int S, int D,
                         int block_k, float scale, float beta, int32_t* sel_idx, int32_t* sel_cnt, float* stats,
                         float* taylor_t, cudaStream_t stream);

// Exact log-sum-exp merge of n partials, rows = B*H*Sq.
cudaError_t launch_merge(const float* o_part, const float* lse_part, uint16_t* out, float* lse, int n, long long rows,
                         int D, cudaStream_t stream);

// tcgen05 attention forward.  mode: kModeDense / kModeSparse / kModeSplit.
cudaError_t launch_attn_fwd_d64(int BK, int mode, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, cudaStream_t stream);
cudaError_t launch_attn_fwd_d128(int BK, int mode, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const FwdParams& p, cudaStream_t stream);

// Query tiles of 128 rows per CTA for a mode (the grid is BH * ceil(Sq / (128 * tiles)) [* n_split]).
inline int fwd_query_tiles(int mode) { return mode == kModeSplit ? 1 : 2; }

// Largest key-block count the fused (on-chip routing) forward accepts.
constexpr int kFusedMaxNKB = 1024;

// Bounded-wait self-test kernel.
cudaError_t launch_wait_selftest(int limit_us, int* status, cudaStream_t stream);

}  // namespace vdtb
