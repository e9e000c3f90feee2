/*
 * attn_api.h -- C ABI of the GB300 (sm_103a) attention hot path of an
 * LTX-2.5-style video+audio diffusion transformer block.
 *
 * Three operations, each a hand-written CUDA kernel path:
 *   - dense bf16 softmax attention over long video token sequences;
 *   - audio->video cross attention as split-KV partial answers plus an exact
 *     log-sum-exp merge;
 *   - Sol-Attn-style training-free block-sparse attention (pool, route,
 *     block-sparse forward with a Taylor term for rejected blocks).
 *
 * Conventions shared by every entry point
 *   Layout      q, k, v and out are [B][H][S][d] row-major (d innermost,
 *               contiguous), bf16 passed as raw 16-bit patterns (attn_bf16).
 *               d is 64 or 128.  Every device pointer must be 16-byte aligned.
 *   Ownership   All pointers are device pointers owned by the caller.  The
 *               library never allocates or frees device memory and keeps no
 *               pointer past the call.  Its only state is one device status
 *               word per device (see attn_last_device_status).
 *   Streams     Every call is asynchronous on `stream` (0 = legacy default
 *               stream) and does not synchronise the host, except
 *               attn_last_device_status.
 *   Errors      Arguments are validated on the host before anything is
 *               launched; an invalid call returns an error and launches
 *               nothing.  A launch failure returns ATTN_ERR_CUDA.  A device
 *               barrier wait that exceeds its time limit (about 2 s) makes
 *               the kernel return early and sets the device status word,
 *               which attn_last_device_status reports as ATTN_ERR_TIMEOUT.
 *               No exception or process exit crosses this ABI.
 *   Lengths     There are no masks: ragged and odd lengths (S not a multiple
 *               of any tile, odd key counts) are handled by in-kernel bounds;
 *               an odd key count is split unevenly rather than padded, as on
 *               the LTX-2.5 page ("LTX-2.5 at 4K, in half the time", section
 *               "Attention across two GPUs").
 *   Numerics    bf16 inputs, fp32 accumulation and softmax, bf16 outputs
 *               rounded to nearest even, lse in natural log (fp32).  The
 *               softmax scale must be finite and positive.
 */
#ifndef ATTN_API_H
#define ATTN_API_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t attn_bf16; /* raw bf16 bit pattern */

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or value */
  ATTN_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement (d, block, length limits) */
  ATTN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than attn_sparse_workspace_bytes() */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
  ATTN_ERR_TIMEOUT = 5      /* a device barrier wait ran out (reported by attn_last_device_status) */
} attn_status_t;

/*
 * Dense attention  O = softmax(scale * Q K^T) V, non-causal, and
 * lse = log sum_k exp(scale * q.k) per query row.
 *   q    [B][H][Sq][d]  bf16      k, v  [B][H][Skv][d]  bf16
 *   out  [B][H][Sq][d]  bf16      lse   [B][H][Sq]      fp32 (nullable)
 * Requires B, H, Sq, Skv >= 1, d in {64, 128}, scale finite and > 0.
 * Source: "Accelerating LTX-2.5 with Sol Engine", section "Stage 2
 * Optimization" (attention over long video sequences dominates Stage 2);
 * "Optimization" (openltx.com, hardware benchmarks), attention-backend paragraph.
 */
attn_status_t attn_dense_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out, float* lse,
                             int B, int H, int Sq, int Skv, int d, float scale, cudaStream_t stream);

/*
 * Split-KV partial answers for few-query cross attention (on the order of a
 * hundred audio queries over 10^4 - 10^5 video keys).  Chunk c of
 * n_split covers keys [floor(c*Skv/n_split), floor((c+1)*Skv/n_split)):
 * balanced bounds, nothing padded.  For each chunk and query row the kernel
 * writes the chunk-normalised output and the chunk's log-sum-exp:
 *   out_part [n_split][B][H][Sq][d] fp32,  lse_part [n_split][B][H][Sq] fp32.
 * An empty chunk (possible only when n_split > Skv, which is rejected) would
 * be o = 0, lse = -inf.  Requires 1 <= n_split <= Skv.
 * Source: "LTX-2.5 at 4K, in half the time", section "Attention across two
 * GPUs" (answers computed over separate slices of the keys keep, per row, the
 * maximum and the exponential sum that make combining them exact; this kernel
 * cuts the keys into such slices on one GPU).
 */
attn_status_t attn_cross_splitkv_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* out_part,
                                     float* lse_part, int B, int H, int Sq, int Skv, int d, int n_split, float scale,
                                     cudaStream_t stream);

/*
 * Exact log-sum-exp merge of n_split partial answers:
 *   L = log sum_c exp(lse_c),  o = sum_c exp(lse_c - L) o_c.
 *   out_part [n_split][B][H][Sq][d] fp32, lse_part [n_split][B][H][Sq] fp32
 *   out [B][H][Sq][d] bf16, lse [B][H][Sq] fp32 (nullable).
 * A row whose partials are all empty (lse = -inf) gets o = 0, lse = -inf.
 * Source: "LTX-2.5 at 4K, in half the time", section "Attention across two
 * GPUs" (partial answers are merged exactly).
 */
attn_status_t attn_lse_merge(const float* out_part, const float* lse_part, attn_bf16* out, float* lse, int n_split,
                             int B, int H, int Sq, int d, cudaStream_t stream);

/*
 * Block mean-pool along the sequence: x_pool[b][h][i] = mean of x[b][h][t]
 * over the tokens t of block i = [i*block, min((i+1)*block, S)).
 *   x [B][H][S][d] bf16  ->  x_pool [B][H][ceil(S/block)][d] fp32.
 * block in {64, 128}.
 * Source: "Accelerating LTX-2.5 with Sol Engine", section "Stage 2
 * Optimization", bullet "On-the-fly routing" (pooled keys).
 */
attn_status_t attn_block_pool(const attn_bf16* x, float* x_pool, int B, int H, int S, int d, int block,
                              cudaStream_t stream);

/*
 * Bytes of device workspace attn_sparse_route_fwd needs for these sizes
 * (pooled Q/K/V, selected-block lists, per-block statistics, Taylor
 * aggregates, and the tf32 hi/lo halves of the pooled keys and of the
 * transposed pooled values that the tensor-core routing multiplies).
 * Returns 0 for sizes the library does not support.
 */
size_t attn_sparse_workspace_bytes(int B, int H, int S, int d, int block_q, int block_k);

/*
 * Sol-Attn block-sparse self-attention (Sq = Skv = S).
 * Source: "Accelerating LTX-2.5 with Sol Engine", section "Stage 2
 * Optimization - Core Technology: Sol-Attn", bullets "Query-dependent
 * thresholding", "On-the-fly routing" and "Proxy-score reuse".
 *
 * With NQB = ceil(S/block_q), NKB = ceil(S/block_k), Qbar/Kbar/Vbar the block
 * means (attn_block_pool), per head and query block i:
 *   s_ij  = scale * Qbar_i . Kbar_j                  (block proxy score)
 *   mu_i, sigma_i = mean and population std of s_ij over j
 *   tau_i = mu_i + beta * sigma_i                    (beta = -INFINITY keeps every block)
 *   Sel_i = { j : s_ij >= tau_i } plus the argmax block (lowest j on ties)
 *   for rejected j: w_ij = n_j * max(0, 1 + s_ij - mu_i)   (n_j = keys in block j)
 *   W_i = sum w_ij,  T_i = sum w_ij Vbar_j
 * and for each query row q of block i, over the keys of the selected blocks,
 *   M = max scale*q.k,  num = sum e^(x-M) v + e^(mu_i-M) T_i,
 *   den = sum e^(x-M) + e^(mu_i-M) W_i,  out = num/den,  lse = M + ln den.
 * (When Sel_i is every block the Taylor terms are skipped.)
 * The proxy scores and T are computed on the tensor cores with fp32-grade
 * accuracy (three tf32 products of hi/lo operand halves); the proxy scores
 * live in tensor memory, are recomputed for the selection pass, and are never
 * written to memory.
 *
 *   q, k, v, out [B][H][S][d] bf16,  lse [B][H][S] fp32 (nullable)
 *   block_q == block_k, in {64, 128}
 *   workspace  device buffer of at least attn_sparse_workspace_bytes(...)
 *              bytes, 256-byte aligned, contents ignored on entry
 *   sel_idx    [B][H][NQB][NKB] int32 (nullable): the first sel_cnt entries of
 *              each row are the selected key blocks in ascending order; the
 *              rest are left unspecified
 *   sel_cnt    [B][H][NQB] int32 (nullable)
 *   stats      [B][H][NQB][4] fp32 (nullable): mu, sigma, tau, W
 *   taylor_t   [B][H][NQB][d] fp32 (nullable): T
 * Null outputs are kept inside the workspace.  S is limited to NKB <= 8192.
 * With 128-token blocks the workspace also holds the query-block order
 * (attn_sparse_route's qb_order) the forward pairs its query tiles by.
 */
attn_status_t attn_sparse_route_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out,
                                    float* lse, int B, int H, int S, int d, float scale, float beta, int block_q,
                                    int block_k, void* workspace, size_t workspace_bytes, int32_t* sel_idx,
                                    int32_t* sel_cnt, float* stats, float* taylor_t, cudaStream_t stream);

/*
 * Routing half of attn_sparse_route_fwd: block mean-pool of Q, K, V and the
 * Sol-Attn selection with its Taylor aggregates (same definitions as
 * attn_sparse_route_fwd).  Here sel_idx, sel_cnt, stats and taylor_t are
 * required (non-null); the workspace holds the pooled tensors.
 *   qb_order   [B][H][NQB] int32 (nullable; 128-token blocks only, else
 *              ATTN_ERR_INVALID_ARG): per head, within each run of 128
 *              consecutive query blocks, the blocks sorted by sel_cnt,
 *              longest list first (ties: lower index first).  The forward
 *              runs the blocks in places 2s and 2s + 1 of this order on one
 *              CTA, whose time is that of the longer list, so neighbours of
 *              nearly equal length waste little; any order gives the same
 *              results bit for bit.
 */
attn_status_t attn_sparse_route(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, int B, int H, int S,
                                int d, float scale, float beta, int block_q, int block_k, void* workspace,
                                size_t workspace_bytes, int32_t* sel_idx, int32_t* sel_cnt, float* stats,
                                float* taylor_t, int32_t* qb_order, cudaStream_t stream);

/*
 * Forward half of attn_sparse_route_fwd: block-sparse attention with the
 * Taylor term, given a routing in the layout attn_sparse_route writes
 * (sel_idx/sel_cnt ascending lists, stats[..][0] = mu, stats[..][3] = W,
 * taylor_t = T).  Lets a caller reuse one routing for several calls.  A list
 * entry outside [0, NKB) is clamped and reported by attn_last_device_status
 * as ATTN_ERR_INVALID_ARG; so is an empty list (sel_cnt 0), whose query rows
 * are written as zeros with lse -inf.  qb_order (nullable; 128-token blocks
 * only): the order attn_sparse_route writes, i.e. per head a permutation of
 * the query blocks; null pairs blocks 2s and 2s + 1.  An entry outside
 * [0, NQB) is clamped and reported like a bad list entry; an order that is not
 * a permutation leaves some query rows unwritten.
 */
attn_status_t attn_sparse_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out, float* lse,
                              int B, int H, int S, int d, float scale, int block_q, int block_k,
                              const int32_t* sel_idx, const int32_t* sel_cnt, const float* stats,
                              const float* taylor_t, const int32_t* qb_order, cudaStream_t stream);

/*
 * attn_sparse_route_fwd with the routing folded into the forward kernel: after
 * the block mean-pool, each CTA of the forward computes the proxy scores of
 * its own query blocks against every pooled key block, their mean, standard
 * deviation and threshold, the compacted selection and the Taylor aggregates
 * in shared memory, and then runs the block-sparse main loop over those
 * on-chip lists.  No routing launch, and neither the proxy map nor the lists
 * are written to memory (unless the optional outputs are given).
 * Source: "Accelerating LTX-2.5 with Sol Engine", section "Stage 2
 * Optimization - Core Technology: Sol-Attn" (block selection folded into the
 * online-softmax pass, no separate routing stage, no proxy map).
 *   Arguments, definitions and optional outputs as attn_sparse_route_fwd;
 *   the workspace (attn_sparse_workspace_bytes) holds the pooled tensors.
 *   Limit: NKB = ceil(S/block_k) <= 1024 (ATTN_ERR_UNSUPPORTED beyond).
 */
attn_status_t attn_sparse_fused_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out,
                                    float* lse, int B, int H, int S, int d, float scale, float beta, int block_q,
                                    int block_k, void* workspace, size_t workspace_bytes, int32_t* sel_idx,
                                    int32_t* sel_cnt, float* stats, float* taylor_t, cudaStream_t stream);

/*
 * Split-KV cross attention with the merge fused into the split kernel's tail.
 * ("LTX-2.5 at 4K, in half the time", section "Attention across two GPUs":
 * partial answers over slices of the keys, merged exactly.)
 *
 *   Computes what attn_cross_splitkv_fwd followed by attn_lse_merge computes,
 *   in one launch: the CTA of the last key chunk to finish for a (head, 128-row
 *   query tile) merges that tile's partials (same arithmetic as
 *   attn_lse_merge, so the results are identical to the two-call path).
 *   q, k, v, out, lse   as attn_dense_fwd (lse nullable); Sq >= 1, Skv >= 1.
 *   n_split             1 <= n_split <= Skv, balanced unpadded chunks; at most
 *                       32 (ATTN_ERR_UNSUPPORTED beyond: use the two calls).
 *   workspace           device, 16-byte aligned, >= attn_cross_workspace_bytes
 *                       bytes: the partials and one arrival counter per
 *                       (head, query tile).  The counters must be zero before
 *                       the first call on a workspace (e.g. a zero-filled
 *                       allocation); every call leaves them at zero.  After a
 *                       call that ended in ATTN_ERR_TIMEOUT, zero the
 *                       workspace again before reusing it.
 *   Errors: ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED (d), ATTN_ERR_WORKSPACE
 *   (too small), ATTN_ERR_CUDA.  Asynchronous on stream; calls sharing a
 *   workspace must be ordered (same stream).
 */
size_t attn_cross_workspace_bytes(int B, int H, int Sq, int d, int n_split);
attn_status_t attn_cross_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out, float* lse,
                             int B, int H, int Sq, int Skv, int d, int n_split, float scale, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * 3D neighbourhood attention over a (T, Y, X) token volume.
 * ("LTX-2.5 at 4K, in half the time", section "Inside the decoder": the video
 * decoder's time goes mostly to a neighbourhood-attention kernel; "Optimization
 * Tips", section "Diffusion VAE Decoder": the decoder's neighbourhood-attention
 * backends.  The window follows the published neighbourhood-attention
 * definition, which the pages do not restate.)
 *
 *   For the query at (t, y, x) the keys are the Kt x Ky x Kx tokens whose
 *   coordinate on each axis lies in [s, s + K) with s = clamp(p - floor(K/2),
 *   0, L - K): the window is centred on the query and moved inward at the
 *   borders, so every query sees exactly Kt*Ky*Kx keys, itself included.
 *   Over them: O = softmax(scale * q k^T) V, lse = log of the denominator
 *   (natural log, including the max).  Non-causal, dilation 1.
 *
 *   q, k, v, out  bf16 [B][H][S][d], S = T*Y*X tokens in raster order
 *                 (t, y, x), x fastest; 16-byte aligned; d in {64, 128}.
 *   lse           nullable, fp32 [B][H][S].
 *   Kt, Ky, Kx    window per axis, 1 <= K <= L (T, Y, X).
 *   scale         softmax scale, finite and > 0.
 *   brick         query/key tile shape, frames x rows x columns of 128 tokens:
 *                 1 = 1x8x16, 2 = 2x8x8, 3 = 4x4x8, 0 = chosen by the library.
 *   pair_axis     the CTA layout: 0 / 1 / 2 = a CTA takes two query bricks
 *                 that are neighbours along frames / rows / columns (one walk
 *                 of the union of their windows); 3 = one brick per CTA, two
 *                 CTAs per SM; 4 = persistent CTAs, one per SM, whose two
 *                 query tiles each run a sequence of bricks (one brick's
 *                 epilogue overlaps the other tile's MMAs) and whose tensor
 *                 cores add the window to the scores (0 inside, -2^120
 *                 outside; for scale * log2(e) < 2^-80, where that would not
 *                 vanish in the exponent, plan 3 runs instead, with the same
 *                 results); 5 = plan 4 with key boxes of 4x2x16 tokens instead
 *                 of the brick's shape (brick 3, i.e. 4x4x8 queries, only),
 *                 which cover a brick's window union with fewer boxes under
 *                 small windows (3x7x7: 5 boxes per brick instead of 6); 6 =
 *                 plan 5 with the window's operands in E5M2 (-57344 outside
 *                 against one-hots of 57344: -49 * 2^26 per missed axis), half
 *                 the shared memory of plan 5's bf16 ones, so each tile keeps
 *                 two window buffers at d = 128; it gives plan 5's results
 *                 bit for bit when every raw score |q.k| < 2^30, and is not
 *                 exact beyond that, so the library never picks it (for
 *                 scale * log2(e) < 2^-22 plan 5 runs instead); -1 = chosen
 *                 by the library: plan 4 or 5, the fastest on GB300 for every
 *                 volume and window measured among the plans exact for all
 *                 inputs.  An open brick minimises a measured cost model of
 *                 key boxes and bricks (see attn_na3d_plan).
 *   The choice only changes speed, never results beyond fp32 rounding order
 *   (plan 6: within its score range).
 *   Errors: ATTN_ERR_INVALID_ARG (null or misaligned pointer, a window outside
 *   [1, L], S > 2^30, non-positive scale, bad brick/pair code (0..3 / -1..6),
 *   pair 5 or 6 with brick 1 or 2), ATTN_ERR_UNSUPPORTED (d), ATTN_ERR_CUDA
 *   (launch).  Asynchronous on stream.
 */
attn_status_t attn_na3d_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* out, float* lse,
                            int B, int H, int T, int Y, int X, int d, int Kt, int Ky, int Kx, float scale, int brick,
                            int pair_axis, cudaStream_t stream);

/*
 * The tile plan attn_na3d_fwd uses for a volume and window (at a scale with
 * scale * log2(e) >= 2^-80).  On entry *brick and *pair_axis hold the
 * caller's request (0 / -1 = open); on return the plan.  An open pair axis
 * takes plan 4 or (brick 3) plan 5 (plan 6 only when asked for, with brick 3
 * or an open brick), an open brick any brick; the choice
 * minimises, in twentieths of a key box, for plans 4 and 5: 20 per box of
 * plan 4 with a 4x4x8 brick and 23 per box otherwise (their window step is 32
 * columns wide) plus 34 per brick; for the other plans: 20 per box plus 40
 * per CTA.  *key_boxes (nullable) receives the number of 128-key boxes the
 * query tiles of one head multiply: the executed work of one head is
 * key_boxes * 4 * 128 * 128 * d floating-point operations (plans 4 and 5 add
 * one or two K = 16 steps per box for the window, plan 6 one K = 32 step of
 * 8-bit operands).  Host only.
 * ATTN_ERR_INVALID_ARG as for attn_na3d_fwd.
 */
attn_status_t attn_na3d_plan(int T, int Y, int X, int Kt, int Ky, int Kx, int* brick, int* pair_axis,
                             long long* key_boxes);

/*
 * Size of the library-owned device scratch used by
 * attn_sparse_route_fwd_noalloc (32 MiB on every device that loads the
 * library, held until the process exits).
 */
#define ATTN_NOALLOC_WORKSPACE_BYTES ((size_t)32 << 20)

/*
 * attn_sparse_route_fwd for callers that must not allocate device memory.
 * (No counterpart on the LTX-2.5 / Sol-Attn pages: this is a packaging
 * variant, not part of the method.)
 *
 * Some callers cannot provide the scratch buffer attn_sparse_route_fwd asks
 * for: code embedded in a host framework that owns every device allocation
 * (a fixed memory arena handed out by an inference server or a plug-in host),
 * or latency-critical threads where cudaMalloc may synchronise the device and
 * stall other work.  This entry point computes exactly what
 * attn_sparse_route_fwd computes, but keeps the pooled tensors and the
 * routing (selected-block lists, statistics, Taylor aggregates) in one
 * file-scope device array of ATTN_NOALLOC_WORKSPACE_BYTES owned by the
 * library.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   Arguments   as attn_sparse_route_fwd, without the workspace and the
 *               optional routing outputs.
 *   Limit       sizes whose attn_sparse_workspace_bytes(...) exceeds
 *               ATTN_NOALLOC_WORKSPACE_BYTES are rejected with
 *               ATTN_ERR_WORKSPACE before anything is launched (for H = 32,
 *               d = 128, block 128 that is S up to about 27K tokens).
 *   Set-up      the first call on a device looks up the device address of
 *               the array (once per device, with that device current); make
 *               that first call before any stream capture.
 *   Sharing     every call on a device uses the same array and leaves its
 *               contents behind; nothing in it has to start at zero (every
 *               byte a call reads was written earlier in the same call), but
 *               calls that overlap on the GPU (different streams, or
 *               different host threads without ordering) race on it and must
 *               be serialised by the caller.
 */
attn_status_t attn_sparse_route_fwd_noalloc(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v,
                                            attn_bf16* out, float* lse, int B, int H, int S, int d, float scale,
                                            float beta, int block_q, int block_k, cudaStream_t stream);

/*
 * Synchronises `stream`, reads and clears the current device's status word.
 * Returns ATTN_OK, ATTN_ERR_TIMEOUT if a kernel gave up on a barrier wait
 * (every wait has a 2 s limit; once one wait of a launch gives up, the rest
 * of that launch's CTAs stop waiting and return, so the launch ends soon
 * after), ATTN_ERR_INVALID_ARG if a kernel met a corrupt selected-block list
 * or (bounds-checked build only) skipped a store outside its output buffer,
 * or ATTN_ERR_CUDA if the synchronisation itself failed.
 */
attn_status_t attn_last_device_status(cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* attn_status_string(attn_status_t status);

/*
 * Self-test of the bounded-wait path: launches one CTA that waits on a
 * barrier nothing ever arrives on, with a limit of `limit_us` microseconds
 * (1..1000000).  The kernel gives up, records the timeout in the status word
 * and exits, so a following attn_last_device_status returns
 * ATTN_ERR_TIMEOUT.  Leaves the context usable.
 */
attn_status_t attn_selftest_wait_timeout(int limit_us, cudaStream_t stream);

/*
 * Self-test of the launch-wide abort: launches `n_ctas` CTAs (1..65536), each
 * holding 160 KB of shared memory so that one runs per SM and the grid runs in
 * waves, and each waiting on a barrier nothing arrives on with a limit of
 * `limit_us` microseconds (1..1000000).  The first wait to give up records the
 * timeout and marks the launch aborted; the CTAs still waiting give up within
 * tens of microseconds and the CTAs that start afterwards return at once, so
 * the launch ends about one limit after it starts instead of one limit per
 * wave.  A following attn_last_device_status returns ATTN_ERR_TIMEOUT; the
 * context stays usable, and later launches are not affected.
 */
attn_status_t attn_selftest_wait_timeout_grid(int limit_us, int n_ctas, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_API_H */
