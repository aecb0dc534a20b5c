/*
 * moe.h — C ABI of the GB300 (sm_103a) routed-expert MoE forward.
 *
 * One shared library, libmoe_gb300.so, of hand-written CUDA kernels.  The
 * entry points are the stages of the single-GPU forward of
 * mslk/moe/layers.py, MetaShufflingMoE._no_comm_forward:
 *
 *   moe_router_scores         router scores sigmoid(tokens @ router_DE), bf16
 *   moe_router_route          ... with the top-k selection in the router's
 *                             epilogue, then the by-expert permutation
 *   moe_route                 top-k routing into per-expert counts and a
 *                             by-expert token permutation (index_shuffling)
 *   moe_gather_scale          gather token rows and multiply by the score
 *   moe_gather_scale_quant    ... and quantise each row to FP8 (e4m3)
 *   moe_grouped_gemm          per-expert GEMM with w13 or w2 (bf16)
 *   moe_grouped_gemm_fp8_rowwise   the same on e4m3 operands with row scales
 *   moe_dense_gemm            split-K dense GEMM (the shared expert of small batches)
 *   moe_silu_mul(_quant)      z = silu(y0) * y1 (and FP8 quantisation)
 *   moe_scatter_add           add routed rows back into token order
 *   moe_scatter_add_padded    the same for the padded-token layout (counts per expert)
 *   moe_topk_finalize         routing weights applied to the expert outputs
 *   moe_quantize_rows         per-row FP8 quantisation of a weight matrix
 *
 * Conventions (every entry point):
 *  - Pointers are DEVICE pointers unless stated; the caller owns all memory.
 *    No entry point allocates device memory; scratch comes from the caller
 *    (moe_route's workspace).
 *  - Matrices are row-major and contiguous unless a stride is given.
 *    bf16 = IEEE binary32 upper half; e4m3 = OCP FP8 E4M3 ("fn": no
 *    infinities, largest finite 448).
 *  - Every call is asynchronous on `stream` and never synchronises with the
 *    host.  Counts that the GPU computes (valid rows, per-expert counts) are
 *    read on the device.
 *  - Return value: MOE_OK, or a negative MOE_ERR_* code.  Argument errors are
 *    detected on the host before anything is launched.  Errors the GPU finds
 *    (an index out of range, a device count larger than its buffer, a wait
 *    that timed out) never fault: the kernel skips the offending work and
 *    records a MOE_DEVERR_* bit, read back with moe_device_error().
 *  - Identical inputs give identical output bytes (no atomics on data).
 *  - Alignment: every matrix base pointer is 16-byte aligned; D, H, N and K
 *    are multiples of 16.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define MOE_OK 0
#define MOE_ERR_INVALID (-1)     /* null required pointer, bad size, top_k outside [1, E] ... */
#define MOE_ERR_UNSUPPORTED (-2) /* alignment, a dimension not a multiple of 16, E > 1024 ... */
#define MOE_ERR_CUDA (-3)        /* a CUDA call failed: moe_last_cuda_error() has the code */
#define MOE_ERR_WORKSPACE (-4)   /* the workspace is smaller than moe_route_workspace_size() */

/* Element types. */
#define MOE_DTYPE_BF16 0
#define MOE_DTYPE_F32 1
#define MOE_DTYPE_E4M3 2

/* Grouped-GEMM epilogues. */
#define MOE_EPILOGUE_NONE 0     /* y[r, n] = (x_r . w_e[n]) (times the two scales for FP8), bf16 */
#define MOE_EPILOGUE_SILU_MUL 1 /* with N = 2H: y[r, j] = silu(v_j) * v_{H+j}, j < H, bf16 */
#define MOE_EPILOGUE_SILU_MUL_QUANT 2 /* SILU_MUL, then each row of y quantised to e4m3 (z_out, z_scale) */
/* OR-ed into `epilogue` of the grouped GEMMs: compute 256-row x 256-column tiles on
 * pairs of SMs (a 2-CTA cluster, tcgen05 cta_group::2).  Same results; faster when
 * experts hold many rows; an expert whose rows end mid-tile still pays for the
 * whole 256-row tile. */
#define MOE_GEMM_CTA_PAIRS 0x100
/* OR-ed into `epilogue` of the grouped GEMMs (and passed in `flags` of
 * moe_expert_mlp): w points to weights in the tile-packed layout of
 * moe_pack_weights instead of row-major [E, N, K].  Same results; the weights
 * stream from HBM as contiguous 16 KB boxes instead of 128-byte pieces of 128
 * rows (decode expert MLP: 602 -> 564 us).  Needs N % 128 == 0 (and (N / 2) % 128
 * with MOE_EPILOGUE_SILU_MUL). */
#define MOE_WEIGHTS_PACKED 0x200

/* Device-side error bits (moe_device_error). */
#define MOE_DEVERR_BAD_INDEX 0x1   /* a token or expert index outside its range was skipped */
#define MOE_DEVERR_BAD_COUNT 0x2   /* a device count exceeded its buffer and was clamped */
#define MOE_DEVERR_TIMEOUT 0x4     /* a bounded pipeline wait gave up; the tile was abandoned */

/* Text for a status code (static storage). */
const char* moe_status_string(int status);

/* The cudaError_t of the last MOE_ERR_CUDA returned on this host thread. */
int moe_last_cuda_error(void);

/*
 * Read and clear the device-side error word of the current device.
 * Synchronises `stream`.  *bits receives an OR of MOE_DEVERR_* (0 = none).
 */
int moe_device_error(unsigned int* bits, cudaStream_t stream);

/* ------------------------------------------------------------ router scores */

/*
 * Bytes of device workspace moe_router_scores needs (host call, no GPU use).
 */
int moe_router_workspace_size(int T, int D, int E, size_t* bytes);

/*
 * Router scores of mslk/moe/layers.py, MetaShufflingMoE._route (the same two
 * steps open BaselineMoE._forward): scores = sigmoid(linear(tokens,
 * router_DE.T)), both steps in bf16.  For every token t < Tv and expert e:
 *   logit        = bf16( sum_d x[t, d] * w_router[e, d] )   fp32 accumulation
 *   scores[t, e] = bf16( 1 / (1 + exp(-logit)) )            fp32
 *
 * x                bf16 [T, D], row-major, 16-byte aligned.
 * w_router         bf16 [E, D], row-major, 16-byte aligned: router_DE [D, E]
 *                  transposed (the caller keeps this copy resident).
 * num_valid_tokens device int32 scalar Tv, or NULL for T.  A value outside
 *                  [0, T] is clamped and flagged (MOE_DEVERR_BAD_COUNT).
 * scores           bf16 [T, E], row-major (row stride E).  Rows t >= Tv are
 *                  not written.  Pass it to moe_route with stride_t = E,
 *                  stride_e = 1.
 * ws, ws_bytes     device workspace of at least moe_router_workspace_size
 *                  bytes, 256-byte aligned, owned by the caller (NULL when that
 *                  size is 0, as it is in this build).  Too small:
 *                  MOE_ERR_WORKSPACE.
 *
 * Supports 1 <= E <= 256 and D a positive multiple of 16
 * (MOE_ERR_UNSUPPORTED otherwise).  T = 0 is a no-op.  The sum over d may be
 * split across the CTAs of a cluster; the partial sums are always added in the
 * same order, so identical inputs on the same device give identical bytes.
 */
int moe_router_scores(const void* x, int T, int D, const void* w_router, int E,
                      const int32_t* num_valid_tokens, void* scores, void* ws, size_t ws_bytes,
                      cudaStream_t stream);

/* ------------------------------------------------------------- diagnostics */

/*
 * Exercises one of the library's bounded device-side waits against a
 * condition that never comes true, so that a caller (or a test) can see the
 * failure path work without a GPU fault: which = 0 waits on an mbarrier phase
 * that no one completes (the wait of every TMA/tensor-core pipeline here);
 * which = 1 runs a cooperative grid whose last block skips the grid barrier
 * (the barrier of the cooperative routing kernel).  The wait gives up after
 * limit_ns (1 us .. 2 s) of the device's global timer, records
 * MOE_DEVERR_TIMEOUT (read it with moe_device_error) and returns; the context
 * stays usable.  Returns MOE_ERR_INVALID for other arguments.
 */
int moe_selftest_bounded_wait(int which, int64_t limit_ns, cudaStream_t stream);

/* ------------------------------------------------------------------ routing */

/*
 * The router and the routing in two kernels: moe_router_scores with the top-k
 * selection of moe_route folded into its reduction epilogue (mslk/moe/layers.py,
 * MetaShufflingMoE._route: sigmoid(linear(tokens, router_DE.T)) followed by
 * index_shuffling).  The CTA that sums a 32-token chunk of router logits over
 * its thread-block cluster forms the chunk's bf16 scores, stores them, picks
 * each token's top_k experts and writes the chunk's expert histogram to the
 * workspace; one cooperative kernel then scans the histograms and emits the
 * routed rows (one grid barrier, against two after a separate moe_route).
 *
 * x, T, D, w_router, E, num_valid_tokens: as moe_router_scores (E <= 256).
 * scores: bf16 [T, E] (required): written exactly as moe_router_scores writes it.
 * counts, expert_offsets, expert_indices, token_indices, inv_rows (nullable),
 * topk_weights (nullable), top_k: as moe_route on those scores, bit for bit.
 * ws, ws_bytes: device workspace of moe_router_route_workspace_size bytes,
 * 256-byte aligned; its contents on entry do not matter.
 * T == 0 writes zero counts and offsets.  The result is deterministic.
 */
int moe_router_route_workspace_size(int T, int D, int E, int top_k, size_t* bytes);
int moe_router_route(const void* x, int T, int D, const void* w_router, int E, int top_k,
                     const int32_t* num_valid_tokens, void* scores, int32_t* counts,
                     int32_t* expert_offsets, int32_t* expert_indices, int32_t* token_indices,
                     int32_t* inv_rows, float* topk_weights, void* ws, size_t ws_bytes,
                     cudaStream_t stream);

/*
 * Bytes of device workspace moe_route needs for T token rows, E experts and
 * top_k (host call, no GPU use).
 */
int moe_route_workspace_size(int T, int E, int top_k, size_t* bytes);

/*
 * Top-k routing and the by-expert permutation: index_shuffling(scores) of
 * mslk/moe/layers.py (MetaShufflingMoE._route); the selection is torch.topk
 * as in BaselineMoE._forward.
 *
 * scores        [T, E] router scores, element (t, e) at
 *               scores + t * stride_t + e * stride_e (elements), dtype
 *               MOE_DTYPE_BF16 or MOE_DTYPE_F32.  NaN scores are undefined.
 * num_valid_tokens  device int32: tokens t < *num_valid_tokens are routed
 *               (NULL: all T).  A value outside [0, T] is clamped and flagged.
 * For each valid token the top_k experts with the largest scores are chosen,
 * equal scores (+0 == -0) going to the lower expert index.  The Tv * top_k
 * (token, expert) pairs are then numbered as routed rows in ascending expert
 * order and, within an expert, ascending token order.  Outputs (device int32):
 *   counts[E + 1]          rows per expert; counts[E] = Tv * top_k (the total,
 *                          which the pages slice off with token_counts[:E])
 *   expert_offsets[E + 1]  exclusive prefix sum of counts; [E] = Tv * top_k
 *   expert_indices[T * top_k], token_indices[T * top_k]
 *                          the pair of each routed row; entries at and past
 *                          Tv * top_k are not written
 *   inv_rows[T * top_k]    (nullable) inv_rows[t * top_k + j] = the j-th
 *                          smallest routed row of token t, for t < Tv
 * topk_weights  (nullable) device float [T * top_k]: topk_weights[t * top_k + j]
 *               = the score (as fp32) of the expert of routed row
 *               inv_rows[t * top_k + j], for t < Tv: the top-k values, in the
 *               order of inv_rows (what moe_topk_finalize takes).
 * ws, ws_bytes  device workspace of at least moe_route_workspace_size bytes,
 *               256-byte aligned; its contents on entry do not matter.
 * Requires 1 <= top_k <= E <= 1024 and T >= 0.  The result is deterministic.
 */
int moe_route(const void* scores, int scores_dtype, int64_t stride_t, int64_t stride_e, int T, int E,
              int top_k, const int32_t* num_valid_tokens, int32_t* counts, int32_t* expert_offsets,
              int32_t* expert_indices, int32_t* token_indices, int32_t* inv_rows,
              float* topk_weights, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * moe_route without a caller workspace: for callers that cannot allocate
 * device memory.  (The pages have no counterpart of this entry point.)
 *
 * Some callers may not call cudaMalloc or any other allocating routine where
 * they route tokens: a plugin inside a framework whose own allocator owns the
 * whole device-memory budget, a serving loop that cannot afford the implicit
 * device synchronisation and unbounded latency of an allocation, or code that
 * must not re-enter the allocator (for example inside an out-of-memory
 * handler).  They pass inputs and outputs exactly as for moe_route; the
 * workspace comes from a fixed array of MOE_ROUTE_NO_ALLOC_SCRATCH_BYTES that
 * the library keeps in global memory of every GPU that loads it, until the
 * process exits.  Nothing is allocated: no cudaMalloc, cudaFree or allocating
 * library routine is called.
 *
 * - Outputs: as moe_route without topk_weights (use moe_route for those).
 * - Sizes: returns MOE_ERR_WORKSPACE (and launches nothing) when
 *   moe_route_workspace_size(T, E, top_k) exceeds
 *   MOE_ROUTE_NO_ALLOC_SCRATCH_BYTES (1 MiB).  For example T = 16384,
 *   top_k = 4, E = 128 needs 0.5 MiB and fits; T = 65536, top_k = 1,
 *   E = 128 needs 1.25 MiB and is rejected.
 * - Set-up: the first call on each device (with that device current) looks up
 *   the array's device address (cudaGetSymbolAddress) and loads the routing
 *   kernels, and keeps the address.  CUDA loads a library's device code
 *   lazily, so that first call is when the driver places this array and the
 *   routing code in device memory: an allocation made by the driver, not by
 *   the caller, which an out-of-memory situation can make fail (MOE_ERR_CUDA).
 *   Make that first call at start-up, before the code that must not allocate
 *   and before any stream capture; a call with T = 0 (valid counts and
 *   expert_offsets pointers) does the set-up, writes zero counts and launches
 *   no routing kernel.  After the device's context changes (cudaDeviceReset)
 *   the next call sets up again.  A failed set-up returns MOE_ERR_CUDA with the
 *   code in moe_last_cuda_error().
 * - Sharing: every call on a device uses the same array and leaves its
 *   contents behind.  The routing kernels write every scratch word before
 *   reading it, except the grid-barrier counter of the large-batch kernel,
 *   which each call zeroes with an asynchronous memset on the stream before
 *   that kernel starts; so nothing needs clearing between calls.  Calls whose
 *   kernels overlap on the GPU (for example on two streams without ordering
 *   between them) race on the array and give wrong results: order them.
 * Arguments, outputs and results are those of moe_route.
 */
#define MOE_ROUTE_NO_ALLOC_SCRATCH_BYTES (1u << 20)
int moe_route_no_alloc(const void* scores, int scores_dtype, int64_t stride_t, int64_t stride_e, int T,
                       int E, int top_k, const int32_t* num_valid_tokens, int32_t* counts,
                       int32_t* expert_offsets, int32_t* expert_indices, int32_t* token_indices,
                       int32_t* inv_rows, cudaStream_t stream);

/* --------------------------------------------------------- gather + scale */

/*
 * gather_scale_dense_tokens (mslk/moe/gather_scatter.py,
 * _mslk_gather_scale_dense_tokens): for routed rows i < valid,
 *   out[i, :] = bf16( f32(x[t, :]) * f32(scores[t, e]) ),
 *   t = token_indices[i], e = expert_indices[i].
 * x [T, D] bf16; token_indices, expert_indices [a] int32; scores as in
 * moe_route (E experts), or NULL for unit scores (the rows are copied, as the
 * output-weighted path of moe_topk_finalize wants; this holds for the
 * quantising variant too); valid_token_count: device int32 count of ROUTED ROWS
 * (NULL: a), e.g. &counts[E] from moe_route.  Rows i >= valid are not written.
 * out [a, D] bf16.  a == 0 or D == 0 is a no-op.
 * inv_rows (nullable) and top_k: moe_route's inverse permutation.  With it
 * (and top_k > 1) the rows are produced token by token, each x row read from
 * HBM once for its top_k routed rows; valid_token_count must then be
 * Tv * top_k.  The output is the same either way.
 * Launch: with programmatic stream serialization, so the kernel may start
 * while the previous kernel in the stream (moe_route) still runs.  It waits for
 * that kernel to finish before reading anything, so stream order holds for
 * every input.
 */
int moe_gather_scale(const void* x, int T, int D, const int32_t* token_indices,
                     const int32_t* expert_indices, int a, const void* scores, int scores_dtype,
                     int64_t stride_t, int64_t stride_e, int E, const int32_t* valid_token_count,
                     const int32_t* inv_rows, int top_k, void* out, cudaStream_t stream);

/*
 * gather_scale_quant_dense_tokens (mslk/moe/gather_scatter.py,
 * _mslk_gather_scale_fp8_rowwise_quant_dense_tokens): the fp32 row
 * v = x[t, :] * scores[t, e] is quantised to e4m3 with one fp32 scale:
 *   m = max |v|, then m = min(max(m, 1e-12), *scale_ub) when scale_ub is
 *   given (device fp32, nullable), else max(m, 1e-12);
 *   s = 448 / m;  out_scale[i] = 1 / s;
 *   out[i, j] = e4m3( clamp(v_j * s, -448, 448) ), round to nearest even.
 * All arithmetic is IEEE fp32 (correctly rounded division and reciprocal).
 * out [a, D] e4m3, out_scale [a] fp32.  Rows i >= valid are not written.
 * inv_rows, top_k, launch: as in moe_gather_scale.
 */
int moe_gather_scale_quant(const void* x, int T, int D, const int32_t* token_indices,
                           const int32_t* expert_indices, int a, const void* scores,
                           int scores_dtype, int64_t stride_t, int64_t stride_e, int E,
                           const int32_t* valid_token_count, const int32_t* inv_rows, int top_k,
                           const float* scale_ub, void* out, float* out_scale, cudaStream_t stream);

/*
 * Per-row FP8 quantisation of an fp32 matrix w [rows, cols] with the rule of
 * moe_gather_scale_quant (score 1), for FP8-rowwise expert weights (the
 * per-row weight scales of mslk/moe/layers.py, RoutedExperts.build).
 * q [rows, cols] e4m3, scale [rows] fp32; scale_ub nullable.
 */
int moe_quantize_rows(const float* w, int64_t rows, int cols, const float* scale_ub, void* q,
                      float* scale, cudaStream_t stream);

/* ----------------------------------------------------------- grouped GEMM */

/*
 * grouped_gemm(x, w.view(-1, K), token_counts) of mslk/moe/layers.py
 * (MetaShufflingMoE._routed_expert).  Expert e owns the rows
 * [off_e, off_e + counts[e]) of x, off_e = counts[0] + ... + counts[e-1], and
 *   v[r, n] = sum_k x[r, k] * w[e, n, k]     (fp32 accumulation)
 * epilogue MOE_EPILOGUE_NONE:     y [a_max, N] bf16, y[r, n] = bf16(v[r, n])
 * epilogue MOE_EPILOGUE_SILU_MUL: N = 2H (the w13 layout of
 *   RoutedExperts.build: rows [0, H) are the SiLU input, [H, 2H) the gate);
 *   y [a_max, H] bf16, y[r, j] = bf16(silu(y0) * y1) with y0 = bf16(v[r, j])
 *   and y1 = bf16(v[r, H + j]), i.e. moe_silu_mul of the unfused output.
 * x [a_max, K] bf16; w [E, N, K] bf16; counts [E] device int32 (the sum is
 * the number of routed rows; rows past it are not written).  Runs on the
 * tensor cores (tcgen05, accumulators in tensor memory, TMA-fed).
 * Requires N, K multiples of 16 (H a multiple of 16 for SILU_MUL), E <= 1024.
 *
 * epilogue may carry MOE_GEMM_CTA_PAIRS (OR-ed in): 256-row x 256-column tiles
 * computed by a cluster of two CTAs with tcgen05.mma.cta_group::2 instead of
 * 128-row tiles on one CTA.  Each output element is accumulated in the same
 * order either way, so the bytes are identical; pairs move a third less operand
 * data per K block but pad each expert to a multiple of 256 rows.
 *
 * scatter_indices (nullable; MOE_EPILOGUE_NONE only): the combine fused into
 * the epilogue, grouped_gemm(..., _output_tensor=out,
 * _scatter_add_indices=token_indices) of _routed_expert, for top_k = 1 where
 * every token has exactly one routed row.  y is then out [T_out, N]; routed
 * row r's bf16 result o goes to y[scatter_indices[r], :]: y = bf16(f32(y) +
 * f32(o)) with accumulate != 0 (moe_scatter_add's arithmetic), y = o with
 * accumulate == 0.  Rows of y that no routed row names are not touched; an
 * index outside [0, T_out) is skipped and flagged.
 *
 * epilogue MOE_EPILOGUE_SILU_MUL_QUANT: the SiLU*mul epilogue followed by the
 *   FP8-rowwise quantisation of z that the FP8 w2 GEMM takes, the
 *   silu_mul_quant(y0, y1, scale_ub) step of _routed_expert's FP8 branch.  y
 *   [a_max, H] bf16 receives z = bf16(silu(y0) * y1) exactly as with SILU_MUL
 *   (the row max spans every N tile of the row, which different CTAs compute,
 *   so z crosses HBM once, as bf16: 2 bytes per element instead of the 4 of
 *   the unfused y0, y1); then each routed row of z is quantised with the rule
 *   of moe_gather_scale_quant at unit score: m = max_j |z_j|, clamped to
 *   [1e-12, *scale_ub] (scale_ub: device fp32, nullable: no upper bound),
 *   s = 448 / m, z_scale[r] = 1 / s, z_out[r, j] = e4m3(clamp(z_j * s, +-448)).
 *   z_out [a_max, H] e4m3 and z_scale [a_max] fp32; rows past sum(counts) are
 *   not written.  The bf16 rounding of z before its quantisation is the order
 *   of BaselineMoE._forward, where routed_z is a bf16 tensor when _fake_quant
 *   quantises it; the result equals SILU_MUL followed by moe_gather_scale_quant
 *   of y with identity indices and unit scores, bit for bit.  H <= 16384.
 *   Two kernels run on the stream: the GEMM, then a row pass over y.
 * scale_ub, z_out, z_scale: used by MOE_EPILOGUE_SILU_MUL_QUANT only (z_out and
 *   z_scale are then required, 16-byte aligned z_out); ignored otherwise.
 */
int moe_grouped_gemm(const void* x, const void* w, const int32_t* counts, int E, int a_max, int N,
                     int K, void* y, int epilogue, const int32_t* scatter_indices, int T_out,
                     int accumulate, const float* scale_ub, void* z_out, float* z_scale,
                     cudaStream_t stream);

/*
 * grouped_gemm_fp8_rowwise(x, w, counts, x_scale, w_scale) of
 * mslk/moe/layers.py: as moe_grouped_gemm on e4m3 operands, with
 *   v[r, n] = (sum_k x[r, k] * w[e, n, k]) * x_scale[r] * w_scale[e * N + n]
 * (fp32; the dequantisation order of BaselineMoE._fake_quant).
 * x [a_max, K] e4m3, w [E, N, K] e4m3, x_scale [a_max] fp32, w_scale [E * N]
 * fp32.  Epilogues and the fused combine as in moe_grouped_gemm; with
 * MOE_EPILOGUE_SILU_MUL_QUANT the v above (dequantised, then rounded to bf16)
 * are the y0, y1 of SiLU*mul, and z_out, z_scale feed the FP8 w2 GEMM as its
 * x, x_scale (_routed_expert's grouped_gemm_fp8_rowwise -> silu_mul_quant ->
 * grouped_gemm_fp8_rowwise).
 */
int moe_grouped_gemm_fp8_rowwise(const void* x, const void* w, const int32_t* counts,
                                 const float* x_scale, const float* w_scale, int E, int a_max,
                                 int N, int K, void* y, int epilogue, const int32_t* scatter_indices,
                                 int T_out, int accumulate, const float* scale_ub, void* z_out,
                                 float* z_scale, cudaStream_t stream);

/*
 * Both grouped GEMMs of the bf16 routed experts in one persistent launch:
 * z = moe_grouped_gemm(x, w13, counts, MOE_EPILOGUE_SILU_MUL) followed by
 * y = moe_grouped_gemm(z, w2, counts) (the two GEMMs of
 * MetaShufflingMoE._routed_expert with silu_mul between them).  Results are
 * bit-identical to the two separate calls.  Each CTA works through its w13
 * tiles, then its w2 tiles; a w2 tile of expert e starts once every w13 tile
 * of e has stored its z rows, so the w2 work fills the tail of the w13 work.
 * x [a_max, D], w13 [E, 2H, D], w2 [E, D, H], z [a_max, H] (written: it is
 * the intermediate), y [a_max, D]; all bf16.  counts [E] device int32.
 * ws: device workspace of moe_expert_mlp_workspace_size(E) bytes: per-expert
 * counters that must be zero before the first call (cudaMemset); every call
 * leaves them zero again, including one that stops on a device error, so a
 * workspace is zeroed once and reused.  One workspace serves one call at a time.
 * All CTAs must be resident at once (a cooperative launch); MOE_ERR_CUDA if the
 * device cannot host them.  D, H multiples of 16.
 * scatter_indices, T_out, accumulate: the fused top_k = 1 combine of the w2
 * GEMM, as in moe_grouped_gemm (y is then out [T_out, D]).
 * flags: 0, or MOE_WEIGHTS_PACKED when w13 and w2 are tile-packed (then H and D
 * must be multiples of 128); other bits: MOE_ERR_INVALID.
 */
int moe_expert_mlp_workspace_size(int E, size_t* bytes);
int moe_expert_mlp(const void* x, const void* w13, const void* w2, const int32_t* counts, int E, int a_max,
                   int D, int H, void* z, void* y, const int32_t* scatter_indices, int T_out, int accumulate,
                   void* ws, size_t ws_bytes, int flags, cudaStream_t stream);

/*
 * Tile-packed weights (a layout of this library, not of the pages): the
 * weights [E, N, K] of a grouped GEMM, viewed as R = E * N rows of K elements
 * (dtype MOE_DTYPE_BF16 or MOE_DTYPE_E4M3), cut into boxes of 128 rows x 128
 * bytes: box (b, c) holds rows 128 b .. 128 b + 127 and bytes 128 c .. 128 c +
 * 127 of each row, zero where a row or a byte lies past R or K.  Boxes are
 * stored whole, 16 KB each, in (row block b, column block c) order, with
 * ceil(K * elem / 128) column blocks per row block.  Each is the unit the
 * GEMMs' TMA loads fetch, so packed weights stream from HBM sequentially.
 * moe_pack_weights_size: bytes of the packed copy (K % 16 == 0, else
 * MOE_ERR_UNSUPPORTED).  moe_pack_weights: write it from row-major w (device,
 * 16-byte aligned; packed must not overlap w).  Asynchronous on stream.  The
 * scales of FP8 weights are not affected.
 */
int moe_pack_weights_size(int E, int N, int K, int dtype, size_t* bytes);
int moe_pack_weights(const void* w, int E, int N, int K, int dtype, void* packed, cudaStream_t stream);

/* ------------------------------------------------------ dense GEMM (shared expert) */

/*
 * The shared expert's dense GEMMs of mslk/moe/layers.py
 * (MetaShufflingMoE._shared_expert_part1 / _part2: x @ w13.T, then z @ w2.T)
 * for batches with few row tiles: the K dimension is split across the CTAs of
 * a thread-block cluster and the fp32 partials are added in a fixed order over
 * distributed shared memory, so more SMs stream the weights.
 *   v[r, n] = sum_k x[r, k] * w[n, k]                   (fp32)
 *   MOE_EPILOGUE_NONE:     y [M, N] bf16, y[r, n] = bf16(v[r, n])
 *   MOE_EPILOGUE_SILU_MUL: N = 2H, y [M, H] bf16,
 *                          y[r, j] = bf16(silu_mul(bf16(v[r, j]), bf16(v[r, H + j])))
 *                          (the grouped GEMM's SiLU*mul epilogue)
 * x [M, K], w [N, K] bf16, row-major, 16-byte aligned; valid_rows: device int32
 * row count (NULL: M), rows at or past it are not written.  K, N multiples of
 * 16 (MOE_ERR_UNSUPPORTED).  Deterministic on a given device.
 */
int moe_dense_gemm(const void* x, int M, int K, const void* w, int N, const int32_t* valid_rows,
                   void* y, int epilogue, cudaStream_t stream);

/* ---------------------------------------------------------------- silu_mul */

/*
 * silu_mul(x0, x1) (MetaShufflingMoE._fused_silu_mul): for rows r < valid,
 *   z[r, j] = bf16( y0 * sigmoid(y0) * y1 ),  y0 = x0[r * ld + j],
 *   y1 = x1[r * ld + j], in fp32 (sigmoid(a) = 1 / (1 + exp(-a))).
 * x0, x1 bf16 with row stride ld elements (ld = 2H for the halves of a
 * [a, 2H] GEMM output); z [a, H] bf16; valid_rows: device int32 routed-row
 * count (nullable: a).  Rows r >= valid are not written.
 */
int moe_silu_mul(const void* x0, const void* x1, int64_t ld, int a, int H,
                 const int32_t* valid_rows, void* z, cudaStream_t stream);

/*
 * silu_mul_quant(x0, x1, scale_ub): the fp32 row of z is quantised over its H
 * entries with the rule of moe_gather_scale_quant.  z [a, H] e4m3,
 * z_scale [a] fp32.
 */
int moe_silu_mul_quant(const void* x0, const void* x1, int64_t ld, int a, int H,
                       const int32_t* valid_rows, const float* scale_ub, void* z, float* z_scale,
                       cudaStream_t stream);

/* ------------------------------------------------------------- scatter-add */

/*
 * scatter_add_dense_tokens (mslk/moe/gather_scatter.py,
 * _mslk_scatter_add_dense_tokens), made deterministic: every routed row
 * r < valid is added into out[token_indices[r], :].  Each output token is
 * owned by one warp: acc = f32(out[t, :]) (accumulate != 0) or 0
 * (accumulate == 0: the routed sum overwrites out, as adding into zeros
 * would); acc += f32(in[r, :]) for t's rows in ascending r;
 * out[t, :] = bf16(acc).  No atomics.
 * out [T, D] bf16 (read and written); in [a, D] bf16; token_indices [a].
 * inv_rows [Tv * top_k] from moe_route (t's rows, ascending) is required when
 * top_k > 1; with top_k == 1 it may be NULL (row r then owns its token).
 * valid_token_count: device int32 routed-row count (NULL: a); with inv_rows
 * it must equal Tv * top_k.  Tokens that receive no row are not written.
 */
int moe_scatter_add(void* out, const void* in, const int32_t* token_indices,
                    const int32_t* inv_rows, int top_k, int a, int T, int D,
                    const int32_t* valid_token_count, int accumulate, cudaStream_t stream);

/*
 * scatter_add_padded_tokens (mslk/moe/gather_scatter.py,
 * _mslk_scatter_add_padded_tokens) on one GPU (EP = 1): in [T_K, D] holds each
 * expert's rows back to back (expert e at rows [sum_{e' < e} counts[e'],
 * ... + counts[e])) followed by padding; the valid rows are the first
 * sum(token_counts[0, E)) and each is added into out[token_indices[row], :].
 * With one rank this is moe_scatter_add with that row count, and it is
 * computed the same deterministic way (token_counts is read on the device).
 * token_counts [E] device int32 (negative entries count as 0 and are flagged
 * MOE_DEVERR_BAD_COUNT); T_K must be a multiple of T (T_K = T * top_k).
 * Other arguments as moe_scatter_add.
 */
int moe_scatter_add_padded(void* out, const void* in, const int32_t* token_counts, int E,
                           const int32_t* token_indices, const int32_t* inv_rows, int top_k,
                           int T_K, int T, int D, int accumulate, cudaStream_t stream);

/* ----------------------------------------------------------- top-k finalize */

/*
 * Top-k finalize of an unfinalized MoE output: the single-GPU part of
 * AllReduceRMSNormWithReduceScatterEarlyExit.finalize on the "kimi_k3 ...
 * allreduce_rmsnorm_reduce_scatter_early_exit" page, where the routing
 * weights act on the expert outputs rather than their inputs.  For every token
 * t < M (or < *valid_token_count) and column d:
 *   acc = 0 (fp32); for slot j = 0 .. top_k-1 in order:
 *     p = expanded_idx_to_permuted_idx[t, j]; skipped when p < 0;
 *     acc = acc + w[t, j] * rows[p, d]        (fp32 multiply, then fp32 add)
 *   r = bf16(acc) with a negative zero written as +0
 *   out[t, d] = r, or bf16(f32(r) + f32(shared_output[t, d])) with a shared output
 * rows [n_rows, D] bf16: the unweighted GEMM2 rows in the routed (by-expert)
 *   order; expert_weights [M, top_k] fp32 (MOE_DTYPE_F32) or bf16
 *   (MOE_DTYPE_BF16); expanded_idx_to_permuted_idx [M, top_k] int32 (moe_route's
 *   inv_rows, with its topk_weights, fit directly); shared_output [M, D] bf16 or
 *   NULL; out [M, D] bf16.  An index >= n_rows is skipped and flagged
 *   MOE_DEVERR_BAD_INDEX.  Tokens t >= the valid count are not written.
 * D a multiple of 16 and 16-byte aligned rows/out/shared (MOE_ERR_UNSUPPORTED).
 */
int moe_topk_finalize(const void* rows, int64_t n_rows, int D, const void* expert_weights,
                      int weights_dtype, const int32_t* expanded_idx_to_permuted_idx, int M,
                      int top_k, const int32_t* valid_token_count, const void* shared_output,
                      void* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
