// Internal launcher interface between the C ABI (api.cu) and the kernel
// translation units.  Arguments are validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

struct RouteArgs {
  const void* scores;
  int dtype;
  int64_t stride_t, stride_e;
  int T, E, top_k;
  const int32_t* num_valid;
  int32_t* counts;
  int32_t* offsets;
  int32_t* expert_indices;
  int32_t* token_indices;
  int32_t* inv;
  float* weights;  // nullable: top-k scores in the order of inv
  void* ws;
  unsigned int* err;
};

size_t route_workspace_bytes(int T, int E, int top_k);
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);

// The routing workspace: the grid-barrier counter, the chosen experts of each
// token [T * top_k] (selection order) and the per-chunk expert histograms
// [E][ceil(T / 32)] (hist_t[e * nblk + c]: tokens of 32-token chunk c choosing e).
struct RouteWorkspace {
  unsigned int* barrier;
  int32_t* chosen;
  int32_t* hist_t;
};
RouteWorkspace route_workspace(void* ws, int T, int top_k);
// The scan and emit phases of routing (one cooperative launch, one grid barrier),
// after the router GEMM's epilogue has filled the workspace's chosen experts and
// chunk histograms and zeroed its barrier counter.
cudaError_t launch_route_emit(const RouteArgs& a, cudaStream_t s);

struct RouterArgs {
  const void* x;       // bf16 [T, D]
  int T, D;
  const void* w;       // bf16 [E, D]
  int E;
  const int32_t* num_valid;
  void* scores;        // bf16 [T, E]
  void* ws;
  unsigned int* err;
};

size_t router_workspace_bytes(int T, int D, int E);
cudaError_t launch_router_scores(const RouterArgs& a, cudaStream_t s);

// Router scores with the routing selection in the reduction epilogue: scores as
// launch_router_scores, plus the chosen experts, chunk histograms and zeroed
// barrier counter of `w` (the routing workspace of T tokens and top_k) for
// launch_route_emit.
cudaError_t launch_router_route(const RouterArgs& a, int top_k, const RouteWorkspace& w, cudaStream_t s);

struct DenseArgs {
  const void* x;             // bf16 [M, K]
  int M, K;
  const void* w;             // bf16 [N, K]
  int N;
  int epilogue;              // MOE_EPILOGUE_NONE or MOE_EPILOGUE_SILU_MUL
  const int32_t* rows_valid; // nullable: M
  void* y;                   // bf16 [M, N] or [M, N / 2]
  unsigned int* err;
};

cudaError_t launch_dense_gemm(const DenseArgs& a, cudaStream_t s);

cudaError_t launch_selftest_wait(int which, uint64_t limit_ns, unsigned int* err, cudaStream_t s);

struct GatherArgs {
  const void* x;
  int T, D;
  const int32_t* token_indices;
  const int32_t* expert_indices;
  int a;
  const void* scores;
  int dtype;
  int64_t stride_t, stride_e;
  int E;
  const int32_t* valid;
  const float* scale_ub;  // quantising variant only
  void* out;
  float* out_scale;       // quantising variant only
  const int32_t* inv;     // nullable: rows of each token (token-major gather)
  int top_k;
  unsigned int* err;
};

cudaError_t launch_gather_scale(const GatherArgs& a, cudaStream_t s);
cudaError_t launch_gather_scale_quant(const GatherArgs& a, cudaStream_t s);
cudaError_t launch_quantize_rows(const float* w, int64_t rows, int cols, const float* ub, void* q, float* scale,
                                 cudaStream_t s);

struct SiluArgs {
  const void* x0;
  const void* x1;
  int64_t ld;
  int a, H;
  const int32_t* valid;
  const float* scale_ub;  // quantising variant only
  void* z;
  float* z_scale;         // quantising variant only
  unsigned int* err;
  const int32_t* sum_counts;  // nullable: the valid row count is sum(sum_counts[0, E)) instead of *valid
  int E;
};

cudaError_t launch_silu_mul(const SiluArgs& a, cudaStream_t s);
cudaError_t launch_silu_mul_quant(const SiluArgs& a, cudaStream_t s);
// Per-row FP8 quantisation of the bf16 rows x0 (row stride ld; x1 unused) with the
// rule of silu_mul_quant: the second half of the SILU_MUL_QUANT GEMM epilogue.
cudaError_t launch_quantize_rows_bf16(const SiluArgs& a, cudaStream_t s);

struct ScatterArgs {
  void* out;
  const void* in;
  const int32_t* token_indices;
  const int32_t* inv;
  int top_k, a, T, D;
  const int32_t* valid;
  bool accumulate;
  const int32_t* sum_counts;  // nullable: the valid row count is sum(sum_counts[0, E)) instead of *valid
  int E;
  unsigned int* err;
};

cudaError_t launch_scatter_add(const ScatterArgs& a, cudaStream_t s);

struct FinalizeArgs {
  const void* rows;          // bf16 [n_rows, D]
  int64_t n_rows;
  int D;
  const void* weights;       // [M, k] f32 or bf16
  int weights_dtype;
  const int32_t* idx;        // [M, k], -1: absent
  int M, k;
  const int32_t* valid;      // nullable: M
  const void* shared;        // nullable: bf16 [M, D]
  void* out;                 // bf16 [M, D]
  unsigned int* err;
};

cudaError_t launch_topk_finalize(const FinalizeArgs& a, cudaStream_t s);

struct GemmArgs {
  const void* x;        // [a_max, K] bf16 or e4m3
  const void* w;        // [E, N, K]
  const int32_t* counts;
  const float* x_scale; // FP8 only
  const float* w_scale; // FP8 only
  int E, a_max, N, K;
  void* y;
  int epilogue;
  bool fp8;
  bool pairs;              // 256-row tiles on CTA pairs (cta_group::2)
  bool packed;             // w in the tile-packed layout (launch_pack_weights)
  const int32_t* scatter;  // nullable: combine row r into y[scatter[r]] (top_k = 1)
  int T_out;               // rows of y when scattering
  int accumulate;
  unsigned int* err;
};

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s);

// Both grouped GEMMs of a bf16 expert MLP in one launch (w13 with SiLU*mul into z, then w2).
struct MlpArgs {
  const void* x;        // [a_max, D] bf16
  const void* w13;      // [E, 2H, D]
  const void* w2;       // [E, D, H]
  const int32_t* counts;
  int E, a_max, D, H;
  void* z;              // [a_max, H] bf16
  void* y;              // [a_max, D] bf16, or [T_out, D] when scattering
  void* ws;             // expert_mlp_workspace_bytes(E)
  const int32_t* scatter;
  int T_out;
  int accumulate;
  unsigned int* err;
  bool packed;          // w13 and w2 in the tile-packed layout
};

size_t expert_mlp_workspace_bytes(int E);
// Tile-packed weights (every 128-row x 128-byte TMA box contiguous): size and packing.
size_t packed_weights_bytes(int64_t rows, int64_t K, bool fp8);
cudaError_t launch_pack_weights(const void* w, int64_t rows, int64_t K, bool fp8, void* out, cudaStream_t s);
cudaError_t launch_expert_mlp(const MlpArgs& a, cudaStream_t s);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Blocks of `kernel` (with `threads` threads, no dynamic shared memory) that
// fit on one SM at once (cached per device and kernel; at least 1).
int resident_blocks_per_sm(const void* kernel, int threads);

// Make `e` (a cudaError_t) what moe_last_cuda_error() reports on this thread.
void record_cuda_error(int e);

// A process-unique id of the calling thread's current CUDA context, 0 when there is
// none or the driver cannot tell.  Device addresses cached per device are looked up
// again when it changes (cudaDeviceReset replaces a device's primary context).
unsigned long long current_context_id();

// Load the routing kernels' device code on the current device (CUDA loads modules
// lazily, at first use); no launch.
cudaError_t preload_route_kernels();

}  // namespace moe
