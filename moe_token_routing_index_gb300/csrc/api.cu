// The C ABI of libmoe_gb300 (declared in include/moe.h): argument checks on
// the host, then the launchers of the kernel translation units.
#include <cuda.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "launch.h"

namespace {

thread_local int t_last_cuda_error = 0;

// Device-side error word (MOE_DEVERR_* bits), one per device that loads the library.
__device__ unsigned int g_moe_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return MOE_ERR_CUDA;
}

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (*dev < 0 || *dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

unsigned long long g_err_ctx[kMaxDevices] = {};

// Device address of the error word on the current device: looked up once per
// device and context (again after the context changed, e.g. after cudaDeviceReset).
int device_error_word(unsigned int** out) {
  int dev;
  int rc = current_device(&dev);
  if (rc != MOE_OK) return rc;
  const unsigned long long ctx = moe::current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev] || ctx == 0 || ctx != g_err_ctx[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_moe_device_error);
    if (e != cudaSuccess) return cuda_fail(e);
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
    g_err_ctx[dev] = moe::current_context_id();  // the lookup made the primary context current if it was not
  }
  *out = g_err_ptr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int finish(cudaError_t e) { return e == cudaSuccess ? MOE_OK : cuda_fail(e); }

int check_scores(const void* scores, int dtype, int E) {
  if (!scores) return MOE_ERR_INVALID;
  if (dtype != MOE_DTYPE_BF16 && dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID;
  if (E < 1) return MOE_ERR_INVALID;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

namespace moe {
void record_cuda_error(int e) { t_last_cuda_error = e; }

unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
    cudaGetLastError();  // a failed lookup leaves no sticky error behind
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

int resident_blocks_per_sm(const void* kernel, int threads) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  static std::map<std::pair<int, const void*>, int> cache;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = cache.find({dev, kernel});
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) n = 1;
  cache[{dev, kernel}] = n;
  return n;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kNumSmsGB300;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kNumSmsGB300;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}
}  // namespace moe

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape, alignment or type";
    case MOE_ERR_CUDA: return "CUDA error (see moe_last_cuda_error)";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int moe_last_cuda_error(void) { return t_last_cuda_error; }

int moe_device_error(unsigned int* bits, cudaStream_t stream) {
  if (!bits) return MOE_ERR_INVALID;
  unsigned int* p;
  int rc = device_error_word(&p);
  if (rc != MOE_OK) return rc;
  cudaError_t e = cudaMemcpyAsync(bits, p, sizeof(unsigned int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(unsigned int), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return finish(e);
}

int moe_route_workspace_size(int T, int E, int top_k, size_t* bytes) {
  if (!bytes || T < 0 || E < 1 || top_k < 1 || top_k > E) return MOE_ERR_INVALID;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)T * top_k > INT32_MAX) return MOE_ERR_INVALID;
  *bytes = moe::route_workspace_bytes(T, E, top_k);
  return MOE_OK;
}

int moe_route(const void* scores, int scores_dtype, int64_t stride_t, int64_t stride_e, int T, int E, int top_k,
              const int32_t* num_valid_tokens, int32_t* counts, int32_t* expert_offsets, int32_t* expert_indices,
              int32_t* token_indices, int32_t* inv_rows, float* topk_weights, void* ws, size_t ws_bytes,
              cudaStream_t stream) {
  size_t need;
  int rc = moe_route_workspace_size(T, E, top_k, &need);
  if (rc != MOE_OK) return rc;
  if (!counts || !expert_offsets) return MOE_ERR_INVALID;
  if (T > 0) {
    rc = check_scores(scores, scores_dtype, E);
    if (rc != MOE_OK) return rc;
    if (!expert_indices || !token_indices || !ws) return MOE_ERR_INVALID;
    if (stride_t < 0 || stride_e < 0) return MOE_ERR_INVALID;
  }
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_INVALID;
  moe::RouteArgs a{scores,         scores_dtype,  stride_t,     stride_e, T,  E,      top_k,
                   num_valid_tokens, counts,      expert_offsets, expert_indices, token_indices, inv_rows,
                   topk_weights,   ws,            nullptr};
  rc = device_error_word(&a.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_route(a, stream));
}

int moe_router_workspace_size(int T, int D, int E, size_t* bytes) {
  if (!bytes || T < 0 || D < 1 || E < 1) return MOE_ERR_INVALID;
  if (E > 256 || D % 16 != 0) return MOE_ERR_UNSUPPORTED;
  *bytes = moe::router_workspace_bytes(T, D, E);
  return MOE_OK;
}

int moe_router_scores(const void* x, int T, int D, const void* w_router, int E, const int32_t* num_valid_tokens,
                      void* scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  size_t need;
  int rc = moe_router_workspace_size(T, D, E, &need);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !scores || (need > 0 && !ws)) return MOE_ERR_INVALID;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w_router) || (reinterpret_cast<uintptr_t>(scores) & 1u)) return MOE_ERR_UNSUPPORTED;
  moe::RouterArgs a{x, T, D, w_router, E, num_valid_tokens, scores, ws, nullptr};
  rc = device_error_word(&a.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_router_scores(a, stream));
}

int moe_router_route_workspace_size(int T, int D, int E, int top_k, size_t* bytes) {
  size_t router = 0;
  int rc = moe_router_workspace_size(T, D, E, &router);
  if (rc != MOE_OK) return rc;
  return moe_route_workspace_size(T, E, top_k, bytes);
}

int moe_router_route(const void* x, int T, int D, const void* w_router, int E, int top_k,
                     const int32_t* num_valid_tokens, void* scores, int32_t* counts, int32_t* expert_offsets,
                     int32_t* expert_indices, int32_t* token_indices, int32_t* inv_rows, float* topk_weights,
                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  size_t need;
  int rc = moe_router_route_workspace_size(T, D, E, top_k, &need);
  if (rc != MOE_OK) return rc;
  if (!counts || !expert_offsets) return MOE_ERR_INVALID;
  if (T > 0 && (!x || !w_router || !scores || !expert_indices || !token_indices || !ws)) return MOE_ERR_INVALID;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_INVALID;
  if (T > 0 && (!aligned16(x) || !aligned16(w_router) || (reinterpret_cast<uintptr_t>(scores) & 1u)))
    return MOE_ERR_UNSUPPORTED;
  moe::RouteArgs r{scores,         MOE_DTYPE_BF16, E,       1,        T,  E,      top_k,
                   num_valid_tokens, counts,       expert_offsets, expert_indices, token_indices, inv_rows,
                   topk_weights,   ws,             nullptr};
  rc = device_error_word(&r.err);
  if (rc != MOE_OK) return rc;
  if (T == 0) return finish(moe::launch_route(r, stream));  // zero counts and offsets
  moe::RouterArgs a{x, T, D, w_router, E, num_valid_tokens, scores, nullptr, r.err};
  cudaError_t e = moe::launch_router_route(a, top_k, moe::route_workspace(ws, T, top_k), stream);
  if (e != cudaSuccess) return finish(e);
  return finish(moe::launch_route_emit(r, stream));
}

int moe_dense_gemm(const void* x, int M, int K, const void* w, int N, const int32_t* valid_rows, void* y,
                   int epilogue, cudaStream_t stream) {
  if (M < 0 || K < 0 || N < 0) return MOE_ERR_INVALID;
  if (epilogue != MOE_EPILOGUE_NONE && epilogue != MOE_EPILOGUE_SILU_MUL) return MOE_ERR_INVALID;
  if (M == 0 || N == 0) return MOE_OK;
  if (!x || !w || !y) return MOE_ERR_INVALID;
  if (K == 0 || K % 16 != 0 || N % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || (reinterpret_cast<uintptr_t>(y) & 1u)) return MOE_ERR_UNSUPPORTED;
  moe::DenseArgs a{x, M, K, w, N, epilogue, valid_rows, y, nullptr};
  int rc = device_error_word(&a.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_dense_gemm(a, stream));
}

int moe_selftest_bounded_wait(int which, int64_t limit_ns, cudaStream_t stream) {
  if (which != 0 && which != 1) return MOE_ERR_INVALID;
  if (limit_ns < 1000 || limit_ns > 2000000000ll) return MOE_ERR_INVALID;
  unsigned int* err = nullptr;
  int rc = device_error_word(&err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_selftest_wait(which, (uint64_t)limit_ns, err, stream));
}

static int check_gather(const void* x, int T, int D, const int32_t* ti, const int32_t* ei, int a,
                        const void* scores, int dtype, int E, const void* out) {
  if (T < 0 || D < 0 || a < 0) return MOE_ERR_INVALID;
  if (a == 0 || D == 0) return MOE_OK;
  if (!x || !ti || !ei || !out) return MOE_ERR_INVALID;
  if (scores) {  // NULL scores: every score is 1 (the rows are copied)
    int rc = check_scores(scores, dtype, E);
    if (rc != MOE_OK) return rc;
  }
  if (D % 16 != 0 || !aligned16(x) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int moe_gather_scale(const void* x, int T, int D, const int32_t* token_indices, const int32_t* expert_indices, int a,
                     const void* scores, int scores_dtype, int64_t stride_t, int64_t stride_e, int E,
                     const int32_t* valid_token_count, const int32_t* inv_rows, int top_k, void* out,
                     cudaStream_t stream) {
  int rc = check_gather(x, T, D, token_indices, expert_indices, a, scores, scores_dtype, E, out);
  if (rc != MOE_OK || a == 0 || D == 0) return rc;
  if (inv_rows && top_k < 1) return MOE_ERR_INVALID;
  moe::GatherArgs g{x, T, D, token_indices, expert_indices, a, scores, scores_dtype, stride_t, stride_e, E,
                    valid_token_count, nullptr, out, nullptr, inv_rows, inv_rows ? top_k : 1, nullptr};
  rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_gather_scale(g, stream));
}

int moe_gather_scale_quant(const void* x, int T, int D, const int32_t* token_indices, const int32_t* expert_indices,
                           int a, const void* scores, int scores_dtype, int64_t stride_t, int64_t stride_e, int E,
                           const int32_t* valid_token_count, const int32_t* inv_rows, int top_k,
                           const float* scale_ub, void* out, float* out_scale, cudaStream_t stream) {
  int rc = check_gather(x, T, D, token_indices, expert_indices, a, scores, scores_dtype, E, out);
  if (rc != MOE_OK || a == 0 || D == 0) return rc;
  if (!out_scale) return MOE_ERR_INVALID;
  if (inv_rows && top_k < 1) return MOE_ERR_INVALID;
  if (D > 16384) return MOE_ERR_UNSUPPORTED;
  moe::GatherArgs g{x, T, D, token_indices, expert_indices, a, scores, scores_dtype, stride_t, stride_e, E,
                    valid_token_count, scale_ub, out, out_scale, inv_rows, inv_rows ? top_k : 1, nullptr};
  rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_gather_scale_quant(g, stream));
}

int moe_quantize_rows(const float* w, int64_t rows, int cols, const float* scale_ub, void* q, float* scale,
                      cudaStream_t stream) {
  if (rows < 0 || cols < 0) return MOE_ERR_INVALID;
  if (rows == 0 || cols == 0) return MOE_OK;
  if (!w || !q || !scale) return MOE_ERR_INVALID;
  if (cols % 16 != 0 || !aligned16(w) || !aligned16(q)) return MOE_ERR_UNSUPPORTED;
  return finish(moe::launch_quantize_rows(w, rows, cols, scale_ub, q, scale, stream));
}

static int check_silu(const void* x0, const void* x1, int64_t ld, int a, int H, const void* z) {
  if (a < 0 || H < 0) return MOE_ERR_INVALID;
  if (a == 0 || H == 0) return MOE_OK;
  if (!x0 || !x1 || !z || ld < H) return MOE_ERR_INVALID;
  if (H % 16 != 0 || ld % 8 != 0 || !aligned16(x0) || !aligned16(x1) || !aligned16(z)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int moe_silu_mul(const void* x0, const void* x1, int64_t ld, int a, int H, const int32_t* valid_rows, void* z,
                 cudaStream_t stream) {
  int rc = check_silu(x0, x1, ld, a, H, z);
  if (rc != MOE_OK || a == 0 || H == 0) return rc;
  moe::SiluArgs g{x0, x1, ld, a, H, valid_rows, nullptr, z, nullptr, nullptr};
  rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_silu_mul(g, stream));
}

int moe_silu_mul_quant(const void* x0, const void* x1, int64_t ld, int a, int H, const int32_t* valid_rows,
                       const float* scale_ub, void* z, float* z_scale, cudaStream_t stream) {
  int rc = check_silu(x0, x1, ld, a, H, z);
  if (rc != MOE_OK || a == 0 || H == 0) return rc;
  if (!z_scale) return MOE_ERR_INVALID;
  if (H > 16384) return MOE_ERR_UNSUPPORTED;
  moe::SiluArgs g{x0, x1, ld, a, H, valid_rows, scale_ub, z, z_scale, nullptr};
  rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_silu_mul_quant(g, stream));
}

int moe_scatter_add(void* out, const void* in, const int32_t* token_indices, const int32_t* inv_rows, int top_k,
                    int a, int T, int D, const int32_t* valid_token_count, int accumulate, cudaStream_t stream) {
  if (a < 0 || T < 0 || D < 0 || top_k < 1) return MOE_ERR_INVALID;
  if (a == 0 || D == 0 || T == 0) return MOE_OK;
  if (!out || !in) return MOE_ERR_INVALID;
  if (top_k > 1 && !inv_rows) return MOE_ERR_INVALID;
  if (!inv_rows && !token_indices) return MOE_ERR_INVALID;
  if (D % 16 != 0 || !aligned16(out) || !aligned16(in)) return MOE_ERR_UNSUPPORTED;
  moe::ScatterArgs g{out, in, token_indices, inv_rows, top_k, a, T, D, valid_token_count, accumulate != 0,
                     nullptr, 0, nullptr};
  int rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_scatter_add(g, stream));
}

int moe_scatter_add_padded(void* out, const void* in, const int32_t* token_counts, int E,
                           const int32_t* token_indices, const int32_t* inv_rows, int top_k, int T_K, int T, int D,
                           int accumulate, cudaStream_t stream) {
  if (E < 1 || T_K < 0 || T < 0 || D < 0 || top_k < 1) return MOE_ERR_INVALID;
  if (T_K == 0 || D == 0 || T == 0) return MOE_OK;
  if (!out || !in || !token_counts) return MOE_ERR_INVALID;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  if (T_K % T != 0) return MOE_ERR_INVALID;  // the padded layout holds T_K = T * top_k rows
  if (top_k > 1 && !inv_rows) return MOE_ERR_INVALID;
  if (!inv_rows && !token_indices) return MOE_ERR_INVALID;
  if (D % 16 != 0 || !aligned16(out) || !aligned16(in)) return MOE_ERR_UNSUPPORTED;
  moe::ScatterArgs g{out, in, token_indices, inv_rows, top_k, T_K, T, D, nullptr, accumulate != 0,
                     token_counts, E, nullptr};
  int rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_scatter_add(g, stream));
}

int moe_topk_finalize(const void* rows, int64_t n_rows, int D, const void* expert_weights, int weights_dtype,
                      const int32_t* expanded_idx_to_permuted_idx, int M, int top_k,
                      const int32_t* valid_token_count, const void* shared_output, void* out, cudaStream_t stream) {
  if (n_rows < 0 || D < 0 || M < 0 || top_k < 1) return MOE_ERR_INVALID;
  if (M == 0 || D == 0) return MOE_OK;
  if (!out || !expert_weights || !expanded_idx_to_permuted_idx || (n_rows > 0 && !rows)) return MOE_ERR_INVALID;
  if (weights_dtype != MOE_DTYPE_F32 && weights_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID;
  if (D % 16 != 0 || !aligned16(out) || (rows && !aligned16(rows)) || (shared_output && !aligned16(shared_output)))
    return MOE_ERR_UNSUPPORTED;
  moe::FinalizeArgs g{rows, n_rows, D, expert_weights, weights_dtype, expanded_idx_to_permuted_idx, M, top_k,
                      valid_token_count, shared_output, out, nullptr};
  int rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  return finish(moe::launch_topk_finalize(g, stream));
}

static int grouped_gemm_common(const void* x, const void* w, const int32_t* counts, const float* x_scale,
                               const float* w_scale, int E, int a_max, int N, int K, void* y, int epilogue,
                               const int32_t* scatter, int T_out, int accumulate, const float* scale_ub,
                               void* z_out, float* z_scale, bool fp8, cudaStream_t stream) {
  if (E < 1 || a_max < 0 || N < 0 || K < 0) return MOE_ERR_INVALID;
  const bool pairs = (epilogue & MOE_GEMM_CTA_PAIRS) != 0;
  const bool packed = (epilogue & MOE_WEIGHTS_PACKED) != 0;
  epilogue &= ~(MOE_GEMM_CTA_PAIRS | MOE_WEIGHTS_PACKED);
  if (epilogue != MOE_EPILOGUE_NONE && epilogue != MOE_EPILOGUE_SILU_MUL && epilogue != MOE_EPILOGUE_SILU_MUL_QUANT)
    return MOE_ERR_INVALID;
  const bool quant = epilogue == MOE_EPILOGUE_SILU_MUL_QUANT;
  const bool silu = epilogue != MOE_EPILOGUE_NONE;
  if (a_max == 0 || N == 0) return MOE_OK;
  if (!x || !w || !counts || !y) return MOE_ERR_INVALID;
  if (fp8 && (!x_scale || !w_scale)) return MOE_ERR_INVALID;
  if (quant && (!z_out || !z_scale)) return MOE_ERR_INVALID;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  if (N % 16 != 0 || K % 16 != 0 || K == 0) return MOE_ERR_UNSUPPORTED;
  if (silu && (N % 32 != 0)) return MOE_ERR_UNSUPPORTED;
  if (quant && (N / 2 > 16384 || !aligned16(z_out))) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return MOE_ERR_UNSUPPORTED;
  if (scatter && (epilogue != MOE_EPILOGUE_NONE || T_out < 0)) return MOE_ERR_INVALID;
  // packed weights: every weight box starts at a 128-row block (SiLU*mul: both halves)
  if (packed && (N % 128 != 0 || (silu && (N / 2) % 128 != 0))) return MOE_ERR_UNSUPPORTED;
  // the GEMM runs the SiLU*mul epilogue into y; SILU_MUL_QUANT then quantises y's rows
  moe::GemmArgs g{x, w, counts, x_scale, w_scale, E, a_max, N, K, y, silu ? MOE_EPILOGUE_SILU_MUL : epilogue, fp8,
                  pairs, packed, scatter, T_out, accumulate, nullptr};
  int rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  cudaError_t e = moe::launch_grouped_gemm(g, stream);
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  if (e != cudaSuccess || !quant) return finish(e);
  const int H = N / 2;
  moe::SiluArgs q{y, nullptr, H, a_max, H, nullptr, scale_ub, z_out, z_scale, g.err, counts, E};
  return finish(moe::launch_quantize_rows_bf16(q, stream));
}

int moe_expert_mlp_workspace_size(int E, size_t* bytes) {
  if (!bytes || E < 1) return MOE_ERR_INVALID;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  *bytes = moe::expert_mlp_workspace_bytes(E);
  return MOE_OK;
}

int moe_expert_mlp(const void* x, const void* w13, const void* w2, const int32_t* counts, int E, int a_max, int D,
                   int H, void* z, void* y, const int32_t* scatter_indices, int T_out, int accumulate, void* ws,
                   size_t ws_bytes, int flags, cudaStream_t stream) {
  size_t need;
  int rc = moe_expert_mlp_workspace_size(E, &need);
  if (rc != MOE_OK) return rc;
  if (a_max < 0 || D < 0 || H < 0) return MOE_ERR_INVALID;
  if (a_max == 0 || D == 0 || H == 0) return MOE_OK;
  if (!x || !w13 || !w2 || !counts || !z || !y || !ws) return MOE_ERR_INVALID;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (D % 16 != 0 || H % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(z) || !aligned16(y) || !aligned16(ws))
    return MOE_ERR_UNSUPPORTED;
  if (scatter_indices && T_out < 0) return MOE_ERR_INVALID;
  if (flags & ~MOE_WEIGHTS_PACKED) return MOE_ERR_INVALID;
  const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
  if (packed && (H % 128 != 0 || D % 128 != 0)) return MOE_ERR_UNSUPPORTED;
  moe::MlpArgs g{x, w13, w2, counts, E, a_max, D, H, z, y, ws, scatter_indices, T_out, accumulate, nullptr, packed};
  rc = device_error_word(&g.err);
  if (rc != MOE_OK) return rc;
  cudaError_t e = moe::launch_expert_mlp(g, stream);
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  return finish(e);
}

int moe_pack_weights_size(int E, int N, int K, int dtype, size_t* bytes) {
  if (!bytes || E < 1 || N < 1 || K < 1) return MOE_ERR_INVALID;
  if (dtype != MOE_DTYPE_BF16 && dtype != MOE_DTYPE_E4M3) return MOE_ERR_INVALID;
  if (K % 16 != 0) return MOE_ERR_UNSUPPORTED;
  *bytes = moe::packed_weights_bytes((int64_t)E * N, K, dtype == MOE_DTYPE_E4M3);
  return MOE_OK;
}

int moe_pack_weights(const void* w, int E, int N, int K, int dtype, void* packed, cudaStream_t stream) {
  size_t need;
  int rc = moe_pack_weights_size(E, N, K, dtype, &need);
  if (rc != MOE_OK) return rc;
  if (!w || !packed) return MOE_ERR_INVALID;
  if (!aligned16(w) || !aligned16(packed)) return MOE_ERR_UNSUPPORTED;
  return finish(moe::launch_pack_weights(w, (int64_t)E * N, K, dtype == MOE_DTYPE_E4M3, packed, stream));
}

int moe_grouped_gemm(const void* x, const void* w, const int32_t* counts, int E, int a_max, int N, int K, void* y,
                     int epilogue, const int32_t* scatter_indices, int T_out, int accumulate, const float* scale_ub,
                     void* z_out, float* z_scale, cudaStream_t stream) {
  return grouped_gemm_common(x, w, counts, nullptr, nullptr, E, a_max, N, K, y, epilogue, scatter_indices, T_out,
                             accumulate, scale_ub, z_out, z_scale, false, stream);
}

int moe_grouped_gemm_fp8_rowwise(const void* x, const void* w, const int32_t* counts, const float* x_scale,
                                 const float* w_scale, int E, int a_max, int N, int K, void* y, int epilogue,
                                 const int32_t* scatter_indices, int T_out, int accumulate, const float* scale_ub,
                                 void* z_out, float* z_scale, cudaStream_t stream) {
  return grouped_gemm_common(x, w, counts, x_scale, w_scale, E, a_max, N, K, y, epilogue, scatter_indices, T_out,
                             accumulate, scale_ub, z_out, z_scale, true, stream);
}

}  // extern "C"
