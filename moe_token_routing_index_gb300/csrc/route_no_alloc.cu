// moe_route_no_alloc: routing with library-owned scratch, for callers that
// cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc (or any allocating
// routine) on the path that routes tokens: a plugin inside a host framework
// whose own allocator owns the whole device-memory budget, a serving loop
// whose latency budget rules out the implicit device synchronisation and
// unbounded cost of an allocation, or code running where the allocator must
// not be re-entered (for example inside an out-of-memory handler).  Such a
// caller still passes its inputs and outputs, but cannot provide moe_route's
// workspace.  This entry point supplies it from a fixed array compiled into
// the library instead.
//
// The array lives in device global memory of every GPU that loads the
// library and stays allocated until the process exits.  Host code cannot use
// its name as a device address (on the host the name is only a stand-in), so
// its address is looked up with cudaGetSymbolAddress, once per device and
// context, the first time this entry point runs there, with that device
// current.  CUDA loads device code lazily: that lookup is also what places
// this file's module (and the array) on the device, and the same set-up loads
// the routing kernels, so later calls find everything in place.  A new context
// on the device (after cudaDeviceReset) gets a new module and array, so the
// set-up runs again when the current context's id changes.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

// Library-owned routing scratch, shared by every call on a device.
constexpr size_t kScratchBytes = MOE_ROUTE_NO_ALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Device address of g_route_scratch on the current device, set up once per device
// and context: the address lookup (which loads this module) and the routing kernels'
// code.  When the driver cannot tell the context apart (id 0) the set-up repeats.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    moe::record_cuda_error((int)e);
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  const unsigned long long ctx = moe::current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e == cudaSuccess && !p) e = cudaErrorInvalidSymbol;
    if (e == cudaSuccess) e = moe::preload_route_kernels();
    if (e != cudaSuccess) {
      moe::record_cuda_error((int)e);
      return MOE_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = moe::current_context_id();
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_route_no_alloc(const void* scores, int scores_dtype, int64_t stride_t, int64_t stride_e, int T,
                                  int E, int top_k, const int32_t* num_valid_tokens, int32_t* counts,
                                  int32_t* expert_offsets, int32_t* expert_indices, int32_t* token_indices,
                                  int32_t* inv_rows, cudaStream_t stream) {
  size_t need = 0;
  int rc = moe_route_workspace_size(T, E, top_k, &need);
  if (rc != MOE_OK) return rc;
  if (need > kScratchBytes) return MOE_ERR_WORKSPACE;  // larger than the library-owned scratch
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  // The routing kernels write every scratch word before they read it, except the
  // grid-barrier counter of the large-batch kernel, which launch_route zeroes with
  // an asynchronous memset on the stream before that kernel starts; so the previous
  // call's leftovers need no clearing here.
  return moe_route(scores, scores_dtype, stride_t, stride_e, T, E, top_k, num_valid_tokens, counts,
                   expert_offsets, expert_indices, token_indices, inv_rows, nullptr, scratch, kScratchBytes,
                   stream);
}
