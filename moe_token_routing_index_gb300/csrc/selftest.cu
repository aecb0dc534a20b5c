// Self-test of the library's bounded device-side waits: each kernel here waits
// on a condition that never comes true, with the same helpers the pipelines
// use, and must give up after its limit, record MOE_DEVERR_TIMEOUT and return,
// leaving the context usable.  No fault, trap or endless loop is involved.
#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

__device__ unsigned int g_selftest_counter;

// One thread waits on phase 0 of an mbarrier that expects one arrival and gets none.
__global__ void selftest_mbarrier_kernel(uint64_t limit_ns, unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = tc::smem_u32(&bar);
  if (threadIdx.x == 0) {
    tc::mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(b, 0, nullptr, limit_ns)) flag_error(err, MOE_DEVERR_TIMEOUT);
}

// A cooperative grid whose last block never reaches the grid barrier.
__global__ void selftest_grid_kernel(unsigned int* counter, uint64_t limit_ns, unsigned int* err) {
  if (blockIdx.x == gridDim.x - 1) return;
  if (!grid_barrier(counter, gridDim.x, limit_ns) && threadIdx.x == 0) flag_error(err, MOE_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(int which, uint64_t limit_ns, unsigned int* err, cudaStream_t s) {
  if (which == 0) {
    selftest_mbarrier_kernel<<<1, 32, 0, s>>>(limit_ns, err);
    return cudaGetLastError();
  }
  void* counter = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&counter, g_selftest_counter);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(counter, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // both blocks resident: only the skipped arrival is missing
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, selftest_grid_kernel, static_cast<unsigned int*>(counter), limit_ns, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
