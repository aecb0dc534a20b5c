// Internal helpers shared by the kernel translation units of libmoe_gb300.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kNumSmsGB300 = 152;
constexpr float kFp8Max = 448.0f;
constexpr float kFp8Eps = 1e-12f;

// Record a device-side error bit (first writer does not matter: bits are OR-ed).
__device__ __forceinline__ void flag_error(unsigned int* err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

// Read a device int32 count, clamped to [0, hi]; NULL means hi.
__device__ __forceinline__ int read_count(const int32_t* p, int hi, unsigned int* err) {
  if (!p) return hi;
  int v = *p;
  if (v < 0 || v > hi) {
    flag_error(err, MOE_DEVERR_BAD_COUNT);
    v = v < 0 ? 0 : hi;
  }
  return v;
}

// Grid-wide barrier of a cooperative launch: every block arrives once per
// barrier on a counter that starts at 0, so barrier n completes at n * grid
// arrivals.  The wait is bounded (limit_ns of %globaltimer, 1 s by default);
// false means it gave up.  Called by every thread of the block.
__device__ __forceinline__ bool grid_barrier(unsigned int* counter, unsigned int target,
                                             uint64_t limit_ns = 1000000000ull) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(counter, 1u);
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    int ok = 1;
    for (uint32_t i = 0;; ++i) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
      if (v >= target) break;
      if ((i & 63) == 63) {
        uint64_t t1;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (t1 - t0 > limit_ns) {
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Programmatic dependent launch.  launch_dependents: the next kernel of the
// stream may start now (its blocks run their prologue beside this grid);
// wait: block until the previous kernel of the stream has completed and its
// writes are visible.  Both are no-ops in a kernel launched without the
// programmatic-serialization attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Host: the launch attribute that lets a kernel start while the previous one in
// the stream runs (it must pdl_wait() before touching that kernel's results).
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// A routing score; NULL scores read as 1.0 (the gathers then copy rows unscaled).
__device__ __forceinline__ float load_score(const void* scores, int dtype, int64_t off) {
  if (!scores) return 1.0f;
  if (dtype == MOE_DTYPE_F32) return __ldg(reinterpret_cast<const float*>(scores) + off);
  return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(scores) + off));
}

// Monotone map of a score to uint32 (larger score -> larger key), -0 folded onto
// +0: the order in which top-k routing compares scores.
__device__ __forceinline__ uint32_t route_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// 8 bf16 in a uint4 <-> 8 floats.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 p = __bfloat1622float2(h[i]);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float* f) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}

// Two fp32 products, each rounded to nearest even with subnormals kept: one
// packed f32x2 multiply, the same bits as two scalar __fmul_rn.
__device__ __forceinline__ float2 fmul2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 pa, pb, pr;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "mul.rn.f32x2 pr, pa, pb;\n\tmov.b64 {%0, %1}, pr;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// The two bf16 of a packed word as fp32 (low half first): exact widening.
__device__ __forceinline__ float2 bf16x2_bits_to_f32(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Two floats -> two e4m3 codes (round to nearest even, saturating to +-448),
// low byte = a, high byte = b.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// silu(a) * b = (a * sigmoid(a)) * b in fp32, sigmoid(a) = 1 / (1 + e^-a), with
// the hardware exponential and fast division: a few fp32 ulps of error, far
// below one bf16 or e4m3 step of the result.  For a < -87, e^-a overflows to
// +inf and the quotient is 0 (the exact value is below 1e-36).
__device__ __forceinline__ float silu_mul_f32(float a, float b) {
  return __fmul_rn(__fdividef(a, __fadd_rn(1.0f, __expf(-a))), b);
}

// The FP8-rowwise scale rule: m = max|v| clamped to [EPS, ub] (or >= EPS);
// returns s = 448 / m and writes the stored dequantisation scale 1 / s.
// fp8_row_scale_val takes the bound already loaded (has_ub false: no bound).
__device__ __forceinline__ float fp8_row_scale_val(float m, bool has_ub, float ubv, float* inv_out) {
  m = fmaxf(m, kFp8Eps);
  if (has_ub) m = fminf(m, ubv);
  float s = __fdiv_rn(kFp8Max, m);
  *inv_out = __frcp_rn(s);
  return s;
}

__device__ __forceinline__ float fp8_row_scale(float m, const float* ub, float* inv_out) {
  return fp8_row_scale_val(m, ub != nullptr, ub ? __ldg(ub) : 0.0f, inv_out);
}

__device__ __forceinline__ float fp8_scaled_clamped(float v, float s) {
  return fminf(fmaxf(__fmul_rn(v, s), -kFp8Max), kFp8Max);
}

// Max over a warp of non-negative floats (their bit patterns order like the values).
__device__ __forceinline__ float warp_max_nonneg(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

}  // namespace moe
