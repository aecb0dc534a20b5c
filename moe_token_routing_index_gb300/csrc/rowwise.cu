// Row-wise, HBM-bound stages of the routed-expert forward:
//   gather * score            (mslk/moe/gather_scatter.py, _mslk_gather_scale_dense_tokens)
//   gather * score -> FP8     (_mslk_gather_scale_fp8_rowwise_quant_dense_tokens)
//   silu_mul, silu_mul_quant  (mslk/moe/layers.py, MetaShufflingMoE._fused_silu_mul)
//   scatter-add combine       (_mslk_scatter_add_dense_tokens), deterministic
//   per-row FP8 quantisation of weight matrices
//
// Every kernel moves rows in 16-byte vectors (8 bf16 / 16 e4m3 / 4 fp32),
// coalesced across a warp, on a persistent grid of (SMs x 8) 256-thread
// blocks.  Plain stages give one warp a row; quantising stages give one
// block a row, held in registers between the row-max reduction and the
// quantisation, so each input byte is read from HBM once.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBlocksPerSm = 8;
constexpr int kUnroll = 4;

inline int persistent_grid(int64_t work_items, int items_per_block) {
  int64_t need = (work_items + items_per_block - 1) / items_per_block;
  int64_t cap = (int64_t)device_sm_count() * kBlocksPerSm;
  if (need < 1) need = 1;
  return (int)(need < cap ? need : cap);
}

__device__ __forceinline__ int global_warp() { return (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); }
__device__ __forceinline__ int num_warps() { return (int)((gridDim.x * blockDim.x) >> 5); }

// Block-wide max of a non-negative float; every thread gets the result.
__device__ __forceinline__ float block_max_nonneg(float m, float* s_red) {
  m = warp_max_nonneg(m);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
  __syncthreads();
  float r = s_red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = fmaxf(r, s_red[w]);
  return r;
}

// 8 floats -> 8 e4m3 codes (already scaled and clamped), packed little-endian.
__device__ __forceinline__ uint2 e4m3x8(const float* f) {
  uint2 q;
  q.x = f32x2_to_e4m3x2(f[0], f[1]) | (f32x2_to_e4m3x2(f[2], f[3]) << 16);
  q.y = f32x2_to_e4m3x2(f[4], f[5]) | (f32x2_to_e4m3x2(f[6], f[7]) << 16);
  return q;
}

// ------------------------------------------------------------ gather*score

__global__ void __launch_bounds__(kThreads) gather_scale_kernel(
    const uint4* __restrict__ x, int T, int D8, const int32_t* __restrict__ ti, const int32_t* __restrict__ ei,
    int a, const void* __restrict__ scores, int dtype, int64_t st, int64_t se, int E,
    const int32_t* __restrict__ valid_p, uint4* __restrict__ out, unsigned int* err) {
  const int valid = read_count(valid_p, a, err);
  const int lane = threadIdx.x & 31;
  for (int r = global_warp(); r < valid; r += num_warps()) {
    const int t = __ldg(ti + r), e = __ldg(ei + r);
    if ((unsigned)t >= (unsigned)T || (unsigned)e >= (unsigned)E) {
      if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    const float s = load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se);
    const uint4* src = x + (int64_t)t * D8;
    uint4* dst = out + (int64_t)r * D8;
    for (int c0 = lane; c0 < D8; c0 += 32 * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (c0 + 32 * u < D8) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (c0 + 32 * u >= D8) break;
        float f[8];
        bf16x8_to_f32(v[u], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], s);
        dst[c0 + 32 * u] = f32_to_bf16x8(f);
      }
    }
  }
}

// ------------------------------------------------- gather*score -> FP8 row

template <int VPT>  // 16-byte vectors per thread: VPT * 256 >= D / 8
__global__ void __launch_bounds__(kThreads) gather_scale_quant_kernel(
    const uint4* __restrict__ x, int T, int D8, const int32_t* __restrict__ ti, const int32_t* __restrict__ ei,
    int a, const void* __restrict__ scores, int dtype, int64_t st, int64_t se, int E,
    const int32_t* __restrict__ valid_p, const float* __restrict__ ub, uint2* __restrict__ out,
    float* __restrict__ out_scale, unsigned int* err) {
  __shared__ float s_red[kWarps];
  const int valid = read_count(valid_p, a, err);
  for (int r = blockIdx.x; r < valid; r += gridDim.x) {
    const int t = __ldg(ti + r), e = __ldg(ei + r);
    if ((unsigned)t >= (unsigned)T || (unsigned)e >= (unsigned)E) {  // uniform over the block
      if (threadIdx.x == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    const float s = load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se);
    const uint4* src = x + (int64_t)t * D8;
    float f[VPT][8];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + kThreads * i;
      if (c < D8) {
        bf16x8_to_f32(__ldg(src + c), f[i]);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          f[i][q] = __fmul_rn(f[i][q], s);
          m = fmaxf(m, fabsf(f[i][q]));
        }
      }
    }
    m = block_max_nonneg(m, s_red);
    float inv;
    const float sc = fp8_row_scale(m, ub, &inv);
    if (threadIdx.x == 0) out_scale[r] = inv;
    uint2* dst = out + (int64_t)r * D8;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + kThreads * i;
      if (c < D8) {
#pragma unroll
        for (int q = 0; q < 8; ++q) f[i][q] = fp8_scaled_clamped(f[i][q], sc);
        dst[c] = e4m3x8(f[i]);
      }
    }
    __syncthreads();  // s_red is reused by the next row
  }
}

// ---------------------------------------------- weight rows -> FP8 (2 pass)

__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(const float4* __restrict__ w, int64_t rows, int C4,
                                                                 const float* __restrict__ ub,
                                                                 uint32_t* __restrict__ q, float* __restrict__ scale) {
  __shared__ float s_red[kWarps];
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const float4* src = w + r * C4;
    float m = 0.0f;
    for (int c = threadIdx.x; c < C4; c += kThreads) {
      const float4 v = __ldg(src + c);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    m = block_max_nonneg(m, s_red);
    float inv;
    const float sc = fp8_row_scale(m, ub, &inv);
    if (threadIdx.x == 0) scale[r] = inv;
    for (int c = threadIdx.x; c < C4; c += kThreads) {
      const float4 v = __ldg(src + c);
      q[r * C4 + c] = f32x2_to_e4m3x2(fp8_scaled_clamped(v.x, sc), fp8_scaled_clamped(v.y, sc)) |
                      (f32x2_to_e4m3x2(fp8_scaled_clamped(v.z, sc), fp8_scaled_clamped(v.w, sc)) << 16);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- silu_mul

__global__ void __launch_bounds__(kThreads) silu_mul_kernel(const __nv_bfloat16* __restrict__ x0,
                                                            const __nv_bfloat16* __restrict__ x1, int64_t ld, int a,
                                                            int H8, const int32_t* __restrict__ valid_p,
                                                            uint4* __restrict__ z, unsigned int* err) {
  const int valid = read_count(valid_p, a, err);
  const int lane = threadIdx.x & 31;
  for (int r = global_warp(); r < valid; r += num_warps()) {
    const uint4* p0 = reinterpret_cast<const uint4*>(x0 + (int64_t)r * ld);
    const uint4* p1 = reinterpret_cast<const uint4*>(x1 + (int64_t)r * ld);
    uint4* dst = z + (int64_t)r * H8;
    for (int c0 = lane; c0 < H8; c0 += 32 * kUnroll) {
      uint4 v0[kUnroll], v1[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (c0 + 32 * u < H8) {
          v0[u] = __ldg(p0 + c0 + 32 * u);
          v1[u] = __ldg(p1 + c0 + 32 * u);
        }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (c0 + 32 * u >= H8) break;
        float f0[8], f1[8];
        bf16x8_to_f32(v0[u], f0);
        bf16x8_to_f32(v1[u], f1);
#pragma unroll
        for (int i = 0; i < 8; ++i) f0[i] = silu_mul_f32(f0[i], f1[i]);
        dst[c0 + 32 * u] = f32_to_bf16x8(f0);
      }
    }
  }
}

template <int VPT>
__global__ void __launch_bounds__(kThreads) silu_mul_quant_kernel(const __nv_bfloat16* __restrict__ x0,
                                                                  const __nv_bfloat16* __restrict__ x1, int64_t ld,
                                                                  int a, int H8, const int32_t* __restrict__ valid_p,
                                                                  const float* __restrict__ ub, uint2* __restrict__ z,
                                                                  float* __restrict__ z_scale, unsigned int* err) {
  __shared__ float s_red[kWarps];
  const int valid = read_count(valid_p, a, err);
  for (int r = blockIdx.x; r < valid; r += gridDim.x) {
    const uint4* p0 = reinterpret_cast<const uint4*>(x0 + (int64_t)r * ld);
    const uint4* p1 = reinterpret_cast<const uint4*>(x1 + (int64_t)r * ld);
    float f[VPT][8];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + kThreads * i;
      if (c < H8) {
        float g[8];
        bf16x8_to_f32(__ldg(p0 + c), f[i]);
        bf16x8_to_f32(__ldg(p1 + c), g);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          f[i][q] = silu_mul_f32(f[i][q], g[q]);
          m = fmaxf(m, fabsf(f[i][q]));
        }
      }
    }
    m = block_max_nonneg(m, s_red);
    float inv;
    const float sc = fp8_row_scale(m, ub, &inv);
    if (threadIdx.x == 0) z_scale[r] = inv;
    uint2* dst = z + (int64_t)r * H8;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + kThreads * i;
      if (c < H8) {
#pragma unroll
        for (int q = 0; q < 8; ++q) f[i][q] = fp8_scaled_clamped(f[i][q], sc);
        dst[c] = e4m3x8(f[i]);
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------- scatter-add

// top_k == 1 without the inverse permutation: routed row r owns token ti[r].
template <bool ACC>
__global__ void __launch_bounds__(kThreads) scatter_add_rows_kernel(uint4* __restrict__ out,
                                                                    const uint4* __restrict__ in,
                                                                    const int32_t* __restrict__ ti, int a, int T,
                                                                    int D8, const int32_t* __restrict__ valid_p,
                                                                    unsigned int* err) {
  const int valid = read_count(valid_p, a, err);
  const int lane = threadIdx.x & 31;
  for (int r = global_warp(); r < valid; r += num_warps()) {
    const int t = __ldg(ti + r);
    if ((unsigned)t >= (unsigned)T) {
      if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    uint4* o = out + (int64_t)t * D8;
    const uint4* src = in + (int64_t)r * D8;
    for (int c0 = lane; c0 < D8; c0 += 32 * kUnroll) {
      uint4 vo[kUnroll], vi[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (c0 + 32 * u < D8) {
          if (ACC) vo[u] = o[c0 + 32 * u];
          vi[u] = __ldg(src + c0 + 32 * u);
        }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (c0 + 32 * u >= D8) break;
        if (ACC) {
          float fo[8], fi[8];
          bf16x8_to_f32(vo[u], fo);
          bf16x8_to_f32(vi[u], fi);
#pragma unroll
          for (int i = 0; i < 8; ++i) fo[i] = __fadd_rn(fo[i], fi[i]);
          o[c0 + 32 * u] = f32_to_bf16x8(fo);
        } else {
          o[c0 + 32 * u] = vi[u];  // bf16(0 + x) = x
        }
      }
    }
  }
}

// With the inverse permutation: one warp owns token t and adds its top_k rows
// in ascending row order into an fp32 accumulator started from out[t] (ACC)
// or from zero.
template <bool ACC>
__global__ void __launch_bounds__(kThreads) scatter_add_tokens_kernel(uint4* __restrict__ out,
                                                                      const uint4* __restrict__ in,
                                                                      const int32_t* __restrict__ inv, int k, int a,
                                                                      int T, int D8,
                                                                      const int32_t* __restrict__ valid_p,
                                                                      unsigned int* err) {
  const int valid = read_count(valid_p, a, err);
  if (valid % k != 0 && blockIdx.x == 0 && threadIdx.x == 0) flag_error(err, MOE_DEVERR_BAD_COUNT);
  int Tv = valid / k;
  if (Tv > T) Tv = T;
  const int lane = threadIdx.x & 31;
  for (int t = global_warp(); t < Tv; t += num_warps()) {
    int my_row = 0;
    bool bad = false;
    if (lane < k) {
      my_row = __ldg(inv + (int64_t)t * k + lane);
      bad = (unsigned)my_row >= (unsigned)a;
    }
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    uint4* o = out + (int64_t)t * D8;
    for (int c0 = lane; c0 < D8; c0 += 32 * 2) {
      float acc[2][8];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (ACC && c0 + 32 * u < D8) {
          bf16x8_to_f32(o[c0 + 32 * u], acc[u]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
        }
      }
      for (int j = 0; j < k; ++j) {
        const int r = (j < 32) ? __shfl_sync(0xffffffffu, my_row, j) : __ldg(inv + (int64_t)t * k + j);
        if ((unsigned)r >= (unsigned)a) {  // only reachable for top_k > 32
          flag_error(err, MOE_DEVERR_BAD_INDEX);
          continue;
        }
        const uint4* src = in + (int64_t)r * D8;
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (c0 + 32 * u < D8) {
            float fi[8];
            bf16x8_to_f32(__ldg(src + c0 + 32 * u), fi);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[u][i] = __fadd_rn(acc[u][i], fi[i]);
          }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (c0 + 32 * u < D8) o[c0 + 32 * u] = f32_to_bf16x8(acc[u]);
    }
  }
}

}  // namespace

cudaError_t launch_gather_scale(const GatherArgs& g, cudaStream_t s) {
  const int grid = persistent_grid(g.a, kWarps);
  gather_scale_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint4*>(g.x), g.T, g.D / 8, g.token_indices,
                                                g.expert_indices, g.a, g.scores, g.dtype, g.stride_t, g.stride_e,
                                                g.E, g.valid, static_cast<uint4*>(g.out), g.err);
  return cudaGetLastError();
}

#define MOE_GATHER_QUANT(VPT)                                                                                     \
  gather_scale_quant_kernel<VPT><<<grid, kThreads, 0, s>>>(                                                      \
      static_cast<const uint4*>(g.x), g.T, D8, g.token_indices, g.expert_indices, g.a, g.scores, g.dtype,         \
      g.stride_t, g.stride_e, g.E, g.valid, g.scale_ub, static_cast<uint2*>(g.out), g.out_scale, g.err)

cudaError_t launch_gather_scale_quant(const GatherArgs& g, cudaStream_t s) {
  const int D8 = g.D / 8;
  const int vpt = (D8 + kThreads - 1) / kThreads;
  const int grid = persistent_grid(g.a, 1);
  if (vpt <= 1) MOE_GATHER_QUANT(1);
  else if (vpt <= 2) MOE_GATHER_QUANT(2);
  else if (vpt <= 3) MOE_GATHER_QUANT(3);
  else if (vpt <= 4) MOE_GATHER_QUANT(4);
  else if (vpt <= 6) MOE_GATHER_QUANT(6);
  else MOE_GATHER_QUANT(8);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const float* w, int64_t rows, int cols, const float* ub, void* q, float* scale,
                                 cudaStream_t s) {
  const int grid = persistent_grid(rows, 1);
  quantize_rows_kernel<<<grid, kThreads, 0, s>>>(reinterpret_cast<const float4*>(w), rows, cols / 4, ub,
                                                 static_cast<uint32_t*>(q), scale);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul(const SiluArgs& g, cudaStream_t s) {
  const int grid = persistent_grid(g.a, kWarps);
  silu_mul_kernel<<<grid, kThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(g.x0),
                                            static_cast<const __nv_bfloat16*>(g.x1), g.ld, g.a, g.H / 8, g.valid,
                                            static_cast<uint4*>(g.z), g.err);
  return cudaGetLastError();
}

#define MOE_SILU_QUANT(VPT)                                                                                        \
  silu_mul_quant_kernel<VPT><<<grid, kThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(g.x0),                 \
                                                       static_cast<const __nv_bfloat16*>(g.x1), g.ld, g.a, H8,    \
                                                       g.valid, g.scale_ub, static_cast<uint2*>(g.z), g.z_scale, \
                                                       g.err)

cudaError_t launch_silu_mul_quant(const SiluArgs& g, cudaStream_t s) {
  const int H8 = g.H / 8;
  const int vpt = (H8 + kThreads - 1) / kThreads;
  const int grid = persistent_grid(g.a, 1);
  if (vpt <= 1) MOE_SILU_QUANT(1);
  else if (vpt <= 2) MOE_SILU_QUANT(2);
  else if (vpt <= 3) MOE_SILU_QUANT(3);
  else if (vpt <= 4) MOE_SILU_QUANT(4);
  else if (vpt <= 6) MOE_SILU_QUANT(6);
  else MOE_SILU_QUANT(8);
  return cudaGetLastError();
}

cudaError_t launch_scatter_add(const ScatterArgs& g, cudaStream_t s) {
  const int D8 = g.D / 8;
  if (g.inv) {
    const int grid = persistent_grid(g.T, kWarps);
    auto k = g.accumulate ? scatter_add_tokens_kernel<true> : scatter_add_tokens_kernel<false>;
    k<<<grid, kThreads, 0, s>>>(static_cast<uint4*>(g.out), static_cast<const uint4*>(g.in), g.inv, g.top_k, g.a,
                                g.T, D8, g.valid, g.err);
  } else {
    const int grid = persistent_grid(g.a, kWarps);
    auto k = g.accumulate ? scatter_add_rows_kernel<true> : scatter_add_rows_kernel<false>;
    k<<<grid, kThreads, 0, s>>>(static_cast<uint4*>(g.out), static_cast<const uint4*>(g.in), g.token_indices, g.a,
                                g.T, D8, g.valid, g.err);
  }
  return cudaGetLastError();
}

}  // namespace moe
