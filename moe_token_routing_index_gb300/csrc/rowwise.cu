// Row-wise, HBM-bound stages of the routed-expert forward:
//   gather * score            (mslk/moe/gather_scatter.py, _mslk_gather_scale_dense_tokens)
//   gather * score -> FP8     (_mslk_gather_scale_fp8_rowwise_quant_dense_tokens)
//   silu_mul, silu_mul_quant  (mslk/moe/layers.py, MetaShufflingMoE._fused_silu_mul)
//   scatter-add combine       (_mslk_scatter_add_dense_tokens), deterministic
//   per-row FP8 quantisation of weight matrices
//
// Every kernel moves rows in 16-byte vectors (8 bf16 / 16 e4m3 / 4 fp32),
// coalesced across a warp, on a persistent grid sized to the blocks the SMs
// hold at once.  Plain stages give a warp (row, chunk) items; the register
// quantising stages give a group of 1-8 warps a row, held in registers between
// the row-max reduction and the quantisation.  The staged gathers (one block of
// 8-16 warps per SM) copy whole x rows into shared memory with bulk copies.
// Each input byte is read from HBM once.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;
constexpr int kChunk = 32 * kUnroll;  // 16-byte vectors per work item of the plain row kernels

// Grid of a persistent kernel: as many blocks as fit on the device at once
// (SMs x resident blocks per SM of this kernel), or fewer when there is less
// work, so every block stays resident and walks a long run of rows.
template <typename Kernel>
int persistent_grid(Kernel kernel, int64_t work_items, int items_per_block) {
  int64_t need = (work_items + items_per_block - 1) / items_per_block;
  int64_t cap = (int64_t)device_sm_count() * resident_blocks_per_sm(reinterpret_cast<const void*>(kernel), kThreads);
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

// Barrier over the `nthreads` threads of one row group (ids 1..8; 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Max of a non-negative float over the G warps of a row group; every thread of
// the group gets the result.  s_red holds one slot per warp of the block.
template <int G>
__device__ __forceinline__ float group_max_nonneg(float m, float* s_red, int group) {
  m = warp_max_nonneg(m);
  if constexpr (G == 1) {
    return m;
  } else {
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) s_red[warp] = m;
    group_sync(1 + group, 32 * G);
    float r = s_red[group * G];
#pragma unroll
    for (int w = 1; w < G; ++w) r = fmaxf(r, s_red[group * G + w]);
    return r;
  }
}

// 8 floats -> 8 e4m3 codes (already scaled and clamped), packed little-endian.
__device__ __forceinline__ uint2 e4m3x8(const float* f) {
  uint2 q;
  q.x = f32x2_to_e4m3x2(f[0], f[1]) | (f32x2_to_e4m3x2(f[2], f[3]) << 16);
  q.y = f32x2_to_e4m3x2(f[4], f[5]) | (f32x2_to_e4m3x2(f[6], f[7]) << 16);
  return q;
}

// ------------------------------------------------------------ gather*score

// Work item = (routed row, chunk of 32 lanes x kGatherUnroll vectors);
// consecutive items are consecutive chunks of a row, spread over all warps of
// the grid.  The indices of a warp's next item are loaded one item ahead.
constexpr int kGatherUnroll = 8;
constexpr int kGatherChunk = 32 * kGatherUnroll;

__global__ void __launch_bounds__(kThreads) gather_scale_kernel(
    const uint4* __restrict__ x, int T, int D8, const int32_t* __restrict__ ti, const int32_t* __restrict__ ei,
    int a, const void* __restrict__ scores, int dtype, int64_t st, int64_t se, int E,
    const int32_t* __restrict__ valid_p, uint4* __restrict__ out, unsigned int* err) {
  pdl_wait();  // launched while the routing kernel runs: its output is visible from here
  const int valid = read_count(valid_p, a, err);
  const int lane = threadIdx.x & 31;
  const int chunks = (D8 + kGatherChunk - 1) / kGatherChunk;
  const int64_t items = (int64_t)valid * chunks;
  const int64_t step = num_warps();
  int64_t it = global_warp();
  int t = 0, e = 0;
  if (it < items) {
    const int r = (int)(it / chunks);
    t = __ldg(ti + r);
    e = __ldg(ei + r);
  }
  for (; it < items; it += step) {
    const int r = (int)(it / chunks);
    const int c0 = (int)(it - (int64_t)r * chunks) * kGatherChunk + lane;
    const int ct = t, ce = e;
    if (it + step < items) {  // next item's indices
      const int rn = (int)((it + step) / chunks);
      t = __ldg(ti + rn);
      e = __ldg(ei + rn);
    }
    // the expert index only addresses the scores (NULL scores: every score is 1)
    if ((unsigned)ct >= (unsigned)T || (scores && (unsigned)ce >= (unsigned)E)) {
      if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    const float s = load_score(scores, dtype, (int64_t)ct * st + (int64_t)ce * se);
    const uint4* src = x + (int64_t)ct * D8;
    uint4* dst = out + (int64_t)r * D8;
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u)
      if (c0 + 32 * u < D8) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      if (c0 + 32 * u >= D8) break;
      float f[8];
      bf16x8_to_f32(v[u], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], s);
      dst[c0 + 32 * u] = f32_to_bf16x8(f);
    }
  }
}

// ------------------------------------------------- gather*score -> FP8 row
//
// A row group of G warps owns one routed row at a time: the fp32 row v = x * s
// stays in registers (VPT 16-byte vectors per thread, G * 32 * VPT >= D / 8),
// the group reduces max|v| (warp shuffles, then one named barrier when G > 1),
// and quantises.  As soon as the current row has been expanded to fp32, the
// packed input of the group's next row is loaded into the freed registers, so
// those loads are in flight while the current row is reduced, quantised and
// stored.  The 8 / G groups of a block walk their rows independently.

template <int G, int VPT>
__global__ void __launch_bounds__(kThreads) gather_scale_quant_kernel(
    const uint4* __restrict__ x, int T, int D8, const int32_t* __restrict__ ti, const int32_t* __restrict__ ei,
    int a, const void* __restrict__ scores, int dtype, int64_t st, int64_t se, int E,
    const int32_t* __restrict__ valid_p, const float* __restrict__ ub, uint2* __restrict__ out,
    float* __restrict__ out_scale, unsigned int* err) {
  constexpr int kGroupThreads = 32 * G, kGroups = kThreads / kGroupThreads;
  __shared__ float s_red[kWarps];
  const int valid = read_count(valid_p, a, err);
  const int group = threadIdx.x / kGroupThreads, gt = threadIdx.x % kGroupThreads;
  const int stride = gridDim.x * kGroups;
  // Software pipeline: the indices of row r + 2*stride and the data of row
  // r + stride are in flight while row r is reduced, quantised and stored.
  uint4 raw[VPT];
  float s = 0.0f;
  bool ok = false;
  int nt = 0, ne = 0;  // indices of the next row
  auto fetch_data = [&](int t, int e) {
    ok = (unsigned)t < (unsigned)T && (!scores || (unsigned)e < (unsigned)E);
    if (ok) {
      s = load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se);
      const uint4* src = x + (int64_t)t * D8;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int c = gt + kGroupThreads * i;
        if (c < D8) raw[i] = __ldg(src + c);
      }
    }
  };
  int r = blockIdx.x * kGroups + group;
  if (r < valid) fetch_data(__ldg(ti + r), __ldg(ei + r));
  if (r + stride < valid) {
    nt = __ldg(ti + r + stride);
    ne = __ldg(ei + r + stride);
  }
  for (; r < valid; r += stride) {
    const bool cur_ok = ok;  // uniform over the group
    float f[VPT][8];
    float m = 0.0f;
    if (cur_ok) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int c = gt + kGroupThreads * i;
        if (c < D8) {
          bf16x8_to_f32(raw[i], f[i]);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            f[i][q] = __fmul_rn(f[i][q], s);
            m = fmaxf(m, fabsf(f[i][q]));
          }
        }
      }
    }
    if (r + stride < valid) fetch_data(nt, ne);
    if (r + 2 * stride < valid) {
      nt = __ldg(ti + r + 2 * stride);
      ne = __ldg(ei + r + 2 * stride);
    }
    if (!cur_ok) {
      if (gt == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    m = group_max_nonneg<G>(m, s_red, group);
    float inv;
    const float sc = fp8_row_scale(m, ub, &inv);
    if (gt == 0) out_scale[r] = inv;
    uint2* dst = out + (int64_t)r * D8;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = gt + kGroupThreads * i;
      if (c < D8) {
#pragma unroll
        for (int q = 0; q < 8; ++q) f[i][q] = fp8_scaled_clamped(f[i][q], sc);
        dst[c] = e4m3x8(f[i]);
      }
    }
    if constexpr (G > 1) group_sync(1 + group, kGroupThreads);  // s_red is reused by the next row
  }
}

// ----------------------------------- gather*score -> FP8, TMA-staged rows
//
// Each warp owns a ring of NB row slots in shared memory.  Lane 0 reads the
// row's token index and issues one bulk copy (cp.async.bulk, completion on
// the slot's mbarrier) of the whole x row into a slot; the warp then makes two
// passes over the staged row (max |x * s|, then scale, quantise and store) and
// hands the slot to the row NB ahead.  Rows in flight per SM = warps x NB, with
// almost no registers, and each x byte crosses HBM once.

__device__ __forceinline__ uint64_t global_timer_ns_rw() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool bar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait (1 s) for the phase with `parity` to complete.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  if (bar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns_rw();
  for (uint32_t i = 1;; ++i) {
    if (bar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0 && global_timer_ns_rw() - t0 > 1000000000ull) return false;
  }
}

// One bulk copy of `bytes` (multiple of 16, 16-byte aligned) global -> shared, tracked by `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

constexpr int kStagedMaxWarps = 16;  // the launch picks 8..16 warps per block

// Largest |bf16| of 8 packed values, as bf16 magnitude bits (the magnitude
// bits of a bf16 order like its absolute value), folded into `m`.
__device__ __forceinline__ uint32_t absmax_bits8(const uint4& v, uint32_t m) {
  uint32_t a = __vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu);
  uint32_t b = __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu);
  a = __vmaxu2(a, b);
  return max(m, max(a & 0xffffu, a >> 16));
}

// Items of the staged gather: row-major (item = routed row r, its token
// ti[r], one output row) or token-major (item = valid token t, its top_k
// routed rows inv[t*k .. t*k+k), so the staged x row serves all of them).
//
// Per warp: a ring of NB slots, each holding one staged x row (one bulk copy,
// completion on the slot's mbarrier).  The routed rows' metadata (row index
// and score) is loaded for 32 rows at a time, one row per lane, so the
// dependent index loads cost one round trip per 32 rows.  For the FP8 output
// the row max uses max |RN(x * s)| = RN(max |x| * |s|) (rounding is
// monotone), taken as an integer max over the packed bf16 magnitudes; the
// clamp to +-448 is the saturation of the e4m3 conversion itself.
template <bool QUANT>
__global__ void __launch_bounds__(kStagedMaxWarps * 32, 1) gather_staged_kernel(
    const uint4* __restrict__ x, int T, int D8, const int32_t* __restrict__ ti, const int32_t* __restrict__ ei,
    const int32_t* __restrict__ inv, int k, int a, const void* __restrict__ scores, int dtype, int64_t st,
    int64_t se, int E, const int32_t* __restrict__ valid_p, const float* __restrict__ ub, void* __restrict__ out,
    float* __restrict__ out_scale, int NB, unsigned int* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwb = blockDim.x >> 5;
  const uint32_t row_bytes = (uint32_t)D8 * 16u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);                      // [warps][NB]
  int* s_tok = reinterpret_cast<int*>(smem + nwb * NB * 8);                // [warps][NB]: staged token or -1
  uint8_t* slots = smem + ((nwb * NB * 16 + 127) / 128) * 128;             // [warps][NB][row_bytes]
  pdl_wait();  // launched while the routing kernel runs: its output is visible from here
  const int valid = read_count(valid_p, a, err);
  const int nrows = inv ? k : 1;  // routed rows per item
  int items = valid;
  if (inv) {
    if (valid % k != 0 && blockIdx.x == 0 && threadIdx.x == 0) flag_error(err, MOE_DEVERR_BAD_COUNT);
    items = min(valid / k, T);
  }
  // warps numbered SM-fastest, so a partial last round of items spreads over all blocks
  const int gw = warp * gridDim.x + blockIdx.x, nw = gridDim.x * nwb;
  auto bar_addr = [&](int b) { return (uint32_t)__cvta_generic_to_shared(&bars[warp * NB + b]); };
  auto slot = [&](int b) { return slots + (size_t)(warp * NB + b) * row_bytes; };
  if (lane == 0)
    for (int b = 0; b < NB; ++b) bar_init(bar_addr(b), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  // lane 0: the token of `item`, and one bulk copy of its x row into slot b
  auto issue = [&](int item, int b) {
    const int t = inv ? item : __ldg(ti + item);
    const bool ok = (unsigned)t < (unsigned)T;
    s_tok[warp * NB + b] = ok ? t : -1;
    if (ok) bulk_load((uint32_t)__cvta_generic_to_shared(slot(b)), x + (int64_t)t * D8, row_bytes, bar_addr(b));
  };
  // metadata of routed-row number q of this warp (item q / nrows, its row q % nrows): lane L holds q = base + L
  int meta_base = -32;
  int m_row = -1;
  float m_s = 0.0f;
  auto load_meta = [&](int base) {
    meta_base = base;
    const int q = base + lane;
    const int i = q / nrows, j = q - (q / nrows) * nrows;
    const int item = gw + i * nw;
    m_row = -1;
    if (item < items) {
      const int r = inv ? __ldg(inv + (int64_t)item * k + j) : item;
      const int t = inv ? item : __ldg(ti + item);
      const int e = (unsigned)r < (unsigned)a ? __ldg(ei + r) : -1;
      if ((unsigned)r < (unsigned)a && (!scores || (unsigned)e < (unsigned)E) && (unsigned)t < (unsigned)T) {
        m_row = r;
        m_s = load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se);
      }
    }
  };
  // the first item's row copy, then its metadata (ahead of the other slots' copies in the memory queues)
  if (lane == 0 && gw < items) issue(gw, 0);
  __syncwarp();
  load_meta(0);
  if (lane == 0)
    for (int b = 1; b < NB; ++b)
      if (gw + b * nw < items) issue(gw + b * nw, b);
  __syncwarp();
  const float ubv = (QUANT && ub) ? __ldg(ub) : 0.0f;
  uint32_t phase = 0;  // bit b: parity of the next completion of slot b
  int i = 0;
  bool timed_out = false;
  for (;; ++i) {
    const int item = gw + i * nw;
    if (item >= items) break;
    const int b = i % NB;
    const int t = s_tok[warp * NB + b];
    if (t >= 0) {
      if (!bar_wait(bar_addr(b), (phase >> b) & 1u)) {
        timed_out = true;
        break;
      }
      phase ^= 1u << b;
      const uint4* row = reinterpret_cast<const uint4*>(slot(b));
      // the item's rows in one metadata window (nrows <= 32); lane j < nrows takes row j
      if (i * nrows + nrows > meta_base + 32) load_meta(i * nrows);
      const int src = i * nrows - meta_base + min(lane, nrows - 1);
      const int r_l = __shfl_sync(0xffffffffu, m_row, src);
      const float s_l = __shfl_sync(0xffffffffu, m_s, src);
      float sc_l = 0.0f;
      if constexpr (QUANT) {  // the row's largest |x|, shared by all of its routed rows
        uint32_t mx = 0;
        for (int c = lane; c < D8; c += 32) mx = absmax_bits8(row[c], mx);
        mx = __reduce_max_sync(0xffffffffu, mx);
        // the rows' scales side by side, one per lane: max_j |x_j * s| = RN(max|x| * |s|)
        float inv_s;
        sc_l = fp8_row_scale_val(__fmul_rn(__uint_as_float(mx << 16), fabsf(s_l)), ub != nullptr, ubv, &inv_s);
        if (lane < nrows && r_l >= 0) out_scale[r_l] = inv_s;
      }
      for (int j = 0; j < nrows; ++j) {
        const int r = __shfl_sync(0xffffffffu, r_l, j);
        const float s = __shfl_sync(0xffffffffu, s_l, j);
        if (r < 0) {
          if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
          continue;
        }
        if constexpr (QUANT) {
          const float sc = __shfl_sync(0xffffffffu, sc_l, j);
          uint2* dst = static_cast<uint2*>(out) + (int64_t)r * D8;
          const float2 s2 = make_float2(s, s), sc2 = make_float2(sc, sc);
#pragma unroll 8
          for (int c = lane; c < D8; c += 32) {
            const uint4 v = row[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t q[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {  // RN(RN(x * s) * sc), two lanes per multiply
              const float2 p = fmul2_rn(fmul2_rn(bf16x2_bits_to_f32(w[h]), s2), sc2);
              q[h] = f32x2_to_e4m3x2(p.x, p.y);  // saturating conversion = the clamp to +-448
            }
            dst[c] = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
          }
        } else {
          uint4* dst = static_cast<uint4*>(out) + (int64_t)r * D8;
          const float2 s2 = make_float2(s, s);
#pragma unroll 8
          for (int c = lane; c < D8; c += 32) {
            const uint4 v = row[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float2 p = fmul2_rn(bf16x2_bits_to_f32(w[h]), s2);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(p.x, p.y);
              o[h] = *reinterpret_cast<uint32_t*>(&b2);
            }
            dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    } else {
      if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
    }
    // the slot's reads (generic proxy) finish before the next bulk copy (async proxy) writes it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0 && item + NB * nw < items) issue(item + NB * nw, b);
    __syncwarp();
  }
  // On a normal exit every issued copy has been consumed (a copy is issued only
  // for an item below `items`, and the loop waits on every such item).  After a
  // timeout, the copies of iterations i .. i+NB-1 may still be in flight: wait
  // for them (bounded) so none lands after the block has exited.
  if (timed_out && lane == 0) {
    flag_error(err, MOE_DEVERR_TIMEOUT);
    for (int j = i; j < i + NB; ++j) {
      const int b = j % NB;
      if (gw + j * nw < items && s_tok[warp * NB + b] >= 0) {
        const uint64_t t0 = global_timer_ns_rw();
        while (!bar_try_wait(bar_addr(b), (phase >> b) & 1u) && global_timer_ns_rw() - t0 < 100000000ull) {
        }
      }
    }
  }
}

// Shape of the staged gather for rows of D8 16-byte vectors: warps per block
// (8..16) and row slots per warp (2..4), within 226 of the 227 KB of shared
// memory a block may hold (the rest: barriers and token slots), and
// with at least two slots per warp (one row consumed while the next lands).
// More warps first: the consume loop needs issue slots more than it needs
// deeper per-warp prefetch.  {0, 0}: two slots of 8 warps do not fit.
struct StagedShape {
  int warps, slots;
};
inline StagedShape staged_shape(int D8) {
  const size_t row_bytes = (size_t)D8 * 16, budget = 226u * 1024u;
  const int warps = (int)std::min<size_t>(kStagedMaxWarps, budget / (2 * row_bytes));
  if (warps < 8) return {0, 0};
  return {warps, (int)std::min<size_t>(4, budget / (warps * row_bytes))};
}

template <bool QUANT>
cudaError_t launch_staged(const GatherArgs& g, StagedShape sh, cudaStream_t s) {
  const int D8 = g.D / 8, nb = sh.slots;
  const size_t row_bytes = (size_t)D8 * 16;
  const size_t smem = (size_t)((sh.warps * nb * 16 + 127) / 128) * 128 + (size_t)sh.warps * nb * row_bytes;
  auto kern = gather_staged_kernel<QUANT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t items = g.inv ? std::min<int64_t>(g.a / g.top_k, g.T) : g.a;
  const int64_t need = (items + sh.warps - 1) / sh.warps;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, device_sm_count()));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(sh.warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};  // may start while the router's kernel runs
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint4*>(g.x), g.T, D8, g.token_indices, g.expert_indices,
                         g.inv, g.top_k, g.a, g.scores, g.dtype, g.stride_t, g.stride_e, g.E, g.valid, g.scale_ub,
                         g.out, g.out_scale, nb, g.err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
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

// The number of valid routed rows: *valid_p (clamped to a), or, when sum_counts is
// given, the sum of the E per-expert counts (the padded-token layout, whose valid
// rows are every expert's rows).  Called by every thread of the block.
__device__ int valid_rows(const int32_t* valid_p, const int32_t* sum_counts, int E, int a, unsigned int* err) {
  if (!sum_counts) return read_count(valid_p, a, err);
  __shared__ int s_rows;
  if (threadIdx.x < 32) {
    int v = 0;
    bool bad = false;
    for (int e = threadIdx.x; e < E; e += 32) {
      const int c = __ldg(sum_counts + e);
      bad |= c < 0;
      v += c > 0 ? c : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    bad = __any_sync(0xffffffffu, bad);
    if (threadIdx.x == 0) {
      if (bad || v > a) {
        if (blockIdx.x == 0) flag_error(err, MOE_DEVERR_BAD_COUNT);
        if (v > a) v = a;
      }
      s_rows = v;
    }
  }
  __syncthreads();
  return s_rows;
}

// ---------------------------------------------------------------- silu_mul

__global__ void __launch_bounds__(kThreads) silu_mul_kernel(const __nv_bfloat16* __restrict__ x0,
                                                            const __nv_bfloat16* __restrict__ x1, int64_t ld, int a,
                                                            int H8, const int32_t* __restrict__ valid_p,
                                                            uint4* __restrict__ z, unsigned int* err) {
  const int valid = read_count(valid_p, a, err);
  const int lane = threadIdx.x & 31;
  const int chunks = (H8 + kChunk - 1) / kChunk;
  const int64_t items = (int64_t)valid * chunks;
  for (int64_t it = global_warp(); it < items; it += num_warps()) {
    const int r = (int)(it / chunks);
    const int c0 = (int)(it - (int64_t)r * chunks) * kChunk + lane;
    const uint4* p0 = reinterpret_cast<const uint4*>(x0 + (int64_t)r * ld);
    const uint4* p1 = reinterpret_cast<const uint4*>(x1 + (int64_t)r * ld);
    uint4* dst = z + (int64_t)r * H8;
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

// Row groups as in the quantising gather; the fp32 row of z is held in
// registers and the next row's packed input is prefetched.  SILU: z =
// silu_mul(x0, x1) (silu_mul_quant); otherwise z = x0, a bf16 row (the row pass
// of the grouped GEMM's SILU_MUL_QUANT epilogue; x1 unused).  The valid row
// count is *valid_p, or the sum of the E counts when sum_counts is given.
template <int G, int VPT, bool SILU>
__global__ void __launch_bounds__(kThreads) silu_mul_quant_kernel(const __nv_bfloat16* __restrict__ x0,
                                                                  const __nv_bfloat16* __restrict__ x1, int64_t ld,
                                                                  int a, int H8, const int32_t* __restrict__ valid_p,
                                                                  const int32_t* __restrict__ sum_counts, int E,
                                                                  const float* __restrict__ ub, uint2* __restrict__ z,
                                                                  float* __restrict__ z_scale, unsigned int* err) {
  constexpr int kGroupThreads = 32 * G, kGroups = kThreads / kGroupThreads;
  __shared__ float s_red[kWarps];
  const int valid = valid_rows(valid_p, sum_counts, E, a, err);
  const int group = threadIdx.x / kGroupThreads, gt = threadIdx.x % kGroupThreads;
  const int stride = gridDim.x * kGroups;
  uint4 r0[VPT], r1[SILU ? VPT : 1];
  auto fetch = [&](int row) {
    const uint4* p0 = reinterpret_cast<const uint4*>(x0 + (int64_t)row * ld);
    const uint4* p1 = reinterpret_cast<const uint4*>(x1 + (int64_t)row * ld);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = gt + kGroupThreads * i;
      if (c < H8) {
        r0[i] = __ldg(p0 + c);
        if constexpr (SILU) r1[i] = __ldg(p1 + c);
      }
    }
  };
  int r = blockIdx.x * kGroups + group;
  if (r < valid) fetch(r);
  for (; r < valid; r += stride) {
    float f[VPT][8];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = gt + kGroupThreads * i;
      if (c < H8) {
        bf16x8_to_f32(r0[i], f[i]);
        if constexpr (SILU) {
          float g[8];
          bf16x8_to_f32(r1[i], g);
#pragma unroll
          for (int q = 0; q < 8; ++q) f[i][q] = silu_mul_f32(f[i][q], g[q]);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(f[i][q]));
      }
    }
    if (r + stride < valid) fetch(r + stride);
    m = group_max_nonneg<G>(m, s_red, group);
    float inv;
    const float sc = fp8_row_scale(m, ub, &inv);
    if (gt == 0) z_scale[r] = inv;
    uint2* dst = z + (int64_t)r * H8;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = gt + kGroupThreads * i;
      if (c < H8) {
#pragma unroll
        for (int q = 0; q < 8; ++q) f[i][q] = fp8_scaled_clamped(f[i][q], sc);
        dst[c] = e4m3x8(f[i]);
      }
    }
    if constexpr (G > 1) group_sync(1 + group, kGroupThreads);
  }
}

// ------------------------------------------------------------- scatter-add

// top_k == 1 without the inverse permutation: routed row r owns token ti[r].
// Work items as in the gather: (row, chunk).
template <bool ACC>
__global__ void __launch_bounds__(kThreads) scatter_add_rows_kernel(uint4* __restrict__ out,
                                                                    const uint4* __restrict__ in,
                                                                    const int32_t* __restrict__ ti, int a, int T,
                                                                    int D8, const int32_t* __restrict__ valid_p,
                                                                    const int32_t* __restrict__ sum_counts, int E,
                                                                    unsigned int* err) {
  const int valid = valid_rows(valid_p, sum_counts, E, a, err);
  const int lane = threadIdx.x & 31;
  const int chunks = (D8 + kChunk - 1) / kChunk;
  const int64_t items = (int64_t)valid * chunks;
  for (int64_t it = global_warp(); it < items; it += num_warps()) {
    const int r = (int)(it / chunks);
    const int c0 = (int)(it - (int64_t)r * chunks) * kChunk + lane;
    const int t = __ldg(ti + r);
    if ((unsigned)t >= (unsigned)T) {
      if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    uint4* o = out + (int64_t)t * D8;
    const uint4* src = in + (int64_t)r * D8;
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

// With the inverse permutation: a warp owns a (token, chunk) item and adds
// the token's top_k rows in ascending row order into an fp32 accumulator
// started from out[t] (ACC) or from zero.
// top_k > 1 with the inverse permutation: a warp owns a (token, chunk) item and
// sums the token's top_k rows in slot order, in fp32, onto out (ACC) or zero.
// K > 0: top_k fixed at compile time, so every row load of the item is issued
// before the first add (K rows x U vectors per lane in flight); K == 0: any
// top_k, one row at a time.  U: 16-byte vectors per lane per row.
template <bool ACC, int K, int U>
__global__ void __launch_bounds__(kThreads) scatter_add_tokens_kernel(uint4* __restrict__ out,
                                                                      const uint4* __restrict__ in,
                                                                      const int32_t* __restrict__ inv, int k, int a,
                                                                      int T, int D8,
                                                                      const int32_t* __restrict__ valid_p,
                                                                      const int32_t* __restrict__ sum_counts, int E,
                                                                      unsigned int* err) {
  const int valid = valid_rows(valid_p, sum_counts, E, a, err);
  if (valid % k != 0 && blockIdx.x == 0 && threadIdx.x == 0) flag_error(err, MOE_DEVERR_BAD_COUNT);
  int Tv = valid / k;
  if (Tv > T) Tv = T;
  const int lane = threadIdx.x & 31;
  constexpr int kItem = 32 * U;  // vectors of a row per item
  const int chunks = (D8 + kItem - 1) / kItem;
  const int64_t items = (int64_t)Tv * chunks;
  for (int64_t it = global_warp(); it < items; it += num_warps()) {
    const int t = (int)(it / chunks);
    const int c0 = (int)(it - (int64_t)t * chunks) * kItem + lane;
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
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (ACC && c0 + 32 * u < D8) {
        bf16x8_to_f32(o[c0 + 32 * u], acc[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
      }
    }
    auto add_row = [&](const uint4* v) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (c0 + 32 * u < D8) {
          float fi[8];
          bf16x8_to_f32(v[u], fi);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[u][i] = __fadd_rn(acc[u][i], fi[i]);
        }
    };
    if constexpr (K > 0) {
      uint4 v[K][U];
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const uint4* src = in + (int64_t)__shfl_sync(0xffffffffu, my_row, j) * D8;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + 32 * u < D8) v[j][u] = __ldg(src + c0 + 32 * u);
      }
#pragma unroll
      for (int j = 0; j < K; ++j) add_row(v[j]);
    } else {
      for (int j = 0; j < k; ++j) {
        const int r = (j < 32) ? __shfl_sync(0xffffffffu, my_row, j) : __ldg(inv + (int64_t)t * k + j);
        if ((unsigned)r >= (unsigned)a) {  // only reachable for top_k > 32
          flag_error(err, MOE_DEVERR_BAD_INDEX);
          continue;
        }
        const uint4* src = in + (int64_t)r * D8;
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + 32 * u < D8) v[u] = __ldg(src + c0 + 32 * u);
        add_row(v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c0 + 32 * u < D8) o[c0 + 32 * u] = f32_to_bf16x8(acc[u]);
  }
}

// Top-k finalize: a warp owns a (token, chunk) item, multiplies each present
// route's row by its weight and adds it in slot order into an fp32 accumulator
// started at zero (fp32 multiply, then fp32 add); the bf16 result has its
// negative zero replaced by +0, and the shared output is added with one more
// rounding.  Tokens t >= the valid count are not written.
template <bool SHARED, bool F32W>
__global__ void __launch_bounds__(kThreads) topk_finalize_kernel(uint4* __restrict__ out,
                                                                 const uint4* __restrict__ rows, int64_t n_rows,
                                                                 int D8, const void* __restrict__ weights,
                                                                 const int32_t* __restrict__ idx, int M, int k,
                                                                 const int32_t* __restrict__ valid_p,
                                                                 const uint4* __restrict__ shared, unsigned int* err) {
  const int Mv = read_count(valid_p, M, err);
  const int lane = threadIdx.x & 31;
  const int chunks = (D8 + kChunk - 1) / kChunk;
  const int64_t items = (int64_t)Mv * chunks;
  for (int64_t it = global_warp(); it < items; it += num_warps()) {
    const int t = (int)(it / chunks);
    const int c0 = (int)(it - (int64_t)t * chunks) * kChunk + lane;
    float acc[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int64_t sj = (int64_t)t * k + j;
      const int p = __ldg(idx + sj);
      if (p < 0) continue;  // a route that is absent
      if (p >= n_rows) {
        if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
        continue;
      }
      const float w = F32W ? __ldg(reinterpret_cast<const float*>(weights) + sj)
                           : __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(weights) + sj));
      const uint4* src = rows + (int64_t)p * D8;
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (c0 + 32 * u < D8) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (c0 + 32 * u < D8) {
          float fi[8];
          bf16x8_to_f32(v[u], fi);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[u][i] = __fadd_rn(acc[u][i], __fmul_rn(w, fi[i]));
        }
    }
    uint4* o = out + (int64_t)t * D8;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (c0 + 32 * u < D8) {
        uint4 r = f32_to_bf16x8(acc[u]);
        uint32_t* h = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // negative zero -> +0, per bf16 half
          if ((h[q] & 0xFFFFu) == 0x8000u) h[q] &= 0xFFFF0000u;
          if ((h[q] >> 16) == 0x8000u) h[q] &= 0x0000FFFFu;
        }
        if (SHARED) {
          float fr[8], fs[8];
          bf16x8_to_f32(r, fr);
          bf16x8_to_f32(__ldg(shared + (int64_t)t * D8 + c0 + 32 * u), fs);
#pragma unroll
          for (int i = 0; i < 8; ++i) fr[i] = __fadd_rn(fr[i], fs[i]);
          r = f32_to_bf16x8(fr);
        }
        o[c0 + 32 * u] = r;
      }
  }
}

}  // namespace

cudaError_t launch_gather_scale(const GatherArgs& g, cudaStream_t s) {
  if (g.inv && g.top_k > 1 && g.top_k <= 32) {  // token-major: each x row is read once for its top_k rows
    const StagedShape sh = staged_shape(g.D / 8);
    if (sh.warps) return launch_staged<false>(g, sh, s);
  }
  const int grid =
      persistent_grid(gather_scale_kernel, (int64_t)g.a * ((g.D / 8 + kGatherChunk - 1) / kGatherChunk), kWarps);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};  // may start while the router's kernel runs
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gather_scale_kernel, static_cast<const uint4*>(g.x), g.T, g.D / 8,
                                     g.token_indices, g.expert_indices, g.a, g.scores, g.dtype, g.stride_t,
                                     g.stride_e, g.E, g.valid, static_cast<uint4*>(g.out), g.err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Plain launch of a row kernel (kThreads per block), after the previous kernel of
// the stream.  Programmatic dependent launch is kept for the gathers only: on the
// row pass, the scatters and the finalize it made the steps slower.
template <typename... KArgs, typename... Args>
cudaError_t launch_rows(void (*kern)(KArgs...), int grid, cudaStream_t s, Args... args) {
  kern<<<grid, kThreads, 0, s>>>(static_cast<KArgs>(args)...);
  return cudaGetLastError();
}

// Row groups: the fewest warps per row (G) with at most 4 vectors (32 fp32) per
// thread, 8 vectors only past 8 warps (D or H above 8192).
inline int pick_group(int nvec) {
  for (int g = 1; g < 8; g <<= 1)
    if (nvec <= 32 * g * 4) return g;
  return 8;
}

#define MOE_GATHER_QUANT(G, VPT)                                                                              \
  gather_scale_quant_kernel<G, VPT><<<persistent_grid(gather_scale_quant_kernel<G, VPT>, g.a, kThreads / (32 * G)), \
                                      kThreads, 0, s>>>(                                                     \
      static_cast<const uint4*>(g.x), g.T, D8, g.token_indices, g.expert_indices, g.a, g.scores, g.dtype,     \
      g.stride_t, g.stride_e, g.E, g.valid, g.scale_ub, static_cast<uint2*>(g.out), g.out_scale, g.err)

cudaError_t launch_gather_scale_quant(const GatherArgs& g, cudaStream_t s) {
  const int D8 = g.D / 8;
  // TMA-staged rows (token-major with the inverse permutation) when two row
  // slots per warp fit in shared memory, else rows held in registers.
  const StagedShape sh = staged_shape(D8);
  if (sh.warps && (!g.inv || g.top_k <= 32)) return launch_staged<true>(g, sh, s);
  const int G = pick_group(D8);
  const bool full = D8 > 32 * G * 4;  // 8 vectors per thread, else 4
  switch (G * 2 + (full ? 1 : 0)) {
    case 2: MOE_GATHER_QUANT(1, 4); break;
    case 4: MOE_GATHER_QUANT(2, 4); break;
    case 8: MOE_GATHER_QUANT(4, 4); break;
    case 16: MOE_GATHER_QUANT(8, 4); break;
    default: MOE_GATHER_QUANT(8, 8); break;  // rows past 8192 elements
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const float* w, int64_t rows, int cols, const float* ub, void* q, float* scale,
                                 cudaStream_t s) {
  const int grid = persistent_grid(quantize_rows_kernel, rows, 1);
  quantize_rows_kernel<<<grid, kThreads, 0, s>>>(reinterpret_cast<const float4*>(w), rows, cols / 4, ub,
                                                 static_cast<uint32_t*>(q), scale);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul(const SiluArgs& g, cudaStream_t s) {
  const int grid = persistent_grid(silu_mul_kernel, (int64_t)g.a * ((g.H / 8 + kChunk - 1) / kChunk), kWarps);
  silu_mul_kernel<<<grid, kThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(g.x0),
                                            static_cast<const __nv_bfloat16*>(g.x1), g.ld, g.a, g.H / 8, g.valid,
                                            static_cast<uint4*>(g.z), g.err);
  return cudaGetLastError();
}

#define MOE_SILU_QUANT(G, VPT)                                                                              \
  do {                                                                                                      \
    auto k = silu_mul_quant_kernel<G, VPT, SILU>;                                                           \
    return launch_rows(k, persistent_grid(k, g.a, kThreads / (32 * G)), s,                                    \
                      static_cast<const __nv_bfloat16*>(g.x0), static_cast<const __nv_bfloat16*>(g.x1), g.ld, \
                      g.a, H8, g.valid, g.sum_counts, g.E, g.scale_ub, static_cast<uint2*>(g.z), g.z_scale,   \
                      g.err);                                                                               \
  } while (0)

template <bool SILU>
cudaError_t launch_row_quant(const SiluArgs& g, cudaStream_t s) {
  const int H8 = g.H / 8;
  const int G = pick_group(H8);
  const bool full = H8 > 32 * G * 4;
  switch (G * 2 + (full ? 1 : 0)) {
    case 2: MOE_SILU_QUANT(1, 4);
    case 4: MOE_SILU_QUANT(2, 4);
    case 8: MOE_SILU_QUANT(4, 4);
    case 16: MOE_SILU_QUANT(8, 4);
    default: MOE_SILU_QUANT(8, 8);  // rows past 8192 elements
  }
}
#undef MOE_SILU_QUANT

cudaError_t launch_silu_mul_quant(const SiluArgs& g, cudaStream_t s) { return launch_row_quant<true>(g, s); }

cudaError_t launch_quantize_rows_bf16(const SiluArgs& g, cudaStream_t s) { return launch_row_quant<false>(g, s); }

cudaError_t launch_scatter_add(const ScatterArgs& g, cudaStream_t s) {
  const int D8 = g.D / 8;
  if (g.inv) {
    // the common top_k values get every row load of an item in flight at once
#define MOE_SCATTER_TOKENS(K, U)                                                                                 \
  do {                                                                                                           \
    auto k = g.accumulate ? scatter_add_tokens_kernel<true, K, U> : scatter_add_tokens_kernel<false, K, U>;       \
    const int grid = persistent_grid(k, (int64_t)g.T * ((D8 + 32 * U - 1) / (32 * U)), kWarps);                 \
    return launch_rows(k, grid, s, static_cast<uint4*>(g.out), static_cast<const uint4*>(g.in), g.inv, g.top_k,    \
                      g.a, g.T, D8, g.valid, g.sum_counts, g.E, g.err);                                          \
  } while (0)
    switch (g.top_k) {
      case 2: MOE_SCATTER_TOKENS(2, 4);
      case 4: MOE_SCATTER_TOKENS(4, 4);
      case 8: MOE_SCATTER_TOKENS(8, 2);
      default: MOE_SCATTER_TOKENS(0, 4);
    }
#undef MOE_SCATTER_TOKENS
  }
  auto k = g.accumulate ? scatter_add_rows_kernel<true> : scatter_add_rows_kernel<false>;
  const int grid = persistent_grid(k, (int64_t)g.a * ((D8 + kChunk - 1) / kChunk), kWarps);
  return launch_rows(k, grid, s, static_cast<uint4*>(g.out), static_cast<const uint4*>(g.in), g.token_indices, g.a,
                    g.T, D8, g.valid, g.sum_counts, g.E, g.err);
}

cudaError_t launch_topk_finalize(const FinalizeArgs& g, cudaStream_t s) {
  const int D8 = g.D / 8;
  const bool f32 = g.weights_dtype == MOE_DTYPE_F32;
  auto k = g.shared ? (f32 ? topk_finalize_kernel<true, true> : topk_finalize_kernel<true, false>)
                    : (f32 ? topk_finalize_kernel<false, true> : topk_finalize_kernel<false, false>);
  const int grid = persistent_grid(k, (int64_t)g.M * ((D8 + kChunk - 1) / kChunk), kWarps);
  return launch_rows(k, grid, s, static_cast<uint4*>(g.out), static_cast<const uint4*>(g.rows), g.n_rows, D8,
                    g.weights, g.idx, g.M, g.k, g.valid, static_cast<const uint4*>(g.shared), g.err);
}

}  // namespace moe
