// Router scores of mslk/moe/layers.py (MetaShufflingMoE._route; the same two
// steps open BaselineMoE._forward): scores = sigmoid(linear(tokens, router_DE.T)),
// both in bf16, for the valid tokens.
//
// logits = x[Tv, D] . w[E, D]^T is a GEMM with a short N (the experts) and a
// long K, so its cost is one read of x.  Tiles of 128 tokens x N = E (rounded
// up to 16, at most 256) run on tcgen05 with fp32 accumulators in tensor
// memory.  With few token tiles K is split S ways so that the read of x is
// spread over every SM: S = CTAs / tiles, each split at least kMinKb K blocks.
// A split writes its fp32 partial tile to the workspace, and each epilogue warp
// bumps the arrival counter of its 32-row quarter of the tile; the warp whose
// arrival completes the count adds the S partials of those rows in split order
// (a fixed order: every run gives the same bits) and finishes them.  Finishing
// a row: logit = bf16(sum), score = bf16(1 / (1 + e^-logit)) with the sigmoid
// in fp32 (expf, IEEE division).
//
// Warp roles as in the grouped GEMM: warp 0 TMA producer (128 x 128-byte A
// boxes of x, N x 128-byte B boxes of w, 128B swizzle), warp 1 MMA issuer and
// owner of the tensor memory (two accumulators), warps 2-5 the epilogue with
// one token row per thread.  Waits are bounded (1 s); on expiry the kernel
// records MOE_DEVERR_TIMEOUT, drains what it issued, frees tensor memory and
// returns.
#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kRBM = 128;          // tokens per tile
constexpr int kRBKBytes = 128;     // bytes of K per stage: 64 bf16
constexpr int kRBK = kRBKBytes / 2;
constexpr int kRThreads = 192;
constexpr int kMinKb = 4;          // K blocks per split, at least
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kRABytes = kRBM * kRBKBytes;  // 16 KB
constexpr int kMaxCtas = 256;      // bounds the partial-tile workspace whatever the SM count

struct RouterParams {
  int T, D, E;
  int n_mma;       // MMA N: E rounded up to 16
  int acc_cols;    // tensor-memory columns of one accumulator (power of two >= 32)
  int stages;
  int num_kb;
  int part_cols;   // row stride of a partial tile: E rounded up to 32
  int vec_store;   // 16-byte score stores are aligned
  const int32_t* num_valid;
  __nv_bfloat16* scores;
  float* partial;  // [CTAs][128][part_cols]
  int* arrivals;   // [token tiles of T][4]: splits stored, per 32-row quarter
  unsigned int* err;
};

struct RouterSmem {
  int a, b, bars, misc, bytes;
  __host__ __device__ RouterSmem(int stages, int n_mma) {
    a = 0;
    b = a + stages * kRABytes;
    bars = b + stages * n_mma * kRBKBytes;       // full[S], empty[S], tfull[2], tempty[2], drain
    misc = bars + (2 * stages + 5) * 8;          // tmem base, abort flag
    bytes = misc + 16;
  }
};

__device__ __forceinline__ uint32_t router_idesc(int n_mma) {
  // fp32 accumulate, A and B bf16 K-major, M = 128, N = n_mma
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n_mma >> 3) << 17) | ((uint32_t)(kRBM >> 4) << 24);
}

// Scores of 32 columns [c, c + 32) of one token row from their fp32 logit sums.
__device__ __forceinline__ void finish_chunk(const RouterParams& p, const float* sum, int t, int c) {
  __nv_bfloat16* row = p.scores + (int64_t)t * p.E;
  float sc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float logit = __bfloat162float(__float2bfloat16_rn(sum[i]));
    sc[i] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-logit)));
  }
  if (p.vec_store) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (c + 8 * q < p.E) *reinterpret_cast<uint4*>(row + c + 8 * q) = f32_to_bf16x8(sc + 8 * q);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c + i < p.E) row[c + i] = __float2bfloat16_rn(sc[i]);
  }
}

__global__ void __launch_bounds__(kRThreads, 1)
    router_scores_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                         const RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  const RouterSmem L(p.stages, p.n_mma);
  const int S_st = p.stages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  auto bar_full = [&](int s) { return smem_u32(&bars[s]); };
  auto bar_empty = [&](int s) { return smem_u32(&bars[S_st + s]); };
  auto bar_tfull = [&](int b) { return smem_u32(&bars[2 * S_st + b]); };
  auto bar_tempty = [&](int b) { return smem_u32(&bars[2 * S_st + 2 + b]); };
  const uint32_t bar_drain = smem_u32(&bars[2 * S_st + 4]);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc + 4);

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S_st; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull(b), 1);
      mbar_init(bar_tempty(b), 4);
    }
    mbar_init(bar_drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_w);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(2 * p.acc_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  // The work list, from the device's valid-token count.
  const int Tv = read_count(p.num_valid, p.T, threadIdx.x == 0 ? p.err : nullptr);
  const int m_tiles = (Tv + kRBM - 1) / kRBM;
  int S = 1;
  if (m_tiles > 0) {
    S = (int)gridDim.x / m_tiles;
    const int cap = p.num_kb / kMinKb;
    if (S > cap) S = cap;
    if (S < 1) S = 1;
  }
  const int items = m_tiles * S;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t stage_bytes = (uint32_t)(kRABytes + p.n_mma * kRBKBytes);
      int s = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
        const int m = item / S, sp = item - m * S;
        const int kb0 = (int)((int64_t)sp * p.num_kb / S), kb1 = (int)((int64_t)(sp + 1) * p.num_kb / S);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(bar_empty(s), phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + L.a + s * kRABytes;
          const uint32_t b_dst = sbase + L.b + s * p.n_mma * kRBKBytes;
          mbar_arrive_expect_tx(bar_full(s), stage_bytes);
          tma_load_2d(a_dst, &map_x, bar_full(s), kb * kRBK, m * kRBM);
          tma_load_2d(b_dst, &map_w, bar_full(s), kb * kRBK, 0);
          issued_mask |= 1u << s;
          issued_parity = (issued_parity & ~(1u << s)) | (phase << s);
          if (++s == S_st) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        flag_error(p.err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        for (int i = 0; i < S_st; ++i)
          if ((issued_mask >> i) & 1u) mbar_wait(bar_full(i), (issued_parity >> i) & 1u, nullptr, kDrainTimeoutNs);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = router_idesc(p.n_mma);
      int s = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued_any = false;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
        const int m = item / S, sp = item - m * S;
        const int kb0 = (int)((int64_t)sp * p.num_kb / S), kb1 = (int)((int64_t)(sp + 1) * p.num_kb / S);
        if (!mbar_wait(bar_tempty(acc), acc_phase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * p.acc_cols);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(bar_full(s), phase, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + L.a + s * kRABytes;
          const uint32_t b_addr = sbase + L.b + s * p.n_mma * kRBKBytes;
#pragma unroll
          for (int kk = 0; kk < kRBKBytes / 32; ++kk)  // K = 16 bf16 per instruction
            mma_issue<false>(d, smem_desc_sw128(a_addr + kk * 32), smem_desc_sw128(b_addr + kk * 32), idesc,
                             (kb != kb0 || kk != 0) ? 1u : 0u);
          issued_any = true;
          mma_commit(bar_empty(s));
          if (++s == S_st) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(bar_tfull(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        flag_error(p.err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        if (issued_any) {
          mma_commit(bar_drain);
          mbar_wait(bar_drain, 0, nullptr, kDrainTimeoutNs);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int sub = warp & 3;  // the TMEM lane quarter this warp may read
    const int r = sub * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
      const int m = item / S;
      const int t = m * kRBM + r;
      const bool row_ok = t < Tv;
      if (!mbar_wait(bar_tfull(acc), acc_phase, s_abort)) {
        if (lane == 0) flag_error(p.err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * p.acc_cols);
      if (S == 1) {
#pragma unroll 1
        for (int c = 0; c < p.E; c += 32) {
          float v[32];
          tmem_ld32(tbase + c, v);
          if (row_ok) finish_chunk(p, v, t, c);
        }
      } else {
        float* part = p.partial + ((int64_t)item * kRBM + r) * p.part_cols;
#pragma unroll 1
        for (int c = 0; c < p.E; c += 32) {
          float v[32];
          tmem_ld32(tbase + c, v);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(part + c)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      if (S > 1) {
        // Publish this warp's 32 rows of the split; the warp whose arrival
        // completes the count of this tile quarter adds the splits and finishes them.
        __syncwarp();
        int before = 0;
        if (lane == 0) {
          __threadfence();
          before = atomicAdd(p.arrivals + m * 4 + sub, 1);
        }
        before = __shfl_sync(0xffffffffu, before, 0);
        __syncwarp();
        if (before == S - 1) {
          __threadfence();
          const int64_t split_stride = (int64_t)kRBM * p.part_cols;
          const float* part0 = p.partial + ((int64_t)m * S * kRBM + r) * p.part_cols;
#pragma unroll 1
          for (int c = 0; c < p.E; c += 32) {
            float sum[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 u = __ldcg(reinterpret_cast<const float4*>(part0 + c) + q);
              sum[4 * q] = u.x;
              sum[4 * q + 1] = u.y;
              sum[4 * q + 2] = u.z;
              sum[4 * q + 3] = u.w;
            }
            for (int sp = 1; sp < S; ++sp) {
              const float4* src = reinterpret_cast<const float4*>(part0 + sp * split_stride + c);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 u = __ldcg(src + q);
                sum[4 * q] = __fadd_rn(sum[4 * q], u.x);
                sum[4 * q + 1] = __fadd_rn(sum[4 * q + 1], u.y);
                sum[4 * q + 2] = __fadd_rn(sum[4 * q + 2], u.z);
                sum[4 * q + 3] = __fadd_rn(sum[4 * q + 3], u.w);
              }
            }
            if (row_ok) finish_chunk(p, sum, t, c);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(2 * p.acc_cols)
                 : "memory");
}

struct RouterPlan {
  int n_mma, acc_cols, stages, num_kb, part_cols, grid, m_tiles;
  size_t arrivals_bytes, partial_bytes;
};

RouterPlan plan_router(int T, int D, int E) {
  RouterPlan q;
  q.n_mma = (E + 15) / 16 * 16;
  q.acc_cols = 32;
  while (q.acc_cols < q.n_mma) q.acc_cols *= 2;
  const int stage_bytes = kRABytes + q.n_mma * kRBKBytes;
  q.stages = kSmemBudget / stage_bytes;
  if (q.stages > kMaxStages) q.stages = kMaxStages;
  q.num_kb = (D + kRBK - 1) / kRBK;
  q.part_cols = (E + 31) / 32 * 32;
  q.m_tiles = (T + kRBM - 1) / kRBM;
  int splits = q.num_kb / kMinKb;
  if (splits < 1) splits = 1;
  const int64_t items = (int64_t)q.m_tiles * splits;
  const int64_t cap = items < kMaxCtas ? items : kMaxCtas;
  q.grid = (int)cap;  // the workspace is sized for this many CTAs
  q.partial_bytes = (size_t)q.grid * kRBM * q.part_cols * 4;
  q.arrivals_bytes = ((size_t)q.m_tiles * 16 + 255) / 256 * 256;
  return q;
}

}  // namespace

size_t router_workspace_bytes(int T, int D, int E) {
  if (T <= 0) return 0;
  const RouterPlan q = plan_router(T, D, E);
  return q.arrivals_bytes + q.partial_bytes;
}

cudaError_t launch_router_scores(const RouterArgs& a, cudaStream_t s) {
  const RouterPlan q = plan_router(a.T, a.D, a.E);
  CUtensorMap mx, mw;
  if (!make_map_sw128(&mx, a.x, a.T, a.D, false, kRBM) || !make_map_sw128(&mw, a.w, a.E, a.D, false, q.n_mma))
    return cudaErrorInvalidValue;
  const int sms = device_sm_count();
  const int grid = q.grid < sms ? q.grid : sms;
  RouterParams p;
  p.T = a.T;
  p.D = a.D;
  p.E = a.E;
  p.n_mma = q.n_mma;
  p.acc_cols = q.acc_cols;
  p.stages = q.stages;
  p.num_kb = q.num_kb;
  p.part_cols = q.part_cols;
  p.vec_store = (a.E % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15) == 0);
  p.num_valid = a.num_valid;
  p.scores = static_cast<__nv_bfloat16*>(a.scores);
  char* ws = static_cast<char*>(a.ws);
  p.arrivals = reinterpret_cast<int*>(ws);
  p.partial = reinterpret_cast<float*>(ws + q.arrivals_bytes);
  p.err = a.err;
  cudaError_t e = cudaMemsetAsync(p.arrivals, 0, (size_t)q.m_tiles * 16, s);
  if (e != cudaSuccess) return e;
  const int smem = RouterSmem(q.stages, q.n_mma).bytes + 1024;
  e = cudaFuncSetAttribute(router_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  router_scores_kernel<<<grid, kRThreads, smem, s>>>(mx, mw, p);
  return cudaGetLastError();
}

}  // namespace moe
