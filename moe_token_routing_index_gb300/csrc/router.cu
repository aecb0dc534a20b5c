// Router scores of mslk/moe/layers.py (MetaShufflingMoE._route; the same two
// steps open BaselineMoE._forward): scores = sigmoid(linear(tokens, router_DE.T)),
// both in bf16, for the valid tokens.
//
// logits = x[Tv, D] . w[E, D]^T is a GEMM with a short N (the experts) and a
// long K, so its cost is one read of x.  Tiles of 128 tokens x N = E (rounded
// up to 16, at most 256) run on tcgen05 with an fp32 accumulator in tensor
// memory.  With few token tiles the reduction over D is split S ways (S in
// {1, 2, 4, 8}, S x tiles about the SM count) and the S CTAs of a tile form a
// thread-block cluster: each CTA streams its share of the K blocks, parks its
// fp32 partial tile in its own shared memory (the operand ring is idle by
// then), and after a cluster barrier CTA s reduces rows [s 128/S, (s+1) 128/S)
// by reading the S partials over distributed shared memory in rank order
// (a fixed order: every run gives the same bits).  Finishing an element:
// logit = bf16(sum), score = bf16(1 / (1 + e^-logit)) with the sigmoid in fp32
// (expf, IEEE division).
//
// Warp roles as in the grouped GEMM: warp 0 TMA producer (128 x 128-byte A
// boxes of x, N x 128-byte B boxes of w, 128B swizzle), warp 1 MMA issuer and
// owner of the tensor memory, warps 2-5 move the accumulator rows to shared
// memory (one token row per thread); all six warps reduce.  Waits on the
// pipeline are bounded (1 s); on expiry the kernel records MOE_DEVERR_TIMEOUT,
// drains what it issued, still meets its cluster at both barriers, frees
// tensor memory and returns.
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
constexpr int kMinKb = 8;          // K blocks per split, at least
constexpr int kMaxSplit = 8;       // portable cluster size
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kRABytes = kRBM * kRBKBytes;  // 16 KB

struct RouterParams {
  int T, D, E;
  int n_mma;       // MMA N: E rounded up to 16
  int tmem_cols;   // power of two >= max(32, n_mma)
  int stages;
  int num_kb;
  int split;       // CTAs per tile (the cluster size)
  int pstride;     // floats per row of the parked partial tile
  int vec_store;   // E % 4 == 0 and scores 8-byte aligned: 8-byte score stores
  const int32_t* num_valid;
  __nv_bfloat16* scores;
  unsigned int* err;
};

struct RouterSmem {
  int a, b, bars, misc, bytes;
  __host__ __device__ RouterSmem(int stages, int n_mma) {
    a = 0;
    b = a + stages * kRABytes;
    bars = b + stages * n_mma * kRBKBytes;       // full[S], empty[S], tfull, drain
    misc = bars + (2 * stages + 2) * 8;          // tmem base, abort flag
    bytes = misc + 16;
  }
};

__device__ __forceinline__ uint32_t router_idesc(int n_mma) {
  // fp32 accumulate, A and B bf16 K-major, M = 128, N = n_mma
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n_mma >> 3) << 17) | ((uint32_t)(kRBM >> 4) << 24);
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ float sigmoid_of_bf16_logit(float sum) {
  const float logit = __bfloat162float(__float2bfloat16_rn(sum));
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-logit)));
}

__global__ void __launch_bounds__(kRThreads, 1)
    router_scores_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                         const RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  const RouterSmem L(p.stages, p.n_mma);
  const int nst = p.stages;

  // A whole cluster works on one tile; clusters past the valid tokens leave at once
  // (every CTA of such a cluster takes this branch, so none waits at a cluster barrier).
  const int S = p.split;
  const int m = blockIdx.x / S;
  const int rank = blockIdx.x - m * S;
  const int Tv = read_count(p.num_valid, p.T, (threadIdx.x == 0 && blockIdx.x == 0) ? p.err : nullptr);
  if (m * kRBM >= Tv) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  auto bar_full = [&](int s) { return smem_u32(&bars[s]); };
  auto bar_empty = [&](int s) { return smem_u32(&bars[nst + s]); };
  const uint32_t bar_tfull = smem_u32(&bars[2 * nst]);
  const uint32_t bar_drain = smem_u32(&bars[2 * nst + 1]);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc + 4);

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_tfull, 1);
    mbar_init(bar_drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_w);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int kb0 = (int)((int64_t)rank * p.num_kb / S), kb1 = (int)((int64_t)(rank + 1) * p.num_kb / S);

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t stage_bytes = (uint32_t)(kRABytes + p.n_mma * kRBKBytes);
      int s = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
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
        if (++s == nst) {
          s = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        flag_error(p.err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        for (int i = 0; i < nst; ++i)
          if ((issued_mask >> i) & 1u) mbar_wait(bar_full(i), (issued_parity >> i) & 1u, nullptr, kDrainTimeoutNs);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = router_idesc(p.n_mma);
      int s = 0;
      uint32_t phase = 0;
      bool ok = true, issued_any = false;
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
          mma_issue<false>(tmem_base, smem_desc_sw128(a_addr + kk * 32), smem_desc_sw128(b_addr + kk * 32), idesc,
                           (kb != kb0 || kk != 0) ? 1u : 0u);
        issued_any = true;
        mma_commit(bar_empty(s));
        if (++s == nst) {
          s = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        mma_commit(bar_tfull);
      } else {
        flag_error(p.err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        if (issued_any) {
          mma_commit(bar_drain);
          mbar_wait(bar_drain, 0, nullptr, kDrainTimeoutNs);
        }
      }
    }
  } else {
    // -------------------------------- epilogue: park the partial tile in shared memory
    // The MMAs that read the operand ring have completed once tfull fires, so the
    // ring's first bytes take the partial: row r at smem + r * pstride floats.
    const int sub = warp & 3;  // the TMEM lane quarter this warp may read
    const int r = sub * 32 + lane;
    if (mbar_wait(bar_tfull, 0, s_abort)) {
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16);
      float* prow = reinterpret_cast<float*>(smem) + r * p.pstride;
#pragma unroll 1
      for (int c = 0; c < p.E; c += 32) {
        float v[32];
        tmem_ld32(tbase + c, v);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (c + 4 * q < p.E)
            *reinterpret_cast<float4*>(prow + c + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2],
                                                                       v[4 * q + 3]);
      }
    } else {
      if (lane == 0) flag_error(p.err, MOE_DEVERR_TIMEOUT);
      *s_abort = 1;
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---- every CTA's partial is parked: reduce this rank's rows over the cluster
  cluster_sync_all();
  {
    const int rows = kRBM / S;
    const int row0 = rank * rows;
    const int groups = (p.E + 3) / 4;  // 4-column groups per row
    uint32_t peer[kMaxSplit];          // the partial tile's base in each CTA of the cluster
#pragma unroll
    for (int j = 0; j < kMaxSplit; ++j) peer[j] = j < S ? map_to_rank(sbase, (uint32_t)j) : 0u;
    for (int i = threadIdx.x; i < rows * groups; i += kRThreads) {
      const int rr = row0 + i / groups;
      const int c = (i % groups) * 4;
      const uint32_t off = (uint32_t)((rr * p.pstride + c) * 4);
      float4 part[kMaxSplit];
#pragma unroll
      for (int j = 0; j < kMaxSplit; ++j)
        if (j < S) part[j] = ld_dsmem_f4(peer[j] + off);
      float4 acc = part[0];
#pragma unroll
      for (int j = 1; j < kMaxSplit; ++j)
        if (j < S) {
          acc.x = __fadd_rn(acc.x, part[j].x);
          acc.y = __fadd_rn(acc.y, part[j].y);
          acc.z = __fadd_rn(acc.z, part[j].z);
          acc.w = __fadd_rn(acc.w, part[j].w);
        }
      const int t = m * kRBM + rr;
      if (t < Tv) {
        __nv_bfloat16* dst = p.scores + (int64_t)t * p.E + c;
        const __nv_bfloat16 s0 = __float2bfloat16_rn(sigmoid_of_bf16_logit(acc.x));
        const __nv_bfloat16 s1 = __float2bfloat16_rn(sigmoid_of_bf16_logit(acc.y));
        const __nv_bfloat16 s2 = __float2bfloat16_rn(sigmoid_of_bf16_logit(acc.z));
        const __nv_bfloat16 s3 = __float2bfloat16_rn(sigmoid_of_bf16_logit(acc.w));
        if (p.vec_store) {
          __nv_bfloat162 lo, hi;
          lo.x = s0;
          lo.y = s1;
          hi.x = s2;
          hi.y = s3;
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&lo);
          u.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(dst) = u;
        } else {
          dst[0] = s0;
          if (c + 1 < p.E) dst[1] = s1;
          if (c + 2 < p.E) dst[2] = s2;
          if (c + 3 < p.E) dst[3] = s3;
        }
      }
    }
  }
  // no CTA leaves (freeing its shared memory) while a peer may still read it
  cluster_sync_all();

  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(p.tmem_cols)
                 : "memory");
}

struct RouterPlan {
  int n_mma, tmem_cols, stages, num_kb, split, pstride, m_tiles;
};

RouterPlan plan_router(int T, int D, int E) {
  RouterPlan q;
  q.n_mma = (E + 15) / 16 * 16;
  q.tmem_cols = 32;
  while (q.tmem_cols < q.n_mma) q.tmem_cols *= 2;
  const int stage_bytes = kRABytes + q.n_mma * kRBKBytes;
  q.stages = kSmemBudget / stage_bytes;
  if (q.stages > kMaxStages) q.stages = kMaxStages;
  q.num_kb = (D + kRBK - 1) / kRBK;
  q.m_tiles = (T + kRBM - 1) / kRBM;
  q.pstride = (E + 3) / 4 * 4 + 4;  // 4 floats of padding spread the rows over the banks
  // splits: a power of two, the tiles' CTAs about the SM count, at least kMinKb K blocks each
  const int sms = device_sm_count();
  q.split = 1;
  while (q.split * 2 <= kMaxSplit && (int64_t)q.m_tiles * q.split * 2 <= sms &&
         q.num_kb / (q.split * 2) >= kMinKb)
    q.split *= 2;
  return q;
}

}  // namespace

size_t router_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_router_scores(const RouterArgs& a, cudaStream_t s) {
  const RouterPlan q = plan_router(a.T, a.D, a.E);
  CUtensorMap mx, mw;
  if (!make_map_sw128(&mx, a.x, a.T, a.D, false, kRBM) || !make_map_sw128(&mw, a.w, a.E, a.D, false, q.n_mma))
    return cudaErrorInvalidValue;
  RouterParams p;
  p.T = a.T;
  p.D = a.D;
  p.E = a.E;
  p.n_mma = q.n_mma;
  p.tmem_cols = q.tmem_cols;
  p.stages = q.stages;
  p.num_kb = q.num_kb;
  p.split = q.split;
  p.pstride = q.pstride;
  p.vec_store = (a.E % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 7) == 0);
  p.num_valid = a.num_valid;
  p.scores = static_cast<__nv_bfloat16*>(a.scores);
  p.err = a.err;
  const RouterSmem L(q.stages, q.n_mma);
  const int smem = L.bytes + 1024;
  // the parked partial tile fits in the operand ring
  if ((int64_t)kRBM * q.pstride * 4 > L.bars) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(router_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(q.m_tiles * q.split);
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = q.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, router_scores_kernel, mx, mw, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
