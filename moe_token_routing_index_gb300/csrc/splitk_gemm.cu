// Split-K GEMMs for skinny problems, reduced over a thread-block cluster:
//
//  * router scores of mslk/moe/layers.py (MetaShufflingMoE._route; the same two
//    steps open BaselineMoE._forward): scores = sigmoid(linear(tokens,
//    router_DE.T)), both in bf16, for the valid tokens;
//  * the shared expert's dense GEMMs (MetaShufflingMoE._shared_expert_part1 /
//    _part2) when the batch is small: y = x @ w13.T with the SiLU*mul epilogue
//    (z = silu(y0) * y1), and out = z @ w2.T.
//
// y = A[rows, K] . B[N, K]^T.  A tile is 128 rows x N_tile columns (N_tile = E
// rounded up to 16 for the router; 256 for the dense GEMMs, w_in and gate rows
// stacked 128 + 128 for SiLU*mul) accumulated by tcgen05 in tensor memory.
// Such problems have few tiles and a long K, so their cost is streaming the
// operands: the K blocks of a tile are split S ways (the largest S <= 8 at which
// every tile's cluster is resident at once, as the occupancy query for clusters
// reports) and the S CTAs of a tile form a thread-block cluster.  Each CTA
// streams its share, parks its fp32 partial tile in its own shared memory (the
// operand ring is idle by then), and after a cluster barrier CTA s reduces its
// slice of the rows by reading the S partials over distributed shared memory
// in rank order (a fixed order: every run gives the same bits) and applies the
// epilogue:
//   sigmoid : logit = bf16(sum), score = bf16(1 / (1 + e^-logit)), fp32 (expf, IEEE division)
//   silu    : z = bf16(silu_mul(bf16(sum_in), bf16(sum_gate))), as the grouped GEMM's epilogue
//   plain   : out = bf16(sum)
//
// Warp roles as in the grouped GEMM: warp 0 TMA producer (128 x 128-byte A
// boxes, B boxes of 128 bytes of K, 128B swizzle), warp 1 MMA issuer and owner
// of the tensor memory, warps 2-5 move the accumulator rows to shared memory
// (one row per thread); all twelve warps (6-11 idle until then) reduce.  Waits on the pipeline are
// bounded (1 s); on expiry the kernel records MOE_DEVERR_TIMEOUT, drains what
// it issued, still meets its cluster at both barriers, frees tensor memory and
// returns.
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kRBM = 128;          // rows per tile
constexpr int kRBKBytes = 128;     // bytes of K per stage: 64 bf16
constexpr int kRBK = kRBKBytes / 2;
constexpr int kRThreads = 384;   // warps 0-5: producer, MMA, 4 to park the partial; all 12 reduce
constexpr int kMinKb = 8;          // K blocks per split, at least
constexpr double kFixedKbPerCta = 6.0;  // a CTA's fixed cost (prologue, epilogue, reduction) in K blocks
constexpr int kMaxSplit = 8;       // portable cluster size
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kRABytes = kRBM * kRBKBytes;  // 16 KB

enum { kEpiSigmoid = 0, kEpiSilu = 1, kEpiPlain = 2, kEpiSigmoidTopK = 3 };
constexpr int kChunkRows = 32;                 // routing chunk: tokens per histogram column
constexpr int kTileChunks = kRBM / kChunkRows;  // 4 chunks per 128-row tile

struct SplitKParams {
  int rows_hi;     // rows of A (the valid count is clamped to it)
  int num_kb;
  int n_mma;       // MMA N, a multiple of 16 (<= 256)
  int b_box;       // rows of one B box
  int b_loads;     // B boxes per stage: 1, or 2 (SiLU*mul: w_in rows, then gate rows)
  int tmem_cols;   // power of two >= max(32, n_mma)
  int stages;
  int split;       // CTAs per tile (the cluster size)
  int n_tiles;     // tiles along N
  int pstride;     // floats per row of the parked partial tile
  int epi;
  int n_out;       // output columns: E, H or N
  int gate_row0;   // SiLU*mul: first gate row of B (H)
  int vec_store;   // n_out % 4 == 0 and out 8-byte aligned
  const int32_t* rows_valid;  // nullable: rows_hi
  __nv_bfloat16* out;         // [rows, n_out]
  unsigned int* err;
  // kEpiSigmoidTopK (the router with the routing selection in its epilogue)
  int top_k;
  int32_t* chosen;            // [rows * top_k]: each valid token's experts, in selection order
  int32_t* hist_t;            // [n_out][nblk]: per 32-token chunk, the tokens that chose each expert
  int nblk;                   // chunks of rows_hi
  unsigned int* barrier;      // the routing kernel's grid-barrier counter, zeroed here
};

struct SplitKSmem {
  int a, b, bars, misc, bytes;
  __host__ __device__ SplitKSmem(int stages, int n_mma) {
    a = 0;
    b = a + stages * kRABytes;
    bars = b + stages * n_mma * kRBKBytes;       // full[S], empty[S], tfull, drain
    misc = bars + (2 * stages + 2) * 8;          // tmem base, abort flag
    bytes = misc + 16;
  }
};

__device__ __forceinline__ uint32_t splitk_idesc(int n_mma) {
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

// The sum over the cluster's S partials of 4 consecutive floats at byte offset off, in rank order.
__device__ __forceinline__ float4 cluster_sum4(const uint32_t* peer, int S, uint32_t off) {
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
  return acc;
}

__device__ __forceinline__ float sigmoid_of_bf16_logit(float sum) {
  const float logit = __bfloat162float(__float2bfloat16_rn(sum));
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-logit)));
}

__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Byte offset of the routing chunk histogram in shared memory: past the parked partial tile.
__host__ __device__ constexpr int topk_hist_offset(int pstride) { return (kRBM * pstride * 4 + 15) / 16 * 16; }

// Store 4 outputs of a row at column c (masked by n_out).
__device__ __forceinline__ void store4(const SplitKParams& p, __nv_bfloat16* row, int c, float v0, float v1, float v2,
                                       float v3) {
  const __nv_bfloat16 s0 = __float2bfloat16_rn(v0), s1 = __float2bfloat16_rn(v1);
  const __nv_bfloat16 s2 = __float2bfloat16_rn(v2), s3 = __float2bfloat16_rn(v3);
  if (p.vec_store && c + 3 < p.n_out) {
    __nv_bfloat162 lo, hi;
    lo.x = s0;
    lo.y = s1;
    hi.x = s2;
    hi.y = s3;
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(row + c) = u;
  } else {
    if (c < p.n_out) row[c] = s0;
    if (c + 1 < p.n_out) row[c + 1] = s1;
    if (c + 2 < p.n_out) row[c + 2] = s2;
    if (c + 3 < p.n_out) row[c + 3] = s3;
  }
}

// kEpiSigmoidTopK reduction of tile m: chunk q (32 rows) of the tile is reduced
// by CTA q % S of the cluster.  A warp takes a row: lane l sums columns 4l..4l+3
// (and 128 + 4l.. when E > 128) of the S partials in rank order, so the scores
// are those of kEpiSigmoid bit for bit, stores them, and the warp selects the
// row's top_k experts as moe_route does (the largest bf16 score, the lower expert
// on equal scores, +0 == -0).  The chunk's expert histogram goes to hist_t[., c];
// every chunk this launch reduces writes all E entries of its column.
template <int G>
__device__ void reduce_sigmoid_topk(const SplitKParams& p, int m, int rank, int S, int Tv, const uint32_t* peer,
                                    int* s_hist) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.n_out, k = p.top_k;
  for (int q = rank; q < kTileChunks; q += S) {
    const int c = m * kTileChunks + q;
    const int t0 = c * kChunkRows;
    if (t0 >= Tv) break;  // the same for every thread of the CTA
    for (int e = threadIdx.x; e < E; e += kRThreads) s_hist[e] = 0;
    __syncthreads();
    for (int r = warp; r < kChunkRows; r += kRThreads / 32) {
      const int t = t0 + r;
      if (t >= Tv) break;  // warp-uniform
      const int rr = q * kChunkRows + r;
      uint32_t key[4 * G];
      uint32_t live = 0;  // bit 4g + i: expert 128 g + 4 lane + i exists and is not yet chosen
      __nv_bfloat16* orow = p.out + (int64_t)t * E;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int c0 = 128 * g + 4 * lane;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c0 < p.n_mma) acc = cluster_sum4(peer, S, (uint32_t)((rr * p.pstride + c0) * 4));
        const float sv[4] = {sigmoid_of_bf16_logit(acc.x), sigmoid_of_bf16_logit(acc.y),
                             sigmoid_of_bf16_logit(acc.z), sigmoid_of_bf16_logit(acc.w)};
        if (c0 < E) store4(p, orow, c0, sv[0], sv[1], sv[2], sv[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          key[4 * g + i] = route_order_key(round_bf16(sv[i]));
          if (c0 + i < E) live |= 1u << (4 * g + i);
        }
      }
      for (int j = 0; j < k; ++j) {
        uint32_t best = 0u;
        int best_i = -1;
#pragma unroll
        for (int i = 0; i < 4 * G; ++i)  // ascending expert index within the lane
          if (((live >> i) & 1u) && (best_i < 0 || key[i] > best)) {
            best = key[i];
            best_i = i;
          }
        const uint32_t wbest = __reduce_max_sync(0xffffffffu, best_i >= 0 ? best : 0u);
        const uint32_t cand =
            (best_i >= 0 && best == wbest) ? (uint32_t)(128 * (best_i >> 2) + 4 * lane + (best_i & 3)) : 0xffffffffu;
        const int we = (int)__reduce_min_sync(0xffffffffu, cand);
        if (((we & 127) >> 2) == lane) live &= ~(1u << (4 * (we >> 7) + (we & 3)));
        if (lane == 0) {
          p.chosen[(int64_t)t * k + j] = we;
          atomicAdd(&s_hist[we], 1);
        }
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kRThreads) p.hist_t[(int64_t)e * p.nblk + c] = s_hist[e];
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kRThreads, 1)
    splitk_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                       const SplitKParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  const SplitKSmem L(p.stages, p.n_mma);
  const int nst = p.stages;

  // A whole cluster works on one tile; clusters past the valid rows leave at once
  // (every CTA of such a cluster takes this branch, so none waits at a cluster barrier).
  const int S = p.split;
  const int tile = blockIdx.x / S;
  const int rank = blockIdx.x - tile * S;
  const int m = tile / p.n_tiles, n = tile - (tile / p.n_tiles) * p.n_tiles;
  // the routing kernel that follows this launch starts its grid barrier from zero
  if (p.barrier && blockIdx.x == 0 && threadIdx.x == 0) *p.barrier = 0u;
  const int Tv = read_count(p.rows_valid, p.rows_hi, (threadIdx.x == 0 && blockIdx.x == 0) ? p.err : nullptr);
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
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
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
      const int b_row0 = p.b_loads == 2 ? n * p.b_box : n * p.n_mma;
      const int b_row1 = p.gate_row0 + n * p.b_box;  // second box (SiLU*mul only)
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
        tma_load_2d(a_dst, &map_a, bar_full(s), kb * kRBK, m * kRBM);
        tma_load_2d(b_dst, &map_b, bar_full(s), kb * kRBK, b_row0);
        if (p.b_loads == 2) tma_load_2d(b_dst + p.b_box * kRBKBytes, &map_b, bar_full(s), kb * kRBK, b_row1);
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
      const uint32_t idesc = splitk_idesc(p.n_mma);
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
  } else if (warp < 6) {
    // -------------------------------- epilogue: park the partial tile in shared memory
    // The MMAs that read the operand ring have completed once tfull fires, so the
    // ring's first bytes take the partial: row r at smem + r * pstride floats.
    // (Warps 6-11 only join the reduction below.)
    const int sub = warp & 3;  // the TMEM lane quarter this warp may read
    const int r = sub * 32 + lane;
    if (mbar_wait(bar_tfull, 0, s_abort)) {
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16);
      float* prow = reinterpret_cast<float*>(smem) + r * p.pstride;
#pragma unroll 1
      for (int c = 0; c < p.n_mma; c += 32) {
        float v[32];
        tmem_ld32(tbase + c, v);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (c + 4 * q < p.n_mma)
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
  if (p.epi == kEpiSigmoidTopK) {
    uint32_t peer[kMaxSplit];
#pragma unroll
    for (int j = 0; j < kMaxSplit; ++j) peer[j] = j < S ? map_to_rank(sbase, (uint32_t)j) : 0u;
    // the chunk histogram sits past the parked partial tile, which peers are reading
    int* s_hist = reinterpret_cast<int*>(smem + topk_hist_offset(p.pstride));
    if (p.n_out > 128) reduce_sigmoid_topk<2>(p, m, rank, S, Tv, peer, s_hist);
    else reduce_sigmoid_topk<1>(p, m, rank, S, Tv, peer, s_hist);
  } else {
    const int row0 = (int)((int64_t)rank * kRBM / S), row1 = (int)((int64_t)(rank + 1) * kRBM / S);
    // 4-column groups per row: the router's E columns, 128 z columns, or 256 output columns
    const int cols = p.epi == kEpiSilu ? p.n_mma / 2 : (p.epi == kEpiSigmoid ? p.n_out : p.n_mma);
    const int groups = (cols + 3) / 4;
    const int col_base = p.epi == kEpiSigmoid ? 0 : n * cols;  // the tile's first output column
    uint32_t peer[kMaxSplit];  // the partial tile's base in each CTA of the cluster
#pragma unroll
    for (int j = 0; j < kMaxSplit; ++j) peer[j] = j < S ? map_to_rank(sbase, (uint32_t)j) : 0u;
    for (int i = threadIdx.x; i < (row1 - row0) * groups; i += kRThreads) {
      const int rr = row0 + i / groups;
      const int c = (i % groups) * 4;
      const int t = m * kRBM + rr;
      const uint32_t off = (uint32_t)((rr * p.pstride + c) * 4);
      const float4 acc = cluster_sum4(peer, S, off);
      if (t >= Tv || col_base + c >= p.n_out) continue;
      __nv_bfloat16* orow = p.out + (int64_t)t * p.n_out + col_base;
      if (p.epi == kEpiSigmoid) {
        store4(p, orow - col_base, c, sigmoid_of_bf16_logit(acc.x), sigmoid_of_bf16_logit(acc.y),
               sigmoid_of_bf16_logit(acc.z), sigmoid_of_bf16_logit(acc.w));
      } else if (p.epi == kEpiSilu) {
        const float4 g = cluster_sum4(peer, S, off + (uint32_t)(cols * 4));  // the gate half of the tile
        // the unfused pipeline rounds the GEMM output to bf16 before silu_mul
        store4(p, p.out + (int64_t)t * p.n_out, col_base + c,
               silu_mul_f32(round_bf16(acc.x), round_bf16(g.x)), silu_mul_f32(round_bf16(acc.y), round_bf16(g.y)),
               silu_mul_f32(round_bf16(acc.z), round_bf16(g.z)), silu_mul_f32(round_bf16(acc.w), round_bf16(g.w)));
      } else {
        store4(p, p.out + (int64_t)t * p.n_out, col_base + c, acc.x, acc.y, acc.z, acc.w);
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

// How many clusters of `split` CTAs (each with `smem` bytes) the device runs at once.  A
// cluster lives inside one GPC, so this is below SMs / split for most sizes.  Cached per
// (device, split, smem).
int max_active_clusters(int split, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_tuple(dev, split, smem);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaFuncSetAttribute(splitk_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(split * 64));
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, splitk_gemm_kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a failed query leaves no sticky error behind
  cache[key] = n;
  return n;
}

// Tiles, splits and shared memory for rows x K against n_tiles tiles of N = n_mma columns.
struct SplitKPlan {
  int tmem_cols, stages, num_kb, split, pstride, m_tiles, smem;
};

SplitKPlan plan_splitk(int rows, int K, int n_mma, int n_tiles) {
  SplitKPlan q;
  q.tmem_cols = 32;
  while (q.tmem_cols < n_mma) q.tmem_cols *= 2;
  const int stage_bytes = kRABytes + n_mma * kRBKBytes;
  q.stages = kSmemBudget / stage_bytes;
  if (q.stages > kMaxStages) q.stages = kMaxStages;
  q.num_kb = (K + kRBK - 1) / kRBK;
  q.m_tiles = (rows + kRBM - 1) / kRBM;
  q.pstride = n_mma + 4;  // 4 floats of padding spread the rows over the banks
  q.smem = SplitKSmem(q.stages, n_mma).bytes + 1024;
  // splits: the cluster size S (at most a portable 8, at least kMinKb K blocks per CTA)
  // of the shortest estimated time: waves of resident clusters x (K blocks per CTA +
  // a fixed cost per CTA for its prologue, epilogue and cluster reduction), the
  // smaller S on ties.  A second wave of clusters can beat one wave of long CTAs:
  // 86 tiles on GB300 (152 SMs) run 3-way split in two waves of 50 clusters.
  const int64_t tiles = (int64_t)q.m_tiles * n_tiles;
  q.split = 1;
  double best = 0.0;
  for (int S = 1; S <= kMaxSplit; ++S) {
    if (S > 1 && q.num_kb / S < kMinKb) break;
    const int64_t clusters = S == 1 ? (int64_t)device_sm_count() : (int64_t)max_active_clusters(S, q.smem);
    if (clusters < 1) continue;
    const int64_t waves = (tiles + clusters - 1) / clusters;
    const double cost = (double)waves * ((double)q.num_kb / S + kFixedKbPerCta);
    if (S == 1 || cost < best) {
      best = cost;
      q.split = S;
    }
  }
  return q;
}

cudaError_t launch_splitk(const CUtensorMap& ma, const CUtensorMap& mb, SplitKParams p, const SplitKPlan& q,
                          int n_tiles, cudaStream_t s) {
  p.tmem_cols = q.tmem_cols;
  p.stages = q.stages;
  p.num_kb = q.num_kb;
  p.split = q.split;
  p.pstride = q.pstride;
  p.n_tiles = n_tiles;
  // the parked partial tile (and the routing chunk histogram after it) fits in the operand ring
  const int64_t parked = p.epi == kEpiSigmoidTopK ? topk_hist_offset(q.pstride) + (int64_t)p.n_out * 4
                                                 : (int64_t)kRBM * q.pstride * 4;
  if (parked > SplitKSmem(q.stages, p.n_mma).bars) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(splitk_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, q.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)q.m_tiles * n_tiles * q.split));
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = q.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = q.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, splitk_gemm_kernel, ma, mb, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

size_t router_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_router_scores(const RouterArgs& a, cudaStream_t s) {
  const int n_mma = (a.E + 15) / 16 * 16;
  const SplitKPlan q = plan_splitk(a.T, a.D, n_mma, 1);
  CUtensorMap ma, mb;
  if (!make_map_sw128(&ma, a.x, a.T, a.D, false, kRBM) || !make_map_sw128(&mb, a.w, a.E, a.D, false, n_mma))
    return cudaErrorInvalidValue;
  SplitKParams p = {};
  p.rows_hi = a.T;
  p.n_mma = n_mma;
  p.b_box = n_mma;
  p.b_loads = 1;
  p.epi = kEpiSigmoid;
  p.n_out = a.E;
  p.gate_row0 = 0;
  p.vec_store = (a.E % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 7) == 0);
  p.rows_valid = a.num_valid;
  p.out = static_cast<__nv_bfloat16*>(a.scores);
  p.err = a.err;
  return launch_splitk(ma, mb, p, q, 1, s);
}

cudaError_t launch_router_route(const RouterArgs& a, int top_k, const RouteWorkspace& w, cudaStream_t s) {
  const int n_mma = (a.E + 15) / 16 * 16;
  const SplitKPlan q = plan_splitk(a.T, a.D, n_mma, 1);
  CUtensorMap ma, mb;
  if (!make_map_sw128(&ma, a.x, a.T, a.D, false, kRBM) || !make_map_sw128(&mb, a.w, a.E, a.D, false, n_mma))
    return cudaErrorInvalidValue;
  SplitKParams p = {};
  p.rows_hi = a.T;
  p.n_mma = n_mma;
  p.b_box = n_mma;
  p.b_loads = 1;
  p.epi = kEpiSigmoidTopK;
  p.n_out = a.E;
  p.gate_row0 = 0;
  p.vec_store = (a.E % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 7) == 0);
  p.rows_valid = a.num_valid;
  p.out = static_cast<__nv_bfloat16*>(a.scores);
  p.err = a.err;
  p.top_k = top_k;
  p.chosen = w.chosen;
  p.hist_t = w.hist_t;
  p.nblk = (a.T + kChunkRows - 1) / kChunkRows;
  p.barrier = w.barrier;
  return launch_splitk(ma, mb, p, q, 1, s);
}

cudaError_t launch_dense_gemm(const DenseArgs& a, cudaStream_t s) {
  const bool silu = a.epilogue == MOE_EPILOGUE_SILU_MUL;
  const int n_mma = 256;
  const int n_out = silu ? a.N / 2 : a.N;
  const int cols = silu ? n_mma / 2 : n_mma;  // output columns per tile
  const int n_tiles = (n_out + cols - 1) / cols;
  const SplitKPlan q = plan_splitk(a.M, a.K, n_mma, n_tiles);
  CUtensorMap ma, mb;
  if (!make_map_sw128(&ma, a.x, a.M, a.K, false, kRBM) ||
      !make_map_sw128(&mb, a.w, a.N, a.K, false, silu ? n_mma / 2 : n_mma))
    return cudaErrorInvalidValue;
  SplitKParams p = {};
  p.rows_hi = a.M;
  p.n_mma = n_mma;
  p.b_box = silu ? n_mma / 2 : n_mma;
  p.b_loads = silu ? 2 : 1;
  p.epi = silu ? kEpiSilu : kEpiPlain;
  p.n_out = n_out;
  p.gate_row0 = silu ? a.N / 2 : 0;
  p.vec_store = (n_out % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.y) & 7) == 0);
  p.rows_valid = a.rows_valid;
  p.out = static_cast<__nv_bfloat16*>(a.y);
  p.err = a.err;
  return launch_splitk(ma, mb, p, q, n_tiles, s);
}

}  // namespace moe
