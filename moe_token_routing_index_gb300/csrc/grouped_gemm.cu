// Grouped GEMM of the routed experts on the 5th-generation tensor cores
// (mslk/moe/layers.py, MetaShufflingMoE._routed_expert: grouped_gemm and
// grouped_gemm_fp8_rowwise over w13 and w2).
//
// y[r, n] = sum_k x[r, k] * w[e, n, k] for the rows r of expert e, i.e. a
// "TN" GEMM per expert with both operands K-major.
//
// Kernel structure (one CTA per SM, persistent, 6 warps):
//   warp 0     TMA producer: 128-row A tile (routed rows) and two 128-row B
//              tiles (weight rows) of 128 bytes of K per stage, 128B-swizzled,
//              into a 4-stage shared-memory ring guarded by mbarriers.
//   warp 1     MMA issuer: tcgen05.mma (M=128, N=256, fp32 accumulate) into one
//              of two 256-column accumulators in tensor memory; tcgen05.commit
//              frees the smem stage and, after the last K block, hands the
//              accumulator to the epilogue.  Also allocates/frees the 512
//              tensor-memory columns.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator rows (one TMEM lane per
//              thread), optional FP8 dequantisation, optional SiLU*mul of the
//              two halves, bf16 rounding, stores with row/column masks.
// Tiles: for each expert e, ceil(count_e / 128) row tiles x the N tiles;
// consecutive tile ids walk the row tiles of one weight slice first, so CTAs
// running together share that slice in L2, in bands of row tiles whose x rows
// fit a share of L2 (band_order).  Every CTA derives the tile list from the
// device counts itself (no host synchronisation).
//
// Every mbarrier wait is bounded (1 s of %globaltimer); on expiry the kernel
// records MOE_DEVERR_TIMEOUT, all roles stop, in-flight copies and MMAs are
// drained with bounded waits, and tensor memory is freed before exit.
#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;            // rows of a tile (routed rows)
constexpr int kBN = 256;            // accumulator columns (MMA N)
constexpr int kBKBytes = 128;       // bytes of K per stage (one 128B swizzle atom per row)
constexpr int kStages = 4;
constexpr int kAccBufs = 2;
constexpr int kTmemCols = kAccBufs * kBN;  // 512
constexpr int kThreads = 192;
constexpr int kABytes = kBM * kBKBytes;          // 16 KB
constexpr int kBBytes = kBN * kBKBytes;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;   // 48 KB
constexpr int kMaxExperts = 1024;
// Per epilogue warp: a staging block of 32 rows x 128 bytes (one 64-column bf16
// chunk of the warp's rows, 16-byte pieces XOR-swizzled by row: the 128-byte
// swizzle of a TMA tile, so a block is 1024-byte aligned) and the tile's column
// scales (FP8).  Layout: the 4 staging blocks, then the 4 scale arrays.
constexpr int kEpiStageBytes = 32 * 128;
constexpr int kEpiScaleBytes = kBN * 4;
constexpr int kEpiBytes = 4 * (kEpiStageBytes + kEpiScaleBytes);  // 20 KB

struct SmemLayout {
  // offsets from the 1024-aligned base
  static constexpr int a = 0;
  static constexpr int b = a + kStages * kABytes;
  static constexpr int epi = b + kStages * kBBytes;         // epilogue staging blocks and scales
  static constexpr int bars = epi + kEpiBytes;              // full[S], empty[S], tfull[2], tempty[2], drain
  static constexpr int nbars = 2 * kStages + 2 * kAccBufs + 1;
  static constexpr int misc = bars + nbars * 8;             // tmem base, abort flag, total tiles, pad
  static constexpr int sched = misc + 16;                   // tile_start[E+1], row_off[E+1], mtiles[E]
  static constexpr int bytes_for(int E) { return sched + (3 * E + 2) * 4; }
};

// ------------------------------------------------------------ PTX helpers

using namespace tc;

// Instruction descriptor: fp32 accumulate, A/B K-major, M = 128, N = 256.
template <bool FP8>
__device__ __forceinline__ uint32_t instr_desc() {
  const uint32_t fmt = FP8 ? 0u /*E4M3*/ : 1u /*BF16*/;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

// ------------------------------------------------------------- scheduling

struct Tile {
  int expert, row0, rows, n_idx;
};

// The row-tile and N-tile index of tile `local` of an expert with mt row tiles and
// n_tiles N tiles.  The tiles are walked in bands of `band` row tiles; inside a band
// N-major with the row tiles innermost, so the CTAs running together share one weight
// slice and the band's rows of x, and every other band walks N backwards, so that it
// starts on the weight slices the band before read last, while they are in L2.
// band >= mt: one band (N-major over all row tiles).
__device__ __forceinline__ void band_order(int local, int mt, int n_tiles, int band, int* m_idx, int* n_idx) {
  const int b = local / (band * n_tiles);
  const int bm = min(band, mt - b * band);
  const int lb = local - b * band * n_tiles;
  int n = lb / bm;
  if (b & 1) n = n_tiles - 1 - n;
  *n_idx = n;
  *m_idx = b * band + lb % bm;
}

// Decode tile id -> (expert, first routed row, valid rows, N-tile index).
__device__ __forceinline__ Tile decode_tile(int tile, int E, int n_tiles, int band, const int* tile_start,
                                            const int* row_off, const int* mtiles) {
  const int mt_global = tile / n_tiles;  // which row tile, counting over experts
  int lo = 0, hi = E - 1;                // find e with tile_start[e] <= mt_global < tile_start[e + 1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= mt_global) lo = mid;
    else hi = mid - 1;
  }
  const int e = lo;
  int m_idx, n_idx;
  band_order(tile - tile_start[e] * n_tiles, mtiles[e], n_tiles, band, &m_idx, &n_idx);
  Tile t;
  t.expert = e;
  t.n_idx = n_idx;
  t.row0 = row_off[e] + m_idx * kBM;
  const int rows_left = row_off[e + 1] - t.row0;
  t.rows = rows_left < kBM ? rows_left : kBM;
  return t;
}

// ----------------------------------------------------------------- kernel

// One grouped GEMM of a launch.  A launch runs one phase, or two: the w13 GEMM
// (SiLU*mul epilogue into z) and then the w2 GEMM reading z.
struct Phase {
  int N, K;           // GEMM output columns (2H for SILU_MUL) and reduction length
  int epi;            // MOE_EPILOGUE_*
  int n_out;          // stored columns: N, or N / 2 for SILU_MUL
  int n_tile_cols;    // stored columns per tile
  int n_tiles;        // tiles along N
  int band;           // row tiles per band of the tile order (band_order)
  int num_kb;         // K blocks
  __nv_bfloat16* y;   // [a_max, n_out], or [T_out, n_out] when scattering
  const float* x_scale;
  const float* w_scale;
  const int32_t* scatter;  // NONE epilogue only: row r goes to y[scatter[r]] (top_k = 1 combine)
  int T_out;               // rows of y when scattering
  int accumulate;          // scatter: add into y (fp32 add of the bf16 row, one rounding) or overwrite
  int tma_store;           // y has a store tensor map (rows of a_max, 32 x 64 boxes): full row chunks use TMA
  int packed;              // weights in the tile-packed layout (every 128-row x 128-byte box contiguous)
};

// TMA coordinates of the weight box (first row `row`, a multiple of 128 when
// packed; K block kb, first element kc).  Row-major weights: (kc, row).  Packed
// weights are a [boxes * 128, 128-byte] matrix whose box (row / 128, kb) starts
// at row ((row / 128) * num_kb + kb) * 128.
__device__ __forceinline__ void weight_box(const Phase& p, int row, int kb, int kc, int* c0, int* c1) {
  if (p.packed) {
    *c0 = 0;
    *c1 = ((row >> 7) * p.num_kb + kb) * kBM;
  } else {
    *c0 = kc;
    *c1 = row;
  }
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Epilogue of one accumulator tile for one warp: its 32 rows of the tile
// (TMEM lanes of the warp's quarter; the calling thread's row is warp_row0 +
// lane), all columns of the phase's N tile.  FP8 scales, the SiLU*mul of the two
// halves or the fused combine, then bf16 stores.  Each 64-column chunk goes
// through the warp's staging block, so that the warp stores 4 rows x 128
// contiguous bytes per instruction instead of 32 rows x 16 bytes.  With a store
// tensor map and all 32 rows inside the tile, lane 0 writes the chunk with one
// TMA store instead (asynchronous; the block is reused once the store has read it).
template <bool FP8>
__device__ __forceinline__ void epilogue_tile(const Phase& p, const Tile& t, int warp_row0, int lane, uint32_t tbase,
                                              uint8_t* stage, float* wsc_s, const CUtensorMap* map_y,
                                              unsigned int* err) {
  const int row_in_tile = warp_row0 + lane;
  const bool row_ok = row_in_tile < t.rows;
  const int row = t.row0 + row_in_tile;
  const int n_out = p.n_out;
  const int col0 = t.n_idx * p.n_tile_cols;
  const bool silu = p.epi == MOE_EPILOGUE_SILU_MUL;
  float xs = 1.0f;
  if (FP8 && row_ok) xs = __ldg(p.x_scale + row);
  if (FP8) {
    // the tile's column scales, clamped to valid columns (SiLU*mul: w_in block, then gate block)
    const float* wsc = p.w_scale + (int64_t)t.expert * p.N;
    const int H = p.N / 2;
#pragma unroll
    for (int k = 0; k < kBN / 32; ++k) {
      const int i = lane + 32 * k;
      const int col = silu ? (i < kBN / 2 ? min(col0 + i, H - 1) : H + min(col0 + i - kBN / 2, H - 1))
                           : min(col0 + i, n_out - 1);
      wsc_s[i] = __ldg(wsc + col);
    }
    __syncwarp();
  }
  // destination row of each tile row: its own, or with the fused combine (top_k = 1)
  // its token's row; -1: nothing to store
  int dst = row_ok ? row : -1;
  if (p.scatter && row_ok) {
    const int tok = __ldg(p.scatter + row);
    if ((unsigned)tok < (unsigned)p.T_out) {
      dst = tok;
    } else {
      dst = -1;
      flag_error(err, MOE_DEVERR_BAD_INDEX);
    }
  }
  // this lane stores rows (lane >> 3) + 4 j of the warp's 32, 16-byte piece lane & 7 of each chunk
  int dst_j[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) dst_j[j] = __shfl_sync(0xffffffffu, dst, (lane >> 3) + 4 * j);
  const bool add = p.scatter && p.accumulate;
  const bool tma = p.tma_store && warp_row0 + 32 <= t.rows;
  const int piece = lane & 7;
  const int out_cols = silu ? kBN / 2 : kBN;
#pragma unroll 1
  for (int c = 0; c < out_cols; c += 64) {
    if (p.tma_store) {  // the previous TMA store from the staging block has read it
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
    }
    // the thread's row: 64 output columns as bf16 into staging row `lane`
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int cc = c + 32 * h;
      float z[32];
      if (silu) {
        float v1[32];
        tmem_ld32(tbase + cc, z);
        tmem_ld32(tbase + kBN / 2 + cc, v1);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          float4 w0 = make_float4(1.f, 1.f, 1.f, 1.f), w1 = w0;
          if (FP8) {
            w0 = reinterpret_cast<const float4*>(wsc_s + cc)[i4];
            w1 = reinterpret_cast<const float4*>(wsc_s + kBN / 2 + cc)[i4];
          }
          const float ws0[4] = {w0.x, w0.y, w0.z, w0.w}, ws1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = 4 * i4 + u;
            float a0 = z[i], a1 = v1[i];
            if (FP8) {
              a0 = __fmul_rn(__fmul_rn(a0, xs), ws0[u]);
              a1 = __fmul_rn(__fmul_rn(a1, xs), ws1[u]);
            }
            // the unfused pipeline rounds the GEMM output to bf16 before silu_mul
            a0 = __bfloat162float(__float2bfloat16_rn(a0));
            a1 = __bfloat162float(__float2bfloat16_rn(a1));
            z[i] = silu_mul_f32(a0, a1);
          }
        }
      } else {
        tmem_ld32(tbase + cc, z);
        if (FP8) {
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 w = reinterpret_cast<const float4*>(wsc_s + cc)[i4];
            z[4 * i4 + 0] = __fmul_rn(__fmul_rn(z[4 * i4 + 0], xs), w.x);
            z[4 * i4 + 1] = __fmul_rn(__fmul_rn(z[4 * i4 + 1], xs), w.y);
            z[4 * i4 + 2] = __fmul_rn(__fmul_rn(z[4 * i4 + 2], xs), w.z);
            z[4 * i4 + 3] = __fmul_rn(__fmul_rn(z[4 * i4 + 3], xs), w.w);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int k = 4 * h + q;  // 16-byte piece of the 128-byte row chunk
        *reinterpret_cast<uint4*>(stage + lane * 128 + ((k ^ (lane & 7)) << 4)) = f32_to_bf16x8(z + 8 * q);
      }
    }
    if (tma) {
      fence_proxy_async_shared();  // this lane's staging writes, visible to the TMA store
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map_y, smem_u32(stage), col0 + c, t.row0 + warp_row0);
        bulk_commit_group();
      }
      continue;
    }
    __syncwarp();
    // the warp's rows: 4 rows x 128 bytes per store instruction
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = (lane >> 3) + 4 * j;
      const int col = col0 + c + 8 * piece;
      if (dst_j[j] >= 0 && col < n_out) {
        uint4 o = *reinterpret_cast<const uint4*>(stage + r * 128 + ((piece ^ (r & 7)) << 4));
        uint4* d = reinterpret_cast<uint4*>(p.y + (int64_t)dst_j[j] * n_out + col);
        if (add) {  // as moe_scatter_add on the bf16 GEMM output: fp32 add, one rounding
          float fo[8], fi[8];
          bf16x8_to_f32(*d, fo);
          bf16x8_to_f32(o, fi);
#pragma unroll
          for (int i = 0; i < 8; ++i) fo[i] = __fadd_rn(fo[i], fi[i]);
          o = f32_to_bf16x8(fo);
        }
        *d = o;
      }
    }
    __syncwarp();  // the staging block is rewritten by the next chunk
  }
}

template <bool FP8, int NPHASE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_b0,
    const __grid_constant__ CUtensorMap map_a1, const __grid_constant__ CUtensorMap map_b1,
    const __grid_constant__ CUtensorMap map_y, const int32_t* __restrict__ counts, const Phase p0, const Phase p1,
    int E, int a_max, int* done, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmemLayout::bars);
  auto bar_full = [&](int s) { return smem_u32(&bars[s]); };
  auto bar_empty = [&](int s) { return smem_u32(&bars[kStages + s]); };
  auto bar_tfull = [&](int b) { return smem_u32(&bars[2 * kStages + b]); };
  auto bar_tempty = [&](int b) { return smem_u32(&bars[2 * kStages + kAccBufs + b]); };
  const uint32_t bar_drain = smem_u32(&bars[2 * kStages + 2 * kAccBufs]);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + SmemLayout::misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + SmemLayout::misc + 4);
  int* s_total = reinterpret_cast<int*>(smem + SmemLayout::misc + 8);
  int* tile_start = reinterpret_cast<int*>(smem + SmemLayout::sched);  // [E + 1]
  int* row_off = tile_start + (E + 1);                                  // [E + 1]
  int* mtiles = row_off + (E + 1);                                      // [E]

  // ---- prologue: barriers, tensor memory, the tile list from the counts
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(bar_tfull(b), 1);
      mbar_init(bar_tempty(b), 4);  // one arrive per epilogue warp
    }
    mbar_init(bar_drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tma_prefetch_desc(&map_a0);
    tma_prefetch_desc(&map_b0);
    if (NPHASE == 2) {
      tma_prefetch_desc(&map_a1);
      tma_prefetch_desc(&map_b1);
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 2) {
    // Row offsets and row-tile starts: warp-wide exclusive scans over the experts.
    // Counts are clamped so that no tile reaches past a_max rows.
    int run_rows = 0, run_tiles = 0;
    bool bad = false;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int c = e < E ? counts[e] : 0;
      if (c < 0) {
        c = 0;
        bad = true;
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int start = run_rows + incl - c;
      if (start > a_max) start = a_max;
      int end = run_rows + incl;
      if (end > a_max) {
        end = a_max;
        bad = true;
      }
      const int mt = (end - start + kBM - 1) / kBM;
      int tincl = mt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, tincl, o);
        if (lane >= o) tincl += v;
      }
      if (e < E) {
        row_off[e] = start;
        tile_start[e] = run_tiles + tincl - mt;
        mtiles[e] = mt;
      }
      run_rows = min(__shfl_sync(0xffffffffu, run_rows + incl, 31), a_max);
      run_tiles += __shfl_sync(0xffffffffu, tincl, 31);
    }
    if (lane == 0) {
      row_off[E] = run_rows;
      tile_start[E] = run_tiles;
      *s_total = run_tiles;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) flag_error(err, MOE_DEVERR_BAD_COUNT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *s_tmem;
  const int tiles0 = *s_total * p0.n_tiles;
  const int total_tiles = tiles0 + (NPHASE == 2 ? *s_total * p1.n_tiles : 0);
  const int elems_per_kb = FP8 ? kBKBytes : kBKBytes / 2;
  // (phase, tile within the phase) of a tile id: phase-0 tiles come first.
  auto locate = [&](int tile, int* ph) {
    *ph = (NPHASE == 2 && tile >= tiles0) ? 1 : 0;
    const Phase& p = *ph ? p1 : p0;
    return decode_tile(*ph ? tile - tiles0 : tile, E, p.n_tiles, p.band, tile_start, row_off, mtiles);
  };

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int s = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;  // per stage: issued since start, parity of that issue
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        int ph;
        const Tile t = locate(tile, &ph);
        const Phase& p = ph ? p1 : p0;
        const CUtensorMap* ma = ph ? &map_a1 : &map_a0;
        const CUtensorMap* mb = ph ? &map_b1 : &map_b0;
        if (NPHASE == 2 && ph == 1) {
          // z rows of this expert come from phase-0 tiles of other CTAs: wait
          // until all of them (4 epilogue warps x row tiles x N tiles) are stored.
          const int target = 4 * mtiles[t.expert] * p0.n_tiles;
          const uint64_t t0 = global_timer_ns();
          for (uint32_t i = 0; ld_acquire(done + t.expert) < target; ++i) {
            if ((i & 63) == 63 && (*s_abort || global_timer_ns() - t0 > kWaitTimeoutNs)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          fence_proxy_async_global();  // the TMA reads below observe those stores
        }
        int b_row0, b_row1;
        if (p.epi == MOE_EPILOGUE_SILU_MUL) {
          b_row0 = t.expert * p.N + t.n_idx * (kBN / 2);
          b_row1 = b_row0 + p.N / 2;
        } else {
          b_row0 = t.expert * p.N + t.n_idx * kBN;
          b_row1 = b_row0 + kBN / 2;
        }
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(bar_empty(s), phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + SmemLayout::a + s * kABytes;
          const uint32_t b_dst = sbase + SmemLayout::b + s * kBBytes;
          mbar_arrive_expect_tx(bar_full(s), kStageBytes);
          const int kc = kb * elems_per_kb;
          tma_load_2d(a_dst, ma, bar_full(s), kc, t.row0);
          int w0, w1;
          weight_box(p, b_row0, kb, kc, &w0, &w1);
          tma_load_2d(b_dst, mb, bar_full(s), w0, w1);
          weight_box(p, b_row1, kb, kc, &w0, &w1);
          tma_load_2d(b_dst + kBBytes / 2, mb, bar_full(s), w0, w1);
          issued_mask |= 1u << s;
          issued_parity = (issued_parity & ~(1u << s)) | (phase << s);
          if (++s == kStages) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        flag_error(err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        // Let the copies already issued land before the CTA can exit.
        for (int i = 0; i < kStages; ++i)
          if ((issued_mask >> i) & 1u) mbar_wait(bar_full(i), (issued_parity >> i) & 1u, nullptr, kDrainTimeoutNs);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = instr_desc<FP8>();
      int s = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued_any = false;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const int num_kb = (NPHASE == 2 && tile >= tiles0) ? p1.num_kb : p0.num_kb;
        if (!mbar_wait(bar_tempty(acc), acc_phase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(bar_full(s), phase, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + SmemLayout::a + s * kABytes;
          const uint32_t b_addr = sbase + SmemLayout::b + s * kBBytes;
#pragma unroll
          for (int kk = 0; kk < kBKBytes / 32; ++kk) {  // 32 bytes of K per instruction
            mma_issue<FP8>(d, smem_desc_sw128(a_addr + kk * 32), smem_desc_sw128(b_addr + kk * 32), idesc,
                           (kb | kk) != 0);
          }
          issued_any = true;
          mma_commit(bar_empty(s));
          if (++s == kStages) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(bar_tfull(acc));
        if (++acc == kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        flag_error(err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        if (issued_any) {  // wait for the MMAs in flight before tensor memory is freed
          mma_commit(bar_drain);
          mbar_wait(bar_drain, 0, nullptr, kDrainTimeoutNs);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int sub = warp & 3;                // TMEM lane quarter this warp may access
    uint8_t* stage = smem + SmemLayout::epi + (warp - 2) * kEpiStageBytes;
    float* wsc_s = reinterpret_cast<float*>(smem + SmemLayout::epi + 4 * kEpiStageBytes + (warp - 2) * kEpiScaleBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int ph;
      const Tile t = locate(tile, &ph);
      const Phase& p = ph ? p1 : p0;
      if (!mbar_wait(bar_tfull(acc), acc_phase, s_abort)) {
        if (lane == 0) flag_error(err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * kBN);
      epilogue_tile<FP8>(p, t, sub * 32, lane, tbase, stage, wsc_s, &map_y, err);
      tc_fence_before();
      if (NPHASE == 2 && ph == 0) {
        // publish this warp's share of the tile's z rows to the phase-1 producers
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async_global();
          red_release_add(done + t.expert, 1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty(acc));
      if (++acc == kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group0();  // this warp's TMA stores are complete before the block exits
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
  if (NPHASE == 2 && threadIdx.x == 0) {
    // The last CTA to finish (every other CTA is past its waits on the counters)
    // leaves done[0..E] zero for the next launch, on every path including aborts.
    __threadfence();
    if (atomicAdd(done + E, 1) == (int)gridDim.x - 1) {
      for (int e = 0; e <= E; ++e) done[e] = 0;
      __threadfence();
    }
  }
}

// ------------------------------------------------- CTA-pair kernel (2 SMs)
//
// A cluster of two CTAs computes one 256 x 256 tile with tcgen05.mma.cta_group::2:
// CTA r holds rows [128 r, 128 r + 128) of the A tile and weight rows
// [128 r, 128 r + 128) of the 256-row B tile (for SiLU*mul: CTA 0 the w_in block,
// CTA 1 the gate block); the leader (rank 0) issues the M = 256, N = 256 MMAs,
// which read both CTAs' shared memory and leave each CTA's 128 rows x 256
// columns in its own tensor memory.  Per CTA a K block moves 32 KB (A 16 + B 16)
// instead of 48, and six stages fit.
//   - TMEM is allocated and freed collectively by the pair (cta_group::2).
//   - Both CTAs' TMA loads complete on the leader's full barrier, whose single
//     arrival (expect_tx of both CTAs' bytes) comes from the leader's producer.
//   - The leader's commits are multicast to the empty and tensor-full barriers
//     of both CTAs; both CTAs' epilogue warps arrive on the leader's
//     tensor-empty barrier (8 arrivals).
//   - Before exit each producer waits until its last stages were consumed, then
//     the pair meets at a cluster barrier and frees TMEM together.
constexpr int kPairStages = 6;
constexpr int kPairBM = 2 * kBM;                           // rows of a pair tile
constexpr int kPairABytes = kBM * kBKBytes;                // 16 KB: this CTA's A rows
constexpr int kPairBBytes = (kBN / 2) * kBKBytes;          // 16 KB: this CTA's half of B
constexpr int kPairStageBytes = kPairABytes + kPairBBytes;  // 32 KB

struct PairSmem {
  static constexpr int a = 0;
  static constexpr int b = a + kPairStages * kPairABytes;
  static constexpr int epi = b + kPairStages * kPairBBytes;   // epilogue staging blocks and scales
  static constexpr int bars = epi + kEpiBytes;                // full[S], empty[S], tfull[2], tempty[2], drain
  static constexpr int nbars = 2 * kPairStages + 2 * kAccBufs + 1;
  static constexpr int misc = bars + nbars * 8;
  static constexpr int sched = misc + 16;
  static constexpr int bytes_for(int E) { return sched + (3 * E + 2) * 4; }
};

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory, completing on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

template <bool FP8>
__device__ __forceinline__ uint32_t instr_desc_pair() {
  const uint32_t fmt = FP8 ? 0u : 1u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kPairBM >> 4) << 24);
}

template <bool FP8>
__device__ __forceinline__ void mma_issue_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (FP8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  }
}

// Arrive on the barrier at this shared-memory offset in both CTAs of the pair once
// the leader's MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)0x3)
      : "memory");
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_pair_kernel(
    const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
    const __grid_constant__ CUtensorMap map_y, const int32_t* __restrict__ counts, const Phase p, int E, int a_max,
    unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PairSmem::bars);
  auto bar_full = [&](int s) { return smem_u32(&bars[s]); };
  auto bar_empty = [&](int s) { return smem_u32(&bars[kPairStages + s]); };
  auto bar_tfull = [&](int b) { return smem_u32(&bars[2 * kPairStages + b]); };
  auto bar_tempty = [&](int b) { return smem_u32(&bars[2 * kPairStages + kAccBufs + b]); };
  const uint32_t bar_drain = smem_u32(&bars[2 * kPairStages + 2 * kAccBufs]);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + PairSmem::misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + PairSmem::misc + 4);
  int* s_total = reinterpret_cast<int*>(smem + PairSmem::misc + 8);
  int* tile_start = reinterpret_cast<int*>(smem + PairSmem::sched);  // [E + 1]
  int* row_off = tile_start + (E + 1);                                // [E + 1]
  int* mtiles = row_off + (E + 1);                                    // [E]

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(bar_tfull(b), 1);
      mbar_init(bar_tempty(b), 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(bar_drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (warp == 2) {
    // 256-row pair tiles per expert (the same scan as the single-CTA kernel).
    int run_rows = 0, run_tiles = 0;
    bool bad = false;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int c = e < E ? counts[e] : 0;
      if (c < 0) {
        c = 0;
        bad = true;
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int start = run_rows + incl - c;
      if (start > a_max) start = a_max;
      int end = run_rows + incl;
      if (end > a_max) {
        end = a_max;
        bad = true;
      }
      const int mt = (end - start + kPairBM - 1) / kPairBM;
      int tincl = mt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, tincl, o);
        if (lane >= o) tincl += v;
      }
      if (e < E) {
        row_off[e] = start;
        tile_start[e] = run_tiles + tincl - mt;
        mtiles[e] = mt;
      }
      run_rows = min(__shfl_sync(0xffffffffu, run_rows + incl, 31), a_max);
      run_tiles += __shfl_sync(0xffffffffu, tincl, 31);
    }
    if (lane == 0) {
      row_off[E] = run_rows;
      tile_start[E] = run_tiles;
      *s_total = run_tiles;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) flag_error(err, MOE_DEVERR_BAD_COUNT);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA arrival
  tc_fence_after();

  const uint32_t tmem_base = *s_tmem;
  const int total_tiles = *s_total * p.n_tiles;
  const int elems_per_kb = FP8 ? kBKBytes : kBKBytes / 2;
  // decode_tile works in 128-row units; a pair tile is decoded in 256-row units
  auto locate = [&](int tile) {
    const int mt_global = tile / p.n_tiles;
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= mt_global) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo;
    int m_idx, n_idx;
    band_order(tile - tile_start[e] * p.n_tiles, mtiles[e], p.n_tiles, p.band, &m_idx, &n_idx);
    Tile t;
    t.expert = e;
    t.n_idx = n_idx;
    t.row0 = row_off[e] + m_idx * kPairBM;
    const int rows_left = row_off[e + 1] - t.row0;
    t.rows = rows_left < kPairBM ? rows_left : kPairBM;
    return t;
  };

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t full_leader0 = map_to_rank(bar_full(0), 0);
      int s = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int tile = cid; tile < total_tiles && ok; tile += nclusters) {
        const Tile t = locate(tile);
        int b_row;
        if (p.epi == MOE_EPILOGUE_SILU_MUL)
          b_row = t.expert * p.N + (int)rank * (p.N / 2) + t.n_idx * (kBN / 2);
        else
          b_row = t.expert * p.N + t.n_idx * kBN + (int)rank * (kBN / 2);
        const int a_row = t.row0 + (int)rank * kBM;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(bar_empty(s), phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(bar_full(s), 2 * kPairStageBytes);
          const uint32_t full_leader = full_leader0 + (uint32_t)(s * 8);
          const int kc = kb * elems_per_kb;
          tma_load_2d_pair(sbase + PairSmem::a + s * kPairABytes, &map_a, full_leader, kc, a_row);
          int w0, w1;
          weight_box(p, b_row, kb, kc, &w0, &w1);
          tma_load_2d_pair(sbase + PairSmem::b + s * kPairBBytes, &map_b, full_leader, w0, w1);
          issued_mask |= 1u << s;
          issued_parity = (issued_parity & ~(1u << s)) | (phase << s);
          if (++s == kPairStages) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      if (ok) {
        // every stage this CTA filled has been consumed by the pair's MMAs
        for (int i = 0; i < kPairStages; ++i)
          if ((issued_mask >> i) & 1u && !mbar_wait(bar_empty(i), (issued_parity >> i) & 1u, s_abort)) ok = false;
      }
      if (!ok) {
        flag_error(err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        spin_ns(kDrainTimeoutNs);  // copies in flight complete on the leader's barrier: give them time to land
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA (leader)
    if (lane == 0 && leader) {
      const uint32_t idesc = instr_desc_pair<FP8>();
      int s = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued_any = false;
      for (int tile = cid; tile < total_tiles && ok; tile += nclusters) {
        if (!mbar_wait(bar_tempty(acc), acc_phase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(bar_full(s), phase, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + PairSmem::a + s * kPairABytes;
          const uint32_t b_addr = sbase + PairSmem::b + s * kPairBBytes;
#pragma unroll
          for (int kk = 0; kk < kBKBytes / 32; ++kk)
            mma_issue_pair<FP8>(d, smem_desc_sw128(a_addr + kk * 32), smem_desc_sw128(b_addr + kk * 32), idesc,
                                (kb | kk) != 0);
          issued_any = true;
          mma_commit_pair_both(bar_empty(s));
          if (++s == kPairStages) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_both(bar_tfull(acc));
        if (++acc == kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        flag_error(err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        if (issued_any) {  // the MMAs in flight finish before tensor memory is freed
          mma_commit_pair_both(bar_drain);
          mbar_wait(bar_drain, 0, nullptr, kDrainTimeoutNs);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue (both CTAs)
    const int sub = warp & 3;
    uint8_t* stage = smem + PairSmem::epi + (warp - 2) * kEpiStageBytes;
    float* wsc_s = reinterpret_cast<float*>(smem + PairSmem::epi + 4 * kEpiStageBytes + (warp - 2) * kEpiScaleBytes);
    const uint32_t tempty_leader0 = map_to_rank(bar_tempty(0), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cid; tile < total_tiles; tile += nclusters) {
      const Tile t = locate(tile);
      if (!mbar_wait(bar_tfull(acc), acc_phase, s_abort)) {
        if (lane == 0) flag_error(err, MOE_DEVERR_TIMEOUT);
        *s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * kBN);
      epilogue_tile<FP8>(p, t, (int)rank * kBM + sub * 32, lane, tbase, stage, wsc_s, &map_y, err);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader0 + (uint32_t)(acc * 8));
      if (++acc == kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group0();  // this warp's TMA stores are complete before the block exits
  }

  // ---- teardown: the pair meets, then frees its tensor memory together
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
}

// ------------------------------------------------------------------- host

// Row-major [rows, cols] matrix of 1- or 2-byte elements, box of 128 rows x 128 bytes, 128B swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, bool fp8) {
  return make_map_sw128(map, base, rows, cols, fp8, kBM);
}

// Weights [rows, K], row-major or tile-packed (see pack_weights_kernel).
bool make_weight_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, bool fp8, bool packed) {
  if (!packed) return make_map(map, base, rows, K, fp8);
  const int64_t kb = (K * (fp8 ? 1 : 2) + kBKBytes - 1) / kBKBytes;
  return make_map(map, base, (rows + kBM - 1) / kBM * kb * kBM, kBKBytes / (fp8 ? 1 : 2), fp8);
}

// Tile-packed weights: for rows r of a [rows, K] matrix and 128-byte column
// blocks c (kb of them, the last zero-padded), box (r / 128, c) holds rows
// r / 128 * 128 .. + 127 (zero rows past the end) as 128 contiguous 128-byte rows,
// boxes in (row block, column block) order.  One thread per 16-byte piece.
__global__ void pack_weights_kernel(const uint8_t* __restrict__ w, int64_t rows, int64_t row_bytes, int64_t kb,
                                    uint4* __restrict__ out, int64_t pieces) {
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < pieces; u += (int64_t)gridDim.x * blockDim.x) {
    const int piece = (int)(u & 7);
    const int64_t box_row = (u >> 3) & (kBM - 1);
    const int64_t box = u >> 10;  // 8 pieces x 128 rows per box
    const int64_t c = box % kb, rb = box / kb;
    const int64_t r = rb * kBM + box_row, off = c * kBKBytes + piece * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows && off < row_bytes) v = *reinterpret_cast<const uint4*>(w + r * row_bytes + off);
    out[u] = v;
  }
}

// Bytes of x rows that one band of the tile order may span: on the fine-grained w13
// GEMM (K = 7168 bf16, 8 experts of 4096 rows) bands of 8 pair row tiles (29 MB of x)
// moved the least DRAM traffic, 2.06 GB per launch against 2.51 GB in one band per
// expert; 6 and 10 row tiles moved 2.23 and 2.17 GB.
constexpr int64_t kBandBytes = 30ll << 20;

int band_rows_tiles(int tile_rows, int K, bool fp8) {
  const int64_t per_tile = (int64_t)tile_rows * K * (fp8 ? 1 : 2);
  const int64_t b = kBandBytes / (per_tile > 0 ? per_tile : 1);
  return (int)(b < 1 ? 1 : (b > 1024 ? 1024 : b));
}

Phase make_phase(int N, int K, int epi, bool fp8, void* y, const float* xs, const float* ws) {
  Phase p;
  p.band = band_rows_tiles(kBM, K, fp8);
  p.N = N;
  p.K = K;
  p.epi = epi;
  p.n_out = epi == MOE_EPILOGUE_SILU_MUL ? N / 2 : N;
  p.n_tile_cols = epi == MOE_EPILOGUE_SILU_MUL ? kBN / 2 : kBN;
  p.n_tiles = (p.n_out + p.n_tile_cols - 1) / p.n_tile_cols;
  const int elems = fp8 ? kBKBytes : kBKBytes / 2;
  p.num_kb = (K + elems - 1) / elems;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.x_scale = xs;
  p.w_scale = ws;
  p.scatter = nullptr;
  p.T_out = 0;
  p.accumulate = 0;
  p.tma_store = 0;
  p.packed = 0;
  return p;
}

template <bool FP8, int NPHASE>
cudaError_t launch_phases(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1,
                          const CUtensorMap& b1, const CUtensorMap& y, const int32_t* counts, const Phase& p0,
                          const Phase& p1, int E, int a_max, int* done, unsigned int* err, cudaStream_t s) {
  const int smem = SmemLayout::bytes_for(E) + 1024;
  auto kern = grouped_gemm_kernel<FP8, NPHASE>;
  // The attribute is per device; setting it on every call is cheap and keeps multi-device use correct.
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int64_t tiles_ub = 0;
  const int64_t mt_ub = (int64_t)(a_max + kBM - 1) / kBM + E;
  tiles_ub += mt_ub * p0.n_tiles;
  if (NPHASE == 2) tiles_ub += mt_ub * p1.n_tiles;
  const int sms = device_sm_count();
  const int grid = (int)(tiles_ub < sms ? tiles_ub : sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  // two phases: phase-1 tiles wait on phase-0 tiles of other CTAs, so all CTAs must be
  // resident at once.  One phase: a plain launch, after the previous kernel of the stream
  // (programmatic dependent launch made the steps slower here: 0.3-2.5% eager, up to 4.4%
  // under CUDA-graph replay)
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = NPHASE == 2 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, a0, b0, a1, b1, y, counts, p0, p1, E, a_max, done, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool FP8>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y, const int32_t* counts,
                        const Phase& p, int E, int a_max, unsigned int* err, cudaStream_t s) {
  const int smem = PairSmem::bytes_for(E) + 1024;
  auto kern = grouped_gemm_pair_kernel<FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * (device_sm_count() / 2));
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorNotSupported;
  const int64_t tiles_ub = ((int64_t)(a_max + kPairBM - 1) / kPairBM + E) * p.n_tiles;
  const int nclusters = (int)(tiles_ub < max_clusters ? tiles_ub : max_clusters);
  cfg.gridDim = dim3(2 * nclusters);
  e = cudaLaunchKernelEx(&cfg, kern, a, b, y, counts, p, E, a_max, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

size_t packed_weights_bytes(int64_t rows, int64_t K, bool fp8) {
  const int64_t kb = (K * (fp8 ? 1 : 2) + kBKBytes - 1) / kBKBytes;
  return (size_t)((rows + kBM - 1) / kBM * kb) * kBM * kBKBytes;
}

cudaError_t launch_pack_weights(const void* w, int64_t rows, int64_t K, bool fp8, void* out, cudaStream_t s) {
  const int64_t row_bytes = K * (fp8 ? 1 : 2);
  const int64_t kb = (row_bytes + kBKBytes - 1) / kBKBytes;
  const int64_t pieces = (int64_t)packed_weights_bytes(rows, K, fp8) / 16;
  if (pieces == 0) return cudaSuccess;
  const int64_t want = (pieces + 255) / 256, cap = (int64_t)device_sm_count() * 16;
  pack_weights_kernel<<<(int)(want < cap ? want : cap), 256, 0, s>>>(static_cast<const uint8_t*>(w), rows, row_bytes,
                                                                    kb, static_cast<uint4*>(out), pieces);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(const GemmArgs& g, cudaStream_t s) {
  if (g.E > kMaxExperts) return cudaErrorNotSupported;
  CUtensorMap ma, mb;
  if (!make_map(&ma, g.x, g.a_max, g.K, g.fp8) ||
      !make_weight_map(&mb, g.w, (int64_t)g.E * g.N, g.K, g.fp8, g.packed))
    return cudaErrorInvalidValue;
  Phase p = make_phase(g.N, g.K, g.epilogue, g.fp8, g.y, g.x_scale, g.w_scale);
  p.packed = g.packed ? 1 : 0;
  p.scatter = g.scatter;
  p.T_out = g.T_out;
  p.accumulate = g.accumulate;
  // rows stored in place (no combine): full 32-row chunks go out as TMA stores when y admits a map
  CUtensorMap my = mb;
  if (!g.scatter) p.tma_store = make_map_sw128(&my, g.y, g.a_max, p.n_out, false, 32) ? 1 : 0;
  if (g.pairs) {
    p.band = band_rows_tiles(kPairBM, g.K, g.fp8);
    if (g.fp8) return launch_pair<true>(ma, mb, my, g.counts, p, g.E, g.a_max, g.err, s);
    return launch_pair<false>(ma, mb, my, g.counts, p, g.E, g.a_max, g.err, s);
  }
  if (g.fp8) return launch_phases<true, 1>(ma, mb, ma, mb, my, g.counts, p, p, g.E, g.a_max, nullptr, g.err, s);
  return launch_phases<false, 1>(ma, mb, ma, mb, my, g.counts, p, p, g.E, g.a_max, nullptr, g.err, s);
}

// Per-expert z-row counters and an exit counter; zero between launches.
size_t expert_mlp_workspace_bytes(int E) { return ((size_t)(E + 1) * sizeof(int) + 255) / 256 * 256; }

cudaError_t launch_expert_mlp(const MlpArgs& g, cudaStream_t s) {
  if (g.E > kMaxExperts) return cudaErrorNotSupported;
  CUtensorMap a0, b0, a1, b1;
  if (!make_map(&a0, g.x, g.a_max, g.D, false) ||
      !make_weight_map(&b0, g.w13, (int64_t)g.E * 2 * g.H, g.D, false, g.packed) ||
      !make_map(&a1, g.z, g.a_max, g.H, false) ||
      !make_weight_map(&b1, g.w2, (int64_t)g.E * g.D, g.H, false, g.packed))
    return cudaErrorInvalidValue;
  Phase p0 = make_phase(2 * g.H, g.D, MOE_EPILOGUE_SILU_MUL, false, g.z, nullptr, nullptr);
  Phase p1 = make_phase(g.D, g.H, MOE_EPILOGUE_NONE, false, g.y, nullptr, nullptr);
  p0.packed = p1.packed = g.packed ? 1 : 0;
  p1.scatter = g.scatter;
  p1.T_out = g.T_out;
  p1.accumulate = g.accumulate;
  int* done = static_cast<int*>(g.ws);  // zero on entry, left zero by the kernel
  return launch_phases<false, 2>(a0, b0, a1, b1, b1, g.counts, p0, p1, g.E, g.a_max, done, g.err, s);
}

}  // namespace moe
