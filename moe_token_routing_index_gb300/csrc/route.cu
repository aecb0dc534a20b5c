// Top-k routing and the stable by-expert permutation (index_shuffling of
// mslk/moe/layers.py, MetaShufflingMoE._route; selection as torch.topk in
// BaselineMoE._forward, ties to the lower expert index).
//
// Small problems (the decode batch) run in one block, all in shared memory.
// Larger ones run as one cooperative launch in three phases over 32-token
// chunks, separated by grid-wide barriers:
//   select : one warp per token; each lane holds the order keys of experts
//            lane, lane+32, ...; top_k rounds of a warp arg-max (redux.sync max
//            on the key, then min on the expert index among the winners).
//            Writes the chosen experts and a per-chunk expert histogram.
//   scan   : one block per expert; exclusive scan of that expert's histogram
//            over the chunks (the chunk's base row within the expert) and the
//            expert's count.
//   emit   : per chunk, a 32-bit bitmap per expert marks which of the chunk's
//            tokens chose it, so a token's rank within the expert is a
//            popcount; row = expert offset + chunk base + rank.
// The barrier is an arrival counter in the workspace (zeroed before the
// launch) with a bounded wait; the cooperative launch keeps every block resident.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int kTokBlock = 32;     // tokens per block (one bitmap word per expert)
constexpr int kRouteThreads = 1024;  // 32 warps: one token of a 32-token chunk per warp
constexpr int kWarps = kRouteThreads / 32;

// Phase 1 for chunk c: select the top_k experts of its valid tokens.
template <int EPL>
__device__ void route_select_chunk(int c, const void* __restrict__ scores, int dtype, int64_t st, int64_t se, int E,
                                   int k, int Tv, int32_t* __restrict__ chosen, int32_t* __restrict__ hist_t, int nblk,
                                   int* s_hist) {
  for (int e = threadIdx.x; e < E; e += kRouteThreads) s_hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = c * kTokBlock;
  for (int t = t0 + warp; t < t0 + kTokBlock && t < Tv; t += kWarps) {
    uint32_t key[EPL];
    uint32_t live = 0;  // bit i: expert lane + 32 i exists and is not yet chosen
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      key[i] = 0u;
      if (e < E) {
        key[i] = route_order_key(load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se));
        live |= 1u << i;
      }
    }
    for (int j = 0; j < k; ++j) {
      uint32_t best = 0u;
      int best_i = -1;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (((live >> i) & 1u) && (best_i < 0 || key[i] > best)) {
          best = key[i];
          best_i = i;
        }
      const uint32_t wbest = __reduce_max_sync(0xffffffffu, best_i >= 0 ? best : 0u);
      const uint32_t cand = (best_i >= 0 && best == wbest) ? (uint32_t)(lane + 32 * best_i) : 0xffffffffu;
      const int we = (int)__reduce_min_sync(0xffffffffu, cand);
      if ((we & 31) == lane) live &= ~(1u << (we >> 5));
      if (lane == 0) {
        chosen[(int64_t)t * k + j] = we;
        atomicAdd(&s_hist[we], 1);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kRouteThreads) hist_t[(int64_t)e * nblk + c] = s_hist[e];
  __syncthreads();
}

// Block-wide exclusive scan of one value per thread; returns the thread's
// exclusive prefix, and the total in *total.  Two levels of warp shuffles: each
// warp scans its 32 values, warp 0 scans the 32 warp totals (s_part[0..32]).
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_part, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_part[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int x = lane < kWarps ? s_part[lane] : 0;
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += t;
    }
    s_part[lane] = xi - x;           // the warps' exclusive bases
    if (lane == 31) s_part[32] = xi;  // the block total
  }
  __syncthreads();
  const int excl = incl - v + s_part[w];
  *total = s_part[32];
  __syncthreads();  // s_part may be reused once every thread has read it
  return excl;
}

// Phase 2 for expert e: exclusive scan of hist_t[e, 0..nchunks) in place (rows of
// hist_t are nblk long); counts[e] = total.
__device__ void route_scan_expert(int e, int32_t* __restrict__ hist_t, int nblk, int nchunks,
                                  int32_t* __restrict__ counts, int* s_part) {
  int32_t* h = hist_t + (int64_t)e * nblk;
  const int per = (nchunks + kRouteThreads - 1) / kRouteThreads;
  const int b0 = threadIdx.x * per;
  int sum = 0;
  // data written by other blocks before a grid barrier is read at L2 (.cg), past any stale L1 line
  for (int b = b0; b < b0 + per && b < nchunks; ++b) sum += __ldcg(h + b);
  int total;
  int run = block_exclusive_scan(sum, s_part, &total);
  for (int b = b0; b < b0 + per && b < nchunks; ++b) {
    const int v = __ldcg(h + b);
    h[b] = run;
    run += v;
  }
  if (threadIdx.x == 0) counts[e] = total;
}

// Phase 3 for chunk c: rows of its tokens.  s_off holds the expert offsets.
__device__ void route_emit_chunk(int c, int E, int k, int Tv, const int32_t* __restrict__ chosen,
                                 const int32_t* __restrict__ hist_t, int nblk, const int* s_off, unsigned int* s_bits,
                                 int32_t* __restrict__ expert_indices, int32_t* __restrict__ token_indices,
                                 int32_t* __restrict__ inv, float* __restrict__ wts, const void* __restrict__ scores,
                                 int dtype, int64_t st, int64_t se) {
  const int tid = threadIdx.x;
  const int t0 = c * kTokBlock;
  const int nt = min(kTokBlock, Tv - t0);
  for (int e = tid; e < E; e += kRouteThreads) s_bits[e] = 0u;
  __syncthreads();
  for (int p = tid; p < nt * k; p += kRouteThreads) {  // mark which tokens of the chunk chose each expert
    const int tl = p / k;
    const int e = __ldcg(chosen + (int64_t)(t0 + tl) * k + (p % k));
    atomicOr(&s_bits[e], 1u << tl);
  }
  __syncthreads();
  for (int p = tid; p < nt * k; p += kRouteThreads) {
    const int tl = p / k, j = p % k, t = t0 + tl;
    const int32_t* ch = chosen + (int64_t)t * k;
    const int e = __ldcg(ch + j);
    const int rank = __popc(s_bits[e] & ((1u << tl) - 1u));
    const int row = s_off[e] + __ldcg(hist_t + (int64_t)e * nblk + c) + rank;
    expert_indices[row] = e;
    token_indices[row] = t;
    if (inv || wts) {
      int pos = 0;  // rows of t ascend with the expert index
      for (int jj = 0; jj < k; ++jj) pos += __ldcg(ch + jj) < e;
      if (inv) inv[(int64_t)t * k + pos] = row;
      if (wts) wts[(int64_t)t * k + pos] = load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se);
    }
  }
  __syncthreads();
}

// SELECT: all three phases from the scores.  Otherwise the selection was done by
// the router GEMM's epilogue (moe_router_route), which left the chosen experts
// and the chunk histograms in the workspace and zeroed the barrier counter: the
// launch starts at the scan, with one grid barrier.
template <int EPL, bool SELECT>
__global__ void __launch_bounds__(kRouteThreads) route_coop_kernel(
    const void* __restrict__ scores, int dtype, int64_t st, int64_t se, int T, int E, int k,
    const int32_t* __restrict__ num_valid, int32_t* __restrict__ chosen, int32_t* __restrict__ hist_t, int nblk,
    unsigned int* barrier, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ expert_indices, int32_t* __restrict__ token_indices, int32_t* __restrict__ inv,
    float* __restrict__ wts, unsigned int* err) {
  __shared__ int s_a[1024];          // select: histogram; emit: expert offsets
  __shared__ unsigned int s_bits[1024];
  __shared__ int s_part[kRouteThreads];
  pdl_launch_dependents();  // the gather may launch and wait for this grid
  const int Tv = read_count(num_valid, T, err);
  const int nchunks = (Tv + kTokBlock - 1) / kTokBlock;
  unsigned int arrivals = 0;
  if constexpr (SELECT) {
    for (int c = blockIdx.x; c < nchunks; c += gridDim.x)
      route_select_chunk<EPL>(c, scores, dtype, st, se, E, k, Tv, chosen, hist_t, nblk, s_a);
    arrivals += gridDim.x;
    if (!grid_barrier(barrier, arrivals)) {
      if (threadIdx.x == 0) flag_error(err, MOE_DEVERR_TIMEOUT);
      return;
    }
  }
  for (int e = blockIdx.x; e < E; e += gridDim.x) route_scan_expert(e, hist_t, nblk, nchunks, counts, s_part);
  arrivals += gridDim.x;
  if (!grid_barrier(barrier, arrivals)) {
    if (threadIdx.x == 0) flag_error(err, MOE_DEVERR_TIMEOUT);
    return;
  }
  // expert offsets (every block recomputes them from the counts)
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  int sum = 0;
  for (int e = threadIdx.x * per; e < (threadIdx.x + 1) * per && e < E; ++e) sum += __ldcg(counts + e);
  int total;
  int run = block_exclusive_scan(sum, s_part, &total);
  for (int e = threadIdx.x * per; e < (threadIdx.x + 1) * per && e < E; ++e) {
    s_a[e] = run;
    run += __ldcg(counts + e);
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += kRouteThreads) offsets[e] = s_a[e];
    if (threadIdx.x == 0) {
      counts[E] = total;
      offsets[E] = total;
      if (total != Tv * k) flag_error(err, MOE_DEVERR_BAD_COUNT);
    }
  }
  for (int c = blockIdx.x; c < nchunks; c += gridDim.x)
    route_emit_chunk(c, E, k, Tv, chosen, hist_t, nblk, s_a, s_bits, expert_indices, token_indices, inv, wts, scores,
                     dtype, st, se);
}

// ---------------------------------------------------------------------------
// Whole routing in one block, for small problems (T <= 1024, T*E <= 16384,
// E <= 256, T*top_k <= 8192).  The scores are staged in shared memory as order
// keys; warp w selects for the contiguous token chunk [w*C, (w+1)*C) and keeps
// a private expert histogram; one scan over (warp, expert) gives each warp's
// base row inside every expert; the warps then walk their chunks in token
// order and hand out rows, which keeps the within-expert order by token.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallMaxT = 1024, kSmallMaxTE = 16384, kSmallMaxE = 256, kSmallMaxTK = 8192;

size_t small_smem_bytes(int T, int E, int k) {
  return (size_t)T * E * 4 + (size_t)kSmallWarps * E * 4 + (size_t)(E + 1) * 4 + ((size_t)T * k * 2 + 15) / 16 * 16;
}

template <int EPL>
__global__ void __launch_bounds__(kSmallThreads) route_small_kernel(
    const void* __restrict__ scores, int dtype, int64_t st, int64_t se, int T, int E, int k,
    const int32_t* __restrict__ num_valid, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ expert_indices, int32_t* __restrict__ token_indices, int32_t* __restrict__ inv,
    float* __restrict__ wts, unsigned int* err) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* s_key = reinterpret_cast<uint32_t*>(smem);                 // [T][E]
  int* s_hist = reinterpret_cast<int*>(s_key + (size_t)T * E);        // [warps][E]: counts, then bases
  int* s_off = s_hist + kSmallWarps * E;                               // [E + 1]
  uint16_t* s_chosen = reinterpret_cast<uint16_t*>(s_off + E + 1);     // [T][k]
  pdl_launch_dependents();  // the gather may launch and wait for this grid
  const int Tv = read_count(num_valid, T, err);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < Tv * E; i += kSmallThreads) {
    const int t = i / E, e = i - t * E;
    s_key[i] = route_order_key(load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se));
  }
  for (int i = tid; i < kSmallWarps * E; i += kSmallThreads) s_hist[i] = 0;
  __syncthreads();

  const int C = (Tv + kSmallWarps - 1) / kSmallWarps;
  const int t_begin = warp * C, t_end = min(Tv, t_begin + C);
  int* my_hist = s_hist + warp * E;
  for (int t = t_begin; t < t_end; ++t) {
    uint32_t key[EPL];
    uint32_t live = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      key[i] = 0u;
      if (e < E) {
        key[i] = s_key[t * E + e];
        live |= 1u << i;
      }
    }
    for (int j = 0; j < k; ++j) {
      uint32_t best = 0u;
      int best_i = -1;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (((live >> i) & 1u) && (best_i < 0 || key[i] > best)) {
          best = key[i];
          best_i = i;
        }
      const uint32_t wbest = __reduce_max_sync(0xffffffffu, best_i >= 0 ? best : 0u);
      const uint32_t cand = (best_i >= 0 && best == wbest) ? (uint32_t)(lane + 32 * best_i) : 0xffffffffu;
      const int we = (int)__reduce_min_sync(0xffffffffu, cand);
      if ((we & 31) == lane) live &= ~(1u << (we >> 5));
      if (lane == 0) {
        s_chosen[t * k + j] = (uint16_t)we;
        my_hist[we] += 1;
      }
    }
  }
  __syncthreads();
  // per expert: exclusive scan over the warps (each warp's base inside the expert)
  for (int e = tid; e < E; e += kSmallThreads) {
    int run = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int v = s_hist[w * E + e];
      s_hist[w * E + e] = run;
      run += v;
    }
    s_off[e] = run;  // the expert's count, for now
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the counts over the experts
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? s_off[e] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) {
        counts[e] = c;
        offsets[e] = carry + incl - c;
        s_off[e] = carry + incl - c;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      counts[E] = carry;
      offsets[E] = carry;
      s_off[E] = carry;
    }
  }
  __syncthreads();
  for (int t = t_begin; t < t_end; ++t) {
    for (int j = lane; j < k; j += 32) {  // a token's experts are distinct: no two lanes share a counter
      const int e = s_chosen[t * k + j];
      const int row = s_off[e] + my_hist[e];
      my_hist[e] += 1;
      expert_indices[row] = e;
      token_indices[row] = t;
      if (inv || wts) {
        int pos = 0;
        for (int jj = 0; jj < k; ++jj) pos += s_chosen[t * k + jj] < e;
        if (inv) inv[(int64_t)t * k + pos] = row;
        if (wts) wts[(int64_t)t * k + pos] = load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se);
      }
    }
    __syncwarp();
  }
}

template <int EPL>
cudaError_t launch_small(const RouteArgs& a, cudaStream_t s) {
  const size_t smem = small_smem_bytes(a.T, a.E, a.top_k);
  auto kern = route_small_kernel<EPL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<1, kSmallThreads, smem, s>>>(a.scores, a.dtype, a.stride_t, a.stride_e, a.T, a.E, a.top_k, a.num_valid,
                                      a.counts, a.offsets, a.expert_indices, a.token_indices, a.inv, a.weights,
                                      a.err);
  return cudaGetLastError();
}

// SELECT: zero the barrier counter first (the fused path's router did it already).
template <int EPL, bool SELECT>
cudaError_t launch_coop(const RouteArgs& a, int32_t* chosen, int32_t* hist_t, int nblk, unsigned int* barrier,
                        cudaStream_t s) {
  auto kern = route_coop_kernel<EPL, SELECT>;
  const int cap = device_sm_count() * resident_blocks_per_sm(reinterpret_cast<const void*>(kern), kRouteThreads);
  const int want = nblk > a.E ? nblk : a.E;   // chunks to select and emit, experts to scan
  const int grid = want < cap ? want : cap;
  cudaError_t e = SELECT ? cudaMemsetAsync(barrier, 0, sizeof(unsigned int), s) : cudaSuccess;
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barriers need every block resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a.scores, a.dtype, a.stride_t, a.stride_e, a.T, a.E, a.top_k, a.num_valid,
                         chosen, hist_t, nblk, barrier, a.counts, a.offsets, a.expert_indices, a.token_indices,
                         a.inv, a.weights, a.err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t preload_route_kernels() {
  const void* kernels[] = {
      reinterpret_cast<const void*>(route_small_kernel<1>), reinterpret_cast<const void*>(route_small_kernel<2>),
      reinterpret_cast<const void*>(route_small_kernel<4>), reinterpret_cast<const void*>(route_small_kernel<8>),
      reinterpret_cast<const void*>(route_coop_kernel<1, true>),
      reinterpret_cast<const void*>(route_coop_kernel<2, true>),
      reinterpret_cast<const void*>(route_coop_kernel<4, true>),
      reinterpret_cast<const void*>(route_coop_kernel<8, true>),
      reinterpret_cast<const void*>(route_coop_kernel<16, true>),
      reinterpret_cast<const void*>(route_coop_kernel<32, true>),
      reinterpret_cast<const void*>(route_coop_kernel<1, false>)};
  for (const void* k : kernels) {
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, k);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Workspace: [barrier counter | pad to 256] [chosen experts T*k] [histogram E x chunks]
size_t route_workspace_bytes(int T, int E, int top_k) {
  const size_t nblk = (size_t)(T + kTokBlock - 1) / kTokBlock;
  const size_t chosen = ((size_t)T * top_k * 4 + 255) / 256 * 256;
  return 256 + chosen + nblk * (size_t)E * 4 + 256;
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  const int nblk = (a.T + kTokBlock - 1) / kTokBlock;
  if (nblk == 0) {
    // No token rows at all: the counts and offsets are all zero.
    cudaError_t e = cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * (a.E + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.offsets, 0, sizeof(int32_t) * (a.E + 1), s);
    return e;
  }
  if (a.T <= kSmallMaxT && a.E <= kSmallMaxE && a.T * a.E <= kSmallMaxTE && a.T * a.top_k <= kSmallMaxTK) {
    const int epl = (a.E + 31) / 32;
    if (epl <= 1) return launch_small<1>(a, s);
    if (epl <= 2) return launch_small<2>(a, s);
    if (epl <= 4) return launch_small<4>(a, s);
    return launch_small<8>(a, s);
  }
  RouteWorkspace w = route_workspace(a.ws, a.T, a.top_k);
  const int epl = (a.E + 31) / 32;
  if (epl <= 1) return launch_coop<1, true>(a, w.chosen, w.hist_t, nblk, w.barrier, s);
  if (epl <= 2) return launch_coop<2, true>(a, w.chosen, w.hist_t, nblk, w.barrier, s);
  if (epl <= 4) return launch_coop<4, true>(a, w.chosen, w.hist_t, nblk, w.barrier, s);
  if (epl <= 8) return launch_coop<8, true>(a, w.chosen, w.hist_t, nblk, w.barrier, s);
  if (epl <= 16) return launch_coop<16, true>(a, w.chosen, w.hist_t, nblk, w.barrier, s);
  return launch_coop<32, true>(a, w.chosen, w.hist_t, nblk, w.barrier, s);
}

cudaError_t launch_route_emit(const RouteArgs& a, cudaStream_t s) {
  const int nblk = (a.T + kTokBlock - 1) / kTokBlock;
  RouteWorkspace w = route_workspace(a.ws, a.T, a.top_k);
  return launch_coop<1, false>(a, w.chosen, w.hist_t, nblk, w.barrier, s);
}

RouteWorkspace route_workspace(void* ws, int T, int top_k) {
  char* b = static_cast<char*>(ws);
  RouteWorkspace w;
  w.barrier = reinterpret_cast<unsigned int*>(b);
  w.chosen = reinterpret_cast<int32_t*>(b + 256);
  w.hist_t = reinterpret_cast<int32_t*>(b + 256 + ((size_t)T * top_k * 4 + 255) / 256 * 256);
  return w;
}

}  // namespace moe
