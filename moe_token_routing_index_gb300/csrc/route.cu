// Top-k routing and the stable by-expert permutation (index_shuffling of
// mslk/moe/layers.py, MetaShufflingMoE._route; selection as torch.topk in
// BaselineMoE._forward, ties to the lower expert index).
//
// Small problems (the decode batch) run in one block, all in shared memory;
// larger ones take three launches over blocks of 32 tokens:
//   select : one warp per token; each lane holds the order keys of experts
//            lane, lane+32, ...; top_k rounds of a warp arg-max (redux.sync max
//            on the key, then min on the expert index among the winners).
//            Writes the chosen experts and a per-block expert histogram.
//   scan   : one block per expert; exclusive scan of that expert's histogram
//            over the token blocks (the block's base row within the expert)
//            and the expert's count.
//   emit   : per token block, a 32-bit bitmap per expert marks which of the
//            block's tokens chose it, so a token's rank within the expert is a
//            popcount; row = expert offset + block base + rank.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int kTokBlock = 32;     // tokens per block (one bitmap word per expert)
constexpr int kRouteThreads = 256;
constexpr int kWarps = kRouteThreads / 32;

// Monotone map of a float to uint32 (larger float -> larger key), -0 folded onto +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int EPL>  // experts per lane: ceil(E / 32) rounded up to the instantiated size
__global__ void __launch_bounds__(kRouteThreads) route_select_kernel(
    const void* __restrict__ scores, int dtype, int64_t st, int64_t se, int T, int E, int k,
    const int32_t* __restrict__ num_valid, int32_t* __restrict__ chosen, int32_t* __restrict__ hist_t,
    int nblk, unsigned int* err) {
  __shared__ int s_hist[1024];
  const int Tv = read_count(num_valid, T, err);
  for (int e = threadIdx.x; e < E; e += kRouteThreads) s_hist[e] = 0;
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTokBlock;
  for (int t = t0 + warp; t < t0 + kTokBlock && t < Tv; t += kWarps) {
    uint32_t key[EPL];
    uint32_t live = 0;  // bit i: expert lane + 32 i exists and is not yet chosen
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      key[i] = 0u;
      if (e < E) {
        key[i] = order_key(load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se));
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
  for (int e = threadIdx.x; e < E; e += kRouteThreads) hist_t[(int64_t)e * nblk + blockIdx.x] = s_hist[e];
}

// Block e: exclusive scan of hist_t[e, 0..nblk) in place; counts[e] = total.
__global__ void __launch_bounds__(kRouteThreads) route_scan_kernel(int32_t* __restrict__ hist_t, int nblk,
                                                                   int32_t* __restrict__ counts) {
  __shared__ int s_part[kRouteThreads];
  const int e = blockIdx.x;
  int32_t* h = hist_t + (int64_t)e * nblk;
  const int per = (nblk + kRouteThreads - 1) / kRouteThreads;
  const int b0 = threadIdx.x * per;
  int sum = 0;
  for (int b = b0; b < b0 + per && b < nblk; ++b) sum += h[b];
  s_part[threadIdx.x] = sum;
  __syncthreads();
  // Hillis-Steele inclusive scan of the per-thread sums.
  for (int o = 1; o < kRouteThreads; o <<= 1) {
    int v = threadIdx.x >= o ? s_part[threadIdx.x - o] : 0;
    __syncthreads();
    s_part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = s_part[threadIdx.x] - sum;
  for (int b = b0; b < b0 + per && b < nblk; ++b) {
    const int v = h[b];
    h[b] = run;
    run += v;
  }
  if (threadIdx.x == kRouteThreads - 1) counts[e] = s_part[kRouteThreads - 1];
}

__global__ void __launch_bounds__(kRouteThreads) route_emit_kernel(
    int T, int E, int k, const int32_t* __restrict__ num_valid, const int32_t* __restrict__ chosen,
    const int32_t* __restrict__ hist_t, int nblk, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ expert_indices, int32_t* __restrict__ token_indices, int32_t* __restrict__ inv,
    unsigned int* err) {
  __shared__ int s_off[1024];
  __shared__ unsigned int s_bits[1024];
  __shared__ int s_scan[kRouteThreads];
  const int Tv = read_count(num_valid, T, nullptr);  // already flagged by select
  const int tid = threadIdx.x;

  // Exclusive scan of counts[0..E) -> expert offsets (each block recomputes it).
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  int sum = 0;
  for (int e = tid * per; e < (tid + 1) * per && e < E; ++e) sum += counts[e];
  s_scan[tid] = sum;
  for (int e = tid; e < E; e += kRouteThreads) s_bits[e] = 0u;
  __syncthreads();
  for (int o = 1; o < kRouteThreads; o <<= 1) {
    int v = tid >= o ? s_scan[tid - o] : 0;
    __syncthreads();
    s_scan[tid] += v;
    __syncthreads();
  }
  int run = s_scan[tid] - sum;
  for (int e = tid * per; e < (tid + 1) * per && e < E; ++e) {
    s_off[e] = run;
    run += counts[e];
  }
  const int total = s_scan[kRouteThreads - 1];
  if (blockIdx.x == 0) {
    for (int e = tid; e < E; e += kRouteThreads) offsets[e] = s_off[e];
    if (tid == 0) {
      counts[E] = total;
      offsets[E] = total;
      if (total != Tv * k) flag_error(err, MOE_DEVERR_BAD_COUNT);
    }
  }

  const int t0 = blockIdx.x * kTokBlock;
  const int nt = min(kTokBlock, Tv - t0);
  if (nt <= 0) return;
  // Mark which tokens of the block chose each expert.
  for (int p = tid; p < nt * k; p += kRouteThreads) {
    const int tl = p / k;
    const int e = chosen[(int64_t)(t0 + tl) * k + (p % k)];
    atomicOr(&s_bits[e], 1u << tl);
  }
  __syncthreads();
  for (int p = tid; p < nt * k; p += kRouteThreads) {
    const int tl = p / k, j = p % k, t = t0 + tl;
    const int32_t* ch = chosen + (int64_t)t * k;
    const int e = ch[j];
    const int rank = __popc(s_bits[e] & ((1u << tl) - 1u));
    const int row = s_off[e] + hist_t[(int64_t)e * nblk + blockIdx.x] + rank;
    expert_indices[row] = e;
    token_indices[row] = t;
    if (inv) {
      int pos = 0;  // rows of t ascend with the expert index
      for (int jj = 0; jj < k; ++jj) pos += ch[jj] < e;
      inv[(int64_t)t * k + pos] = row;
    }
  }
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
    unsigned int* err) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* s_key = reinterpret_cast<uint32_t*>(smem);                 // [T][E]
  int* s_hist = reinterpret_cast<int*>(s_key + (size_t)T * E);        // [warps][E]: counts, then bases
  int* s_off = s_hist + kSmallWarps * E;                               // [E + 1]
  uint16_t* s_chosen = reinterpret_cast<uint16_t*>(s_off + E + 1);     // [T][k]
  const int Tv = read_count(num_valid, T, err);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < Tv * E; i += kSmallThreads) {
    const int t = i / E, e = i - t * E;
    s_key[i] = order_key(load_score(scores, dtype, (int64_t)t * st + (int64_t)e * se));
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
      if (inv) {
        int pos = 0;
        for (int jj = 0; jj < k; ++jj) pos += s_chosen[t * k + jj] < e;
        inv[(int64_t)t * k + pos] = row;
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
                                      a.counts, a.offsets, a.expert_indices, a.token_indices, a.inv, a.err);
  return cudaGetLastError();
}

template <int EPL>
void launch_select(const RouteArgs& a, int32_t* chosen, int32_t* hist_t, int nblk, cudaStream_t s) {
  route_select_kernel<EPL><<<nblk, kRouteThreads, 0, s>>>(a.scores, a.dtype, a.stride_t, a.stride_e, a.T, a.E,
                                                          a.top_k, a.num_valid, chosen, hist_t, nblk, a.err);
}

}  // namespace

size_t route_workspace_bytes(int T, int E, int top_k) {
  const size_t nblk = (size_t)(T + kTokBlock - 1) / kTokBlock;
  const size_t chosen = ((size_t)T * top_k * 4 + 255) / 256 * 256;
  return chosen + nblk * (size_t)E * 4 + 256;
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
  char* ws = static_cast<char*>(a.ws);
  int32_t* chosen = reinterpret_cast<int32_t*>(ws);
  int32_t* hist_t = reinterpret_cast<int32_t*>(ws + ((size_t)a.T * a.top_k * 4 + 255) / 256 * 256);
  const int epl = (a.E + 31) / 32;
  if (epl <= 1) launch_select<1>(a, chosen, hist_t, nblk, s);
  else if (epl <= 2) launch_select<2>(a, chosen, hist_t, nblk, s);
  else if (epl <= 4) launch_select<4>(a, chosen, hist_t, nblk, s);
  else if (epl <= 8) launch_select<8>(a, chosen, hist_t, nblk, s);
  else if (epl <= 16) launch_select<16>(a, chosen, hist_t, nblk, s);
  else launch_select<32>(a, chosen, hist_t, nblk, s);
  route_scan_kernel<<<a.E, kRouteThreads, 0, s>>>(hist_t, nblk, a.counts);
  route_emit_kernel<<<nblk, kRouteThreads, 0, s>>>(a.T, a.E, a.top_k, a.num_valid, chosen, hist_t, nblk,
                                                   a.counts, a.offsets, a.expert_indices, a.token_indices,
                                                   a.inv, a.err);
  return cudaGetLastError();
}

}  // namespace moe
