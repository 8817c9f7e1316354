// MoE routing prep: counting sort of the T*topk (token, slot) routes by
// expert, stable by token ("The FP4 Frontier", Finding 5: one grouped GEMM
// over all experts needs each expert's token rows contiguous).
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

constexpr int ROUTE_THREADS = 1024;
constexpr int ROUTE_WARPS = ROUTE_THREADS / 32;

// One CTA.  Pass 1 histograms the experts; pass 2 walks the routes in
// chunks of 1024 consecutive flat indices and gives each route its position
// base[e] + (same-expert routes of earlier warps in the chunk) + (same-expert
// lanes before it in its warp), which keeps flat (= token-major) order.  Per
// chunk, each warp's leader lane of an expert records the warp's count, one
// thread per expert turns its column of counts into the warps' first
// positions (advancing base[e]), and each route adds its rank in the warp.
__global__ void __launch_bounds__(ROUTE_THREADS) route_kernel(
    const int32_t* __restrict__ ids, int64_t R, int topk, int E,
    int32_t* __restrict__ offsets, int32_t* __restrict__ route_token,
    int32_t* __restrict__ route_slot, int32_t* __restrict__ route_pos, int* status) {
  extern __shared__ int32_t sh[];
  int32_t* base = sh;                       // [E]
  int32_t* wcnt = sh + E;                   // [ROUTE_WARPS][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int e_nxt = -1;                                 // the first chunk's expert (pass 2)
  if (tid < R) { e_nxt = ids[tid]; if (e_nxt < 0 || e_nxt >= E) e_nxt = -1; }
  for (int i = tid; i < E * (ROUTE_WARPS + 1); i += ROUTE_THREADS) sh[i] = 0;
  __syncthreads();
  int bad = 0;
  for (int64_t i = tid; i < R; i += ROUTE_THREADS) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&base[e], 1); else bad = 1;
  }
  if (__syncthreads_or(bad) && tid == 0) raise_status(status, NVFP4_ERR_DEVICE_CHECK);
  // exclusive scan of the counts (E <= 1024: one element per thread)
  int32_t c = tid < E ? base[tid] : 0;
  int32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  __shared__ int32_t wsum[ROUTE_WARPS];
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t v = wsum[lane];
    int32_t s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += u;
    }
    wsum[lane] = s - v;                     // exclusive over warps
  }
  __syncthreads();
  const int32_t excl = incl - c + wsum[warp];
  if (tid < E) { offsets[tid] = excl; base[tid] = excl; }
  if (tid == E - 1) offsets[E] = excl + c;
  if (E == 0 && tid == 0) offsets[0] = 0;
  __syncthreads();

  for (int64_t c0 = 0; c0 < R; c0 += ROUTE_THREADS) {
    const int64_t i = c0 + tid;
    const int e = e_nxt;
    e_nxt = -1;                                     // the next chunk's expert, loaded early
    if (i + ROUTE_THREADS < R) {
      e_nxt = ids[i + ROUTE_THREADS];
      if (e_nxt < 0 || e_nxt >= E) e_nxt = -1;
    }
    const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(same);
    __syncthreads();
    // counts -> first positions, only where a warp has routes of the expert:
    // those entries are the ones their warps' leaders zero after use, so
    // every entry is zero again when the next chunk's counts arrive
    for (int ee = tid; ee < E; ee += ROUTE_THREADS) {
      int32_t run = base[ee];
      for (int w = 0; w < ROUTE_WARPS; ++w) {
        const int32_t v = wcnt[w * E + ee];
        if (v != 0) wcnt[w * E + ee] = run;
        run += v;
      }
      base[ee] = run;
    }
    __syncthreads();
    if (e >= 0) {
      const int32_t pos = wcnt[warp * E + e] + rank;
      route_token[pos] = static_cast<int32_t>(i / topk);
      route_slot[pos] = static_cast<int32_t>(i % topk);
      if (route_pos) route_pos[i] = pos;
    } else if (i < R && route_pos) {
      route_pos[i] = -1;
    }
    // the warp's entries back to zero for the next chunk (its lanes have read
    // them; the next chunk's first barrier orders this before the scan)
    __syncwarp();
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = 0;
    __syncwarp();                                   // before the next chunk's counts
  }
}

cudaError_t init_route_attributes() {
  return cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(int32_t) * 1024 * (ROUTE_WARPS + 1)));
}

cudaError_t launch_route(const int32_t* ids, int64_t T, int topk, int E, int32_t* offsets,
                         int32_t* route_token, int32_t* route_slot, int32_t* route_pos,
                         int* status, cudaStream_t s) {
  const size_t shmem = sizeof(int32_t) * static_cast<size_t>(E) * (ROUTE_WARPS + 1);
  route_kernel<<<1, ROUTE_THREADS, shmem, s>>>(ids, T * topk, topk, E, offsets, route_token,
                                               route_slot, route_pos, status);
  return cudaGetLastError();
}

}  // namespace nvfp4
