// BF16 -> NVFP4 quantiser kernels: tensor amax -> global scale, per-16-block
// E4M3 scale + E2M1 codes (row-major, atom layout, or dispatched to route
// order), and the offline prepack of row-major weight scales.
//
// Format: "The Blackwell architectural split", Preserving precision --
// dual-tier scale handling (E2M1 elements, a global tensor scale and one
// block scale per 16 values).  Recipe: g = amax / (6 * 448),
// s = (amax_b / 6) / g, each step binary32 round-to-nearest-even.
#include "common.cuh"
#include "kernels.h"
#include "format.cuh"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Tensor amax -> global scale
// ---------------------------------------------------------------------------
// Each block reduces |x| over its share of the tensor (BF16 magnitudes
// compare as integers).  Work item: a warp reads 128 consecutive 16-byte
// vectors of one row (four loads in flight per lane); one integer division
// per item maps it to its row.  With `g`, the block turns its maximum into
// g_b = amax_b / 2688 and folds it into *g with an integer atomicMax on the
// float bits (valid for g_b >= 0; *g starts at 0).  Division by a positive
// constant is monotone, so max_b(g_b) = max(amax)/2688.  With `partials`, it
// stores its maximum's magnitude bits in partials[block] and a later kernel
// reduces them.  Rows must be 16-byte aligned with cols % 8 == 0.
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ x,
                                                   int64_t rows, int64_t cols, int64_t ld,
                                                   float* g, uint32_t* partials) {
  uint32_t m = 0;
  const int lane = threadIdx.x & 31;
  const uint32_t vpr = static_cast<uint32_t>(cols >> 3);          // vectors per row
  const uint32_t segs = (vpr + 127u) / 128u;                       // items per row
  const uint64_t items = static_cast<uint64_t>(rows) * segs;
  const uint64_t wstride = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
  for (uint64_t it = static_cast<uint64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < items; it += wstride) {
    const uint64_t r = it / segs;
    const uint32_t v0 = static_cast<uint32_t>(it - r * segs) * 128u + lane;
    const uint4* row = reinterpret_cast<const uint4*>(x + r * ld);
    uint4 q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      q[k] = (v0 + 32u * k < vpr) ? __ldg(row + v0 + 32u * k) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // BF16 magnitudes compare as unsigned 16-bit integers, two per instruction
      m = __vmaxu2(m, __vmaxu2(__vmaxu2(q[k].x & 0x7FFF7FFFu, q[k].y & 0x7FFF7FFFu),
                                __vmaxu2(q[k].z & 0x7FFF7FFFu, q[k].w & 0x7FFF7FFFu)));
    }
  }
  m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ uint32_t wm[8];
  if (lane == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (blockDim.x >> 5); ++w) m = max(m, wm[w]);
    if (partials) {
      partials[blockIdx.x] = m;
    } else {
      const float gb = __fdiv_rn(bf16_bits_to_f32(m), 2688.0f);
      atomicMax(reinterpret_cast<unsigned int*>(g), __float_as_uint(gb));
    }
  }
}

// Lane 4j of a warp returns the bytes of lanes 4j..4j+3 as one little-endian
// word (for scale bytes that sit four to an aligned word).
__device__ __forceinline__ uint32_t gather4_bytes(uint32_t byte) {
  const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, byte, 1);
  const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, byte, 2);
  const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, byte, 3);
  return __byte_perm(__byte_perm(byte, b1, 0x0040u), __byte_perm(b2, b3, 0x0040u), 0x5410u);
}

// One 16-element block of BF16 (two 16-byte vectors) -> codes + scale.
__device__ __forceinline__ Block16 quantize_block(const uint4 lo, const uint4 hi, const ScaleK& k,
                                                  const float4* table) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  return quantize_bf16x16(w, k, table);
}

__device__ __forceinline__ int64_t atom_offset(int64_t r, int64_t c, int64_t n_cgroups) {
  return ((r >> 7) * n_cgroups + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// Work item: a warp quantises 64 consecutive 16-element blocks of one row,
// lane l taking the two consecutive blocks 2l and 2l + 1 (64 bytes of BF16:
// four 16-byte loads in flight per lane, whose lines the warp's loads fill
// between them).  A lane stores its 16 bytes of codes with one 16-byte store;
// in the atom layout the scale word of blocks 4j .. 4j + 3 is put together
// by the even lane of a pair from its own two scale bytes and its neighbour's
// (one shuffle), so the addressing and the stores are paid once per two
// blocks.  (Four blocks per lane needed 78 registers and ran slower at three
// blocks per SM.)  The item index is split into (row, segment) once and then
// stepped by the grid stride with a borrow, so no division sits in the loop.
constexpr uint32_t kQuantLaneBlocks = 2;
constexpr uint32_t kQuantItemBlocks = 32 * kQuantLaneBlocks;

__global__ void __launch_bounds__(256, 4) quantize_kernel(const uint16_t* __restrict__ x,
                                                       int64_t rows, int64_t cols, int64_t ld,
                                                       uint8_t* __restrict__ packed,
                                                       uint8_t* __restrict__ scales,
                                                       int sf_atoms, const float* g_ptr) {
  __shared__ float4 s_elem[kElemTable];
  const float g = *g_ptr;
  const ScaleK k = scale_consts(g);
  fill_elem_table(s_elem, g);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint32_t bpr = static_cast<uint32_t>(cols >> 4);
  const uint32_t segs = (bpr + kQuantItemBlocks - 1) / kQuantItemBlocks;
  const uint64_t items = static_cast<uint64_t>(rows) * segs;
  const uint64_t wstride = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t ncg = (cols + 63) >> 6;                 // 4-block scale groups per row
  const uint64_t j0 = static_cast<uint64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (j0 >= items) return;
  // one 16-byte code store per lane when every row starts on 16 bytes; one
  // 2-byte scale store (row-major scales) when every row's scales start on 2
  const size_t half_row = static_cast<size_t>(cols >> 1);
  const bool codes16 = (half_row % 16 == 0) && (reinterpret_cast<uintptr_t>(packed) % 16 == 0);
  const bool sf16 = (bpr % 2 == 0) && (reinterpret_cast<uintptr_t>(scales) % 2 == 0);
  // Items run from the end of the tensor backwards: the tensor amax pass
  // that precedes this kernel swept it front to back, so its tail is what
  // L2 still holds.  Item it = items - 1 - j is (row r, segment sg).
  const uint64_t it0 = items - 1 - j0;
  int64_t r = static_cast<int64_t>(it0 / segs);
  uint32_t sg = static_cast<uint32_t>(it0 - static_cast<uint64_t>(r) * segs);
  const int64_t dr = static_cast<int64_t>(wstride / segs);
  const uint32_t ds = static_cast<uint32_t>(wstride - static_cast<uint64_t>(dr) * segs);
  for (uint64_t j = j0; j < items; j += wstride) {
    const uint32_t b0 = sg * kQuantItemBlocks + kQuantLaneBlocks * lane;   // lane's first block
    uint32_t sfw = 0u;                             // the lane's scale bytes, block b0 lowest
    if (b0 < bpr) {
      const uint32_t nb = min(kQuantLaneBlocks, bpr - b0);                 // its valid blocks
      const uint4* src = reinterpret_cast<const uint4*>(x + r * ld) + 2 * b0;
      uint4 v[2 * kQuantLaneBlocks];
#pragma unroll
      for (int i = 0; i < 2 * static_cast<int>(kQuantLaneBlocks); ++i)
        v[i] = (static_cast<uint32_t>(i >> 1) < nb) ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
      uint32_t c[2 * kQuantLaneBlocks];
#pragma unroll
      for (int bb = 0; bb < static_cast<int>(kQuantLaneBlocks); ++bb) {
        const Block16 q = quantize_block(v[2 * bb], v[2 * bb + 1], k, s_elem);
        c[2 * bb] = q.packed.x;
        c[2 * bb + 1] = q.packed.y;
        sfw |= q.sf << (8 * bb);
      }
      uint8_t* dst = packed + r * half_row + static_cast<size_t>(b0) * 8;
      if (codes16 && nb == kQuantLaneBlocks) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(c[0], c[1], c[2], c[3]);
      } else {
#pragma unroll
        for (int bb = 0; bb < static_cast<int>(kQuantLaneBlocks); ++bb)
          if (static_cast<uint32_t>(bb) < nb)
            reinterpret_cast<uint2*>(dst)[bb] = make_uint2(c[2 * bb], c[2 * bb + 1]);
      }
      if (!sf_atoms) {
        uint8_t* sdst = scales + r * bpr + b0;
        if (sf16 && nb == kQuantLaneBlocks) {
          *reinterpret_cast<uint16_t*>(sdst) = static_cast<uint16_t>(sfw);
        } else {
#pragma unroll
          for (int bb = 0; bb < static_cast<int>(kQuantLaneBlocks); ++bb)
            if (static_cast<uint32_t>(bb) < nb) sdst[bb] = static_cast<uint8_t>(sfw >> (8 * bb));
        }
      }
    }
    if (sf_atoms) {
      // cols % 64 == 0: an even lane's pair of lanes covers one whole
      // 4-block scale word (both lanes valid or neither)
      const uint32_t other = __shfl_down_sync(0xFFFFFFFFu, sfw, 1);
      if ((lane & 1) == 0 && b0 < bpr)
        *reinterpret_cast<uint32_t*>(scales + atom_offset(r, b0, ncg)) = sfw | (other << 16);
    }
    // the next item: it - wstride = (r - dr) * segs + (sg - ds), with a borrow
    if (sg >= ds) {
      sg -= ds;
    } else {
      sg += segs - ds;
      r -= 1;
    }
    r -= dr;
  }
}

// Per-expert prefix tables held in shared memory by the dispatch kernel.
// tb[e] = first 128-row scale tile of expert e.
__device__ __forceinline__ int find_expert(const int32_t* off, int E, int32_t p) {
  int lo = 0, hi = E;                        // off[lo] <= p < off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= p) lo = mid; else hi = mid;
  }
  return lo;
}

// Operand tiles: 128 rows x 256 K-elements per tile, 16384 bytes of codes
// (row r at r * 128, 16-byte chunk j at position j ^ (r % 8): the 128-byte
// swizzle the tensor cores read) followed by 2048 bytes of scale atoms; tiles
// ordered row-tile major, then K block.
constexpr int64_t kTileBytes = 16384 + 2048;

__device__ __forceinline__ int64_t tile_code_offset(int64_t rt, int r, int64_t kb, int c,
                                                    int64_t n_kb) {
  return (rt * n_kb + kb) * kTileBytes + r * 128 + ((((c >> 4) ^ (r & 7))) << 4) + (c & 15);
}

__device__ __forceinline__ int64_t tile_scale_offset(int64_t rt, int r, int64_t kb, int s,
                                                     int64_t n_kb) {
  return (rt * n_kb + kb) * kTileBytes + 16384 + (s >> 2) * 512 + (r & 31) * 16 +
         ((r >> 5) & 3) * 4 + (s & 3);
}

// Quantise source rows and write each one to its route positions, in the
// grouped operand-tile layout: each expert's routes are cut into chunks of
// `chunk` rows and every chunk starts a fresh row tile (route p, local index
// j = p - off[e], is row j % chunk of tile tb[e] + j / chunk).
__global__ void __launch_bounds__(256) quantize_dispatch_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t K, int64_t ld,
    const int32_t* __restrict__ route_pos, int fanout,
    const int32_t* __restrict__ expert_offsets, int E, int64_t R, int chunk,
    uint8_t* __restrict__ tiles, float* g_ptr, const uint32_t* __restrict__ partials,
    int n_partials, int* status) {
  extern __shared__ int32_t sh[];
  int32_t* off = sh;              // [E + 1]
  int32_t* tb = sh + (E + 1);     // [E]
  __shared__ int32_t s_bad;
  __shared__ uint32_t s_wmax[8];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) off[e] = expert_offsets[e];
  // tensor amax: every block reduces the amax kernel's per-block maxima
  // itself (a few KB from L2), so no reset or atomic sits between the calls
  if (partials) {
    uint32_t m = 0;
    for (int i = threadIdx.x; i < n_partials; i += blockDim.x) m = max(m, partials[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) s_wmax[threadIdx.x >> 5] = m;
  }
  __syncthreads();
  // tile prefix: one warp scans the per-expert tile counts
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int32_t sum = 0;
    bool ok = true;
    for (int e = e0; e < e1; ++e) {
      const int32_t c = off[e + 1] - off[e];
      ok = ok && c >= 0;
      sum += (c + chunk - 1) / chunk;
    }
    int32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int32_t acc = incl - sum;
    for (int e = e0; e < e1; ++e) {
      tb[e] = acc;
      acc += (off[e + 1] - off[e] + chunk - 1) / chunk;
    }
    const bool all_ok = __all_sync(0xFFFFFFFFu, ok) && off[0] == 0 && off[E] <= R;
    if (lane == 0) {
      s_bad = all_ok ? 0 : 1;
      if (!all_ok) raise_status(status, NVFP4_ERR_DEVICE_CHECK);
    }
  }
  __syncthreads();
  float g;
  if (partials) {
    uint32_t m = s_wmax[0];
    for (int w = 1; w < (blockDim.x >> 5); ++w) m = max(m, s_wmax[w]);
    g = __fdiv_rn(bf16_bits_to_f32(m), 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_ptr = g;
  } else {
    g = *g_ptr;
  }
  const ScaleK k = scale_consts(g);
  __shared__ float4 s_elem[kElemTable];
  fill_elem_table(s_elem, g);
  __syncthreads();
  if (s_bad) return;
  // Work item: a warp quantises 32 consecutive 16-element blocks of one
  // source row (K % 64 == 0, so every group of four blocks is whole) and
  // writes them to each of the row's routes: 256 bytes of codes and one
  // scale word per four blocks per route.
  const int lane = threadIdx.x & 31;
  const uint32_t bpr = static_cast<uint32_t>(K >> 4);
  const uint32_t segs = (bpr + 31u) / 32u;
  const int64_t n_kb = (K + 255) >> 8;
  const uint64_t items = static_cast<uint64_t>(rows) * segs;
  const uint64_t wstride = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
  const int32_t nroutes = off[E];
  for (uint64_t it = static_cast<uint64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < items; it += wstride) {
    const int64_t r = static_cast<int64_t>(it / segs);
    const uint32_t b = static_cast<uint32_t>(it - static_cast<uint64_t>(r) * segs) * 32u + lane;
    const bool valid = b < bpr;
    Block16 q;
    q.packed = make_uint2(0u, 0u);
    q.sf = 0u;
    if (valid) {
      const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + static_cast<int64_t>(b) * 16);
      q = quantize_block(__ldg(src), __ldg(src + 1), k, s_elem);
    }
    const uint32_t word = gather4_bytes(q.sf);
    const int64_t kb = b >> 4;
    const int bb = static_cast<int>(b & 15);        // 16-element block inside the K block
    // The row's routes, 32 at a time: lane j looks up route j (its position,
    // expert and place in the tile layout) so that the lookups of all routes
    // overlap, then every route's codes and scales are stored by the warp.
    for (int j0 = 0; j0 < fanout; j0 += 32) {
      int32_t p = -1;
      int32_t rt_l = 0, row_l = 0;
      if (j0 + lane < fanout) {
        p = route_pos ? route_pos[r * fanout + j0 + lane] : static_cast<int32_t>(r);
        if (p >= 0 && p < nroutes) {
          const int e = find_expert(off, E, p);
          const int32_t local = p - off[e];
          rt_l = tb[e] + local / chunk;
          row_l = local % chunk;
        } else {
          p = -1;                                   // dropped route
        }
      }
      const int nj = min(32, fanout - j0);
      for (int j = 0; j < nj; ++j) {
        if (__shfl_sync(0xFFFFFFFFu, p, j) < 0) continue;
        const int64_t rt = __shfl_sync(0xFFFFFFFFu, rt_l, j);
        const int row = __shfl_sync(0xFFFFFFFFu, row_l, j);
        if (valid) {
          *reinterpret_cast<uint2*>(tiles + tile_code_offset(rt, row, kb, bb * 8, n_kb)) =
              q.packed;
          if ((lane & 3) == 0)
            *reinterpret_cast<uint32_t*>(tiles + tile_scale_offset(rt, row, kb, bb, n_kb)) = word;
        }
      }
    }
  }
}

// Already-quantised rows into route order: route p copies row src(p) of the
// packed codes [rows, K/2] and row-major scales [rows, K/16], src(p) =
// route_token[p] (or p itself without a gather list), into the grouped
// operand-tile layout the dispatch quantiser writes (same chunking, same
// positions).  Work item: one 16-byte chunk of codes or one 4-byte word of
// scales of one route; the expert of a route comes from a binary search of
// the offsets.  A source row outside [0, rows) is a device-side input error:
// the route is skipped and the status word records it.
__global__ void __launch_bounds__(256) gather_dispatch_kernel(
    const uint8_t* __restrict__ packed, const uint8_t* __restrict__ sf, int64_t rows, int64_t K,
    const int32_t* __restrict__ route_token, const int32_t* __restrict__ expert_offsets, int E,
    int64_t R, int chunk, uint8_t* __restrict__ tiles, int* status) {
  extern __shared__ int32_t sh[];
  int32_t* off = sh;              // [E + 1]
  int32_t* tb = sh + (E + 1);     // [E]
  __shared__ int32_t s_bad;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) off[e] = expert_offsets[e];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int32_t sum = 0;
    bool ok = true;
    for (int e = e0; e < e1; ++e) {
      const int32_t c = off[e + 1] - off[e];
      ok = ok && c >= 0;
      sum += (c + chunk - 1) / chunk;
    }
    int32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int32_t acc = incl - sum;
    for (int e = e0; e < e1; ++e) {
      tb[e] = acc;
      acc += (off[e + 1] - off[e] + chunk - 1) / chunk;
    }
    const bool all_ok = __all_sync(0xFFFFFFFFu, ok) && off[0] == 0 && off[E] <= R;
    if (lane == 0) {
      s_bad = all_ok ? 0 : 1;
      if (!all_ok) raise_status(status, NVFP4_ERR_DEVICE_CHECK);
    }
  }
  __syncthreads();
  if (s_bad) return;
  const int64_t half = K >> 1, kblk = K >> 4;
  const int64_t n_kb = (K + 255) >> 8;
  const int64_t per_route = (half >> 4) + (kblk >> 2);   // 16-byte code chunks + scale words
  const int64_t total = static_cast<int64_t>(off[E]) * per_route;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int32_t p = static_cast<int32_t>(i / per_route);
    const int64_t w = i - static_cast<int64_t>(p) * per_route;
    const int64_t src = route_token ? static_cast<int64_t>(route_token[p]) : p;
    if (src < 0 || src >= rows) {
      if (w == 0) raise_status(status, NVFP4_ERR_DEVICE_CHECK);
      continue;
    }
    const int e = find_expert(off, E, p);
    const int32_t local = p - off[e];
    const int64_t rt = tb[e] + local / chunk;
    const int row = local % chunk;
    if (w < (half >> 4)) {
      const int64_t byte = w << 4;
      *reinterpret_cast<uint4*>(tiles + tile_code_offset(rt, row, byte >> 7,
                                                         static_cast<int>(byte & 127), n_kb)) =
          *reinterpret_cast<const uint4*>(packed + src * half + byte);
    } else {
      const int64_t col = (w - (half >> 4)) << 2;        // first of four scale columns
      const uint8_t* q = sf + src * kblk + col;
      const uint32_t v = static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 8) |
                         (static_cast<uint32_t>(q[2]) << 16) | (static_cast<uint32_t>(q[3]) << 24);
      *reinterpret_cast<uint32_t*>(tiles + tile_scale_offset(rt, row, col >> 4,
                                                             static_cast<int>(col & 15), n_kb)) = v;
    }
  }
}

// Packed rows [rows, K/2] + row-major scales [rows, K/16] -> operand tiles,
// rows padded to 128 and K to 256 with zeros.  One thread per 16-byte chunk
// of codes (and per 4 scale bytes).
__global__ void __launch_bounds__(256) prepack_tiles_kernel(const uint8_t* __restrict__ packed,
                                                            const uint8_t* __restrict__ sf,
                                                            int64_t rows, int64_t K,
                                                            uint8_t* __restrict__ tiles) {
  const int64_t rows_pad = (rows + 127) & ~static_cast<int64_t>(127);
  const int64_t n_kb = (K + 255) >> 8;
  const int64_t half = K >> 1;
  const int64_t chunks = n_kb * 8;                  // 16-byte chunks per padded row
  const int64_t sgroups = n_kb * 4;                 // 4-byte scale groups per padded row
  const int64_t per_row = chunks + sgroups;
  const int64_t total = rows_pad * per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t r = i / per_row, w = i - r * per_row;
    const int64_t rt = r >> 7;
    const int row = static_cast<int>(r & 127);
    if (w < chunks) {
      const int64_t kb = w >> 3;
      const int c = static_cast<int>(w & 7) * 16;
      const int64_t byte = kb * 128 + c;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows && byte < half) v = *reinterpret_cast<const uint4*>(packed + r * half + byte);
      *reinterpret_cast<uint4*>(tiles + tile_code_offset(rt, row, kb, c, n_kb)) = v;
    } else {
      const int64_t gidx = w - chunks;
      const int64_t kb = gidx >> 2;
      const int sg = static_cast<int>(gidx & 3) * 4;
      const int64_t col = kb * 16 + sg;
      uint32_t v = 0;
      if (r < rows && col < (K >> 4)) v = *reinterpret_cast<const uint32_t*>(sf + r * (K >> 4) + col);
      *reinterpret_cast<uint32_t*>(tiles + tile_scale_offset(rt, row, kb, sg, n_kb)) = v;
    }
  }
}

// Row-major scales [rows, kblk] -> atom layout; one thread per (padded row,
// group of 4 scale columns), padding rows written as zero.
__global__ void __launch_bounds__(256) prepack_kernel(const uint8_t* __restrict__ src,
                                                      int64_t rows, int64_t kblk,
                                                      uint8_t* __restrict__ dst) {
  const int64_t rows_pad = (rows + 127) & ~static_cast<int64_t>(127);
  const int64_t ncg = kblk >> 2;
  const int64_t total = rows_pad * ncg;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t r = i / ncg, cg = i - r * ncg;
    uint32_t v = 0;
    if (r < rows) {
      const uint8_t* p = src + r * kblk + cg * 4;
      v = static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
          (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24);
    }
    *reinterpret_cast<uint32_t*>(dst + atom_offset(r, cg * 4, ncg)) = v;
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
static int grid_for(int64_t work, int sms) {
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : static_cast<int>(blocks);
}

// Blocks of 256 threads (8 warps) for `items` warp work items, capped at what
// the GPU holds at once (one wave, so no block waits for a second one).  The
// resident count per SM comes from the occupancy calculator, once per kernel.
template <typename Kernel>
static int grid_for_items(Kernel kernel, size_t smem, int64_t items, int sms) {
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, smem) != cudaSuccess ||
        n < 1)
      n = 1;
    per_sm = n;
  }
  int64_t blocks = (items + 7) / 8;
  const int64_t cap = static_cast<int64_t>(per_sm) * sms;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : static_cast<int>(blocks);
}

static int amax_grid(int64_t rows, int64_t cols, int sms) {
  const int64_t segs = ((cols >> 3) + 127) / 128;
  return grid_for_items(amax_kernel, 0, rows * segs, sms);
}

// Dispatch shared memory is at most 2 * 1024 + 1 ints (E <= 1024); the
// occupancy is taken at that size.
constexpr size_t kDispatchSmemMax = sizeof(int32_t) * (2 * 1024 + 1);

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float* g,
                        int sms, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(g, 0, sizeof(float), s);
  if (err != cudaSuccess) return err;
  if (rows == 0 || cols == 0) return cudaSuccess;
  amax_kernel<<<amax_grid(rows, cols, sms), 256, 0, s>>>(x, rows, cols, ld, g, nullptr);
  return cudaGetLastError();
}

int amax_partials_count(int64_t rows, int64_t cols, int sms) {
  return amax_grid(rows, cols, sms);
}

cudaError_t launch_amax_partials(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                 uint32_t* partials, int sms, cudaStream_t s) {
  amax_kernel<<<amax_partials_count(rows, cols, sms), 256, 0, s>>>(x, rows, cols, ld, nullptr,
                                                                 partials);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                            uint8_t* packed, uint8_t* scales, int sf_atoms, const float* g,
                            int sms, cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int64_t items =
      rows * (((cols >> 4) + kQuantItemBlocks - 1) / kQuantItemBlocks);
  quantize_kernel<<<grid_for_items(quantize_kernel, 0, items, sms), 256, 0, s>>>(
      x, rows, cols, ld, packed, scales, sf_atoms, g);
  return cudaGetLastError();
}

cudaError_t launch_quantize_dispatch(const uint16_t* x, int64_t rows, int64_t K, int64_t ld,
                                     const int32_t* route_pos, int fanout,
                                     const int32_t* expert_offsets, int E, int64_t R,
                                     int chunk_rows, uint8_t* tiles, float* g,
                                     const uint32_t* partials, int n_partials, int* status,
                                     int sms, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const size_t shmem = sizeof(int32_t) * (2 * static_cast<size_t>(E) + 1);
  const int64_t items = rows * (((K >> 4) + 31) / 32);
  quantize_dispatch_kernel<<<grid_for_items(quantize_dispatch_kernel, kDispatchSmemMax, items, sms),
                             256, shmem, s>>>(
      x, rows, K, ld, route_pos, fanout, expert_offsets, E, R, chunk_rows, tiles, g, partials,
      n_partials, status);
  return cudaGetLastError();
}

cudaError_t launch_gather_dispatch(const uint8_t* packed, const uint8_t* sf, int64_t rows,
                                   int64_t K, const int32_t* route_token,
                                   const int32_t* expert_offsets, int E, int64_t R, int chunk_rows,
                                   uint8_t* tiles, int* status, int sms, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const size_t shmem = sizeof(int32_t) * (2 * static_cast<size_t>(E) + 1);
  const int64_t work = R * ((K >> 5) + (K >> 6));
  gather_dispatch_kernel<<<grid_for(work, sms), 256, shmem, s>>>(
      packed, sf, rows, K, route_token, expert_offsets, E, R, chunk_rows, tiles, status);
  return cudaGetLastError();
}

cudaError_t launch_prepack_tiles(const uint8_t* packed, const uint8_t* sf, int64_t rows,
                                 int64_t K, uint8_t* tiles, int sms, cudaStream_t s) {
  const int64_t rows_pad = (rows + 127) & ~static_cast<int64_t>(127);
  const int64_t n_kb = (K + 255) >> 8;
  const int64_t work = rows_pad * n_kb * 12;
  if (work == 0) return cudaSuccess;
  prepack_tiles_kernel<<<grid_for(work, sms), 256, 0, s>>>(packed, sf, rows, K, tiles);
  return cudaGetLastError();
}

cudaError_t launch_prepack(const uint8_t* src, int64_t rows, int64_t kblk, uint8_t* dst,
                           int sms, cudaStream_t s) {
  const int64_t rows_pad = (rows + 127) & ~static_cast<int64_t>(127);
  if (rows_pad == 0) return cudaSuccess;
  prepack_kernel<<<grid_for(rows_pad * (kblk >> 2), sms), 256, 0, s>>>(src, rows, kblk, dst);
  return cudaGetLastError();
}

}  // namespace nvfp4
