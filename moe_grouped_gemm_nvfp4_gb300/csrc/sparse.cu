// 2:4-sparse NVFP4 weights: pruning and the sparse operand-tile layout.
//
// "The FP4 Frontier", Finding 6 (sparse FP4 assessment): structured 2:4
// sparsity halves the bits of an NVFP4 weight, and the experts of an MoE
// model can be pruned independently.  Here the unit of sparsity is the
// packed byte (the two E2M1 values at K = 2i, 2i+1): every aligned group of
// four bytes keeps two.  In decode the grouped GEMM is bound by the weight
// bytes it streams, so the weights travel compressed (kept bytes + a 4-bit
// combination index + the scales: two thirds of the dense tile) and are
// expanded in shared memory before the dense block-scaled MMA reads them.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

// Magnitude pruning of BF16 weights, one thread per group of four element
// pairs (16 bytes): pair i scores |w[2i]| + |w[2i+1]| (one binary32
// addition); the two best pairs stay, equal scores favouring the lower
// position; the other two become +0.
__global__ void __launch_bounds__(256) prune_2of4_kernel(const uint16_t* __restrict__ w,
                                                         int64_t rows, int64_t groups_per_row,
                                                         int64_t ld, uint16_t* out,
                                                         int64_t ld_out) {
  const int64_t total = rows * groups_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t r = i / groups_per_row, g = i - r * groups_per_row;
    const uint4 v = *reinterpret_cast<const uint4*>(w + r * ld + 8 * g);
    uint32_t pair[4] = {v.x, v.y, v.z, v.w};     // pair p: elements 2p (low half), 2p + 1
    float score[4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
      score[p] = __fadd_rn(bf16_bits_to_f32(pair[p] & 0x7FFFu),
                           bf16_bits_to_f32((pair[p] >> 16) & 0x7FFFu));
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      int ahead = 0;                             // pairs ranked before pair p
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q != p) ahead += (score[q] > score[p]) || (score[q] == score[p] && q < p);
      if (ahead >= 2) pair[p] = 0u;
    }
    *reinterpret_cast<uint4*>(out + r * ld_out + 8 * g) = make_uint4(pair[0], pair[1], pair[2], pair[3]);
  }
}

// Combination index of the kept positions of a group whose non-zero bytes
// form `mask`: the non-zero positions, made up to two with the lowest zero
// positions; (i0, i1) numbered lexicographically, i.e. i0 (7 - i0) / 2 +
// (i1 - i0 - 1).
__device__ __forceinline__ void kept_positions(uint32_t mask, int& i0, int& i1) {
  uint32_t m = mask & 0xFu;
  while (__popc(m) < 2) m |= ~m & (m + 1u);       // lowest zero position
  i0 = __ffs(m) - 1;
  i1 = 31 - __clz(m);
}

// Sparse operand tiles.  One thread per (padded row, K block, 64-K slice j):
// the slice's 32 packed bytes (eight groups) become 16 kept bytes at
// j * 2048 + row * 16, eight combination nibbles (one 32-bit word of the
// row's 128-K half j / 2) and the slice's four scales (one 32-bit word of
// scale atom j).  Padding rows and K blocks are zero (combination 0).
// A group with more than two non-zero bytes raises NVFP4_ERR_DEVICE_CHECK.
__global__ void __launch_bounds__(256) prepack_sparse_tiles_kernel(
    const uint8_t* __restrict__ packed, const uint8_t* __restrict__ sf, int64_t rows, int64_t K,
    uint8_t* __restrict__ tiles, int* status) {
  const int64_t rows_pad = (rows + 127) & ~static_cast<int64_t>(127);
  const int64_t n_kb = (K + 255) >> 8;
  const int64_t half = K >> 1;
  const int64_t total = rows_pad * n_kb * 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t r = i / (n_kb * 4);
    const int64_t rem = i - r * n_kb * 4;
    const int64_t kb = rem >> 2;
    const int j = static_cast<int>(rem & 3);
    const int row = static_cast<int>(r & 127);
    const int64_t byte0 = kb * 128 + j * 32;     // first packed byte of the slice
    const bool valid = r < rows && byte0 < half;
    uint32_t src[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (valid) {
      const uint4 a = *reinterpret_cast<const uint4*>(packed + r * half + byte0);
      const uint4 b = *reinterpret_cast<const uint4*>(packed + r * half + byte0 + 16);
      src[0] = a.x; src[1] = a.y; src[2] = a.z; src[3] = a.w;
      src[4] = b.x; src[5] = b.y; src[6] = b.z; src[7] = b.w;
    }
    uint32_t kept[4] = {0u, 0u, 0u, 0u};
    uint32_t combos = 0;
    bool ok = true;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint32_t word = src[g];
      uint32_t mask = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p) mask |= (((word >> (8 * p)) & 0xFFu) != 0u ? 1u : 0u) << p;
      ok = ok && __popc(mask) <= 2;
      int i0, i1;
      kept_positions(mask, i0, i1);
      const uint32_t two = ((word >> (8 * i0)) & 0xFFu) | (((word >> (8 * i1)) & 0xFFu) << 8);
      kept[g >> 1] |= two << (16 * (g & 1));
      combos |= static_cast<uint32_t>(i0 * (7 - i0) / 2 + (i1 - i0 - 1)) << (4 * g);
    }
    if (!ok) raise_status(status, NVFP4_ERR_DEVICE_CHECK);
    uint32_t scales = 0;
    const int64_t col = kb * 16 + j * 4;
    if (r < rows && col < (K >> 4))
      scales = *reinterpret_cast<const uint32_t*>(sf + r * (K >> 4) + col);
    uint8_t* tile = tiles + ((r >> 7) * n_kb + kb) * kSparseTileBytes;
    *reinterpret_cast<uint4*>(tile + j * 2048 + row * 16) =
        make_uint4(kept[0], kept[1], kept[2], kept[3]);
    *reinterpret_cast<uint32_t*>(tile + kSparseComboOffset + (j >> 1) * 1024 + row * 8 +
                                 4 * (j & 1)) = combos;
    *reinterpret_cast<uint32_t*>(tile + kSparseScaleOffset + j * 512 + (row & 31) * 16 +
                                 ((row >> 5) & 3) * 4) = scales;
  }
}

int grid_for(int64_t work, int sms) {
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_prune_2of4(const uint16_t* w, int64_t rows, int64_t cols, int64_t ld,
                              uint16_t* out, int64_t ld_out, int sms, cudaStream_t s) {
  const int64_t work = rows * (cols / 8);
  if (work == 0) return cudaSuccess;
  prune_2of4_kernel<<<grid_for(work, sms), 256, 0, s>>>(w, rows, cols / 8, ld, out, ld_out);
  return cudaGetLastError();
}

cudaError_t launch_prepack_sparse_tiles(const uint8_t* packed, const uint8_t* sf, int64_t rows,
                                        int64_t K, uint8_t* tiles, int* status, int sms,
                                        cudaStream_t s) {
  const int64_t work = ((rows + 127) / 128) * 128 * ((K + 255) / 256) * 4;
  if (work == 0) return cudaSuccess;
  prepack_sparse_tiles_kernel<<<grid_for(work, sms), 256, 0, s>>>(packed, sf, rows, K, tiles,
                                                                   status);
  return cudaGetLastError();
}

}  // namespace nvfp4
