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

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Number formats (implemented from the format definitions)
// ---------------------------------------------------------------------------

// binary32 (s >= 0, finite) -> E4M3 code, round to nearest even, saturating
// at 448 (0x7E).  Normal range: keep 3 mantissa bits with RNE (a carry into
// the exponent is the correct next code).  Below 2^-6: subnormal quantum
// 2^-9, so the code is s * 2^9 rounded to the nearest even integer.
__device__ __forceinline__ uint32_t e4m3_from_f32(float s) {
  if (!(s < 448.0f)) return 0x7Eu;
  const uint32_t b = __float_as_uint(s);
  const uint32_t exp = (b >> 23) & 0xFFu;
  if (exp >= 121u) {                       // s >= 2^-6
    const uint32_t mant = b & 0x7FFFFFu;
    const uint32_t keep = mant >> 20;
    const uint32_t rest = mant & 0xFFFFFu;
    uint32_t v = ((exp - 120u) << 3) | keep;
    if (rest > 0x80000u || (rest == 0x80000u && (keep & 1u))) v += 1u;
    return v;
  }
  return __float2uint_rn(s * 512.0f);      // 0..8; 8 is the smallest normal
}

// E4M3 code (never NaN here) -> binary32, exact.
__device__ __forceinline__ float f32_from_e4m3(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu;
  const uint32_t m = c & 7u;
  const float mag = (e == 0u) ? static_cast<float>(m) * 0.001953125f
                              : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -mag : mag;
}

// |q| -> E2M1 magnitude code with round to nearest even and saturation to 6:
// each threshold is a midpoint between neighbouring magnitudes, inclusive
// when the upper neighbour has the even code.
__device__ __forceinline__ uint32_t e2m1_mag_code(float a) {
  return static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) +
         static_cast<uint32_t>(a > 1.25f) + static_cast<uint32_t>(a >= 1.75f) +
         static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) +
         static_cast<uint32_t>(a > 5.0f);
}

// ---------------------------------------------------------------------------
// Tensor amax -> global scale
// ---------------------------------------------------------------------------
// Each block reduces |x| over a grid-stride slice (BF16 magnitudes compare as
// integers), turns its maximum into g_b = amax_b / 2688 and folds it into
// *g with an integer atomicMax on the float bits (valid for g_b >= 0).
// Division by a positive constant is monotone, so max_b(g_b) = max(amax)/2688.
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ x,
                                                   int64_t rows, int64_t cols, int64_t ld,
                                                   float* g) {
  uint32_t m = 0;
  const bool vec = ((cols & 7) == 0) && ((ld & 7) == 0) &&
                   ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (vec) {
    const int64_t vpr = cols >> 3;
    const int64_t total = rows * vpr;
    for (int64_t i = tid; i < total; i += stride) {
      const int64_t r = i / vpr, v = i - r * vpr;
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(x + r * ld) + v);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        m = max(m, w[j] & 0x7FFFu);
        m = max(m, (w[j] >> 16) & 0x7FFFu);
      }
    }
  } else {
    const int64_t total = rows * cols;
    for (int64_t i = tid; i < total; i += stride) {
      const int64_t r = i / cols, c = i - r * cols;
      m = max(m, static_cast<uint32_t>(x[r * ld + c]) & 0x7FFFu);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ uint32_t wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (blockDim.x >> 5); ++w) m = max(m, wm[w]);
    const float gb = __fdiv_rn(bf16_bits_to_f32(m), 2688.0f);
    atomicMax(reinterpret_cast<unsigned int*>(g), __float_as_uint(gb));
  }
}

// ---------------------------------------------------------------------------
// Quantise one 16-element block
// ---------------------------------------------------------------------------
struct Block16 {
  uint2 packed;     // 16 codes, low nibble = lower K index
  uint32_t sf;      // E4M3 code
};

__device__ __forceinline__ Block16 quantize_block(const uint4 lo, const uint4 hi, float g) {
  uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t amax_bits = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    amax_bits = max(amax_bits, w[j] & 0x7FFFu);
    amax_bits = max(amax_bits, (w[j] >> 16) & 0x7FFFu);
  }
  const float amax_b = bf16_bits_to_f32(amax_bits);
  const float s = (g > 0.0f) ? __fdiv_rn(__fdiv_rn(amax_b, 6.0f), g) : 0.0f;
  const uint32_t sf = e4m3_from_f32(s);
  const float d = __fmul_rn(f32_from_e4m3(sf), g);
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t bits = (w[j] >> (16 * h)) & 0xFFFFu;
      const uint32_t sign = (bits >> 15) << 3;
      uint32_t code = sign;
      if (d != 0.0f) {
        const float q = __fdiv_rn(bf16_bits_to_f32(bits), d);
        code |= e2m1_mag_code(fabsf(q));
      }
      const int e = 2 * j + h;                 // element index 0..15
      out[e >> 3] |= code << (4 * (e & 7));
    }
  }
  Block16 b;
  b.packed = make_uint2(out[0], out[1]);
  b.sf = sf;
  return b;
}

__device__ __forceinline__ int64_t atom_offset(int64_t r, int64_t c, int64_t n_cgroups) {
  return ((r >> 7) * n_cgroups + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// One thread per 16-element block of x [rows, cols].
__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t* __restrict__ x,
                                                       int64_t rows, int64_t cols, int64_t ld,
                                                       uint8_t* __restrict__ packed,
                                                       uint8_t* __restrict__ scales,
                                                       int sf_atoms, const float* g_ptr) {
  const float g = *g_ptr;
  const int64_t bpr = cols >> 4;
  const int64_t total = rows * bpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t r = i / bpr, b = i - r * bpr;
    const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + b * 16);
    const Block16 q = quantize_block(__ldg(src), __ldg(src + 1), g);
    *reinterpret_cast<uint2*>(packed + r * (cols >> 1) + b * 8) = q.packed;
    const int64_t so = sf_atoms ? atom_offset(r, b, cols >> 6) : r * bpr + b;
    scales[so] = static_cast<uint8_t>(q.sf);
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

// Quantise source rows and write each one to its route positions: packed
// data in route order [R, K/2], scales in the grouped atom layout (each
// expert's routes start a fresh 128-row tile).
__global__ void __launch_bounds__(256) quantize_dispatch_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t K, int64_t ld,
    const int32_t* __restrict__ route_pos, int fanout,
    const int32_t* __restrict__ expert_offsets, int E, int64_t R,
    uint8_t* __restrict__ packed, uint8_t* __restrict__ scales, const float* g_ptr,
    int* status) {
  extern __shared__ int32_t sh[];
  int32_t* off = sh;              // [E + 1]
  int32_t* tb = sh + (E + 1);     // [E]
  for (int e = threadIdx.x; e <= E; e += blockDim.x) off[e] = expert_offsets[e];
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    bool ok = off[0] == 0 && off[E] <= R;
    for (int e = 0; e < E; ++e) {
      const int32_t c = off[e + 1] - off[e];
      if (c < 0) ok = false;
      tb[e] = acc;
      acc += (c + 127) >> 7;
    }
    if (!ok) { raise_status(status, NVFP4_ERR_DEVICE_CHECK); tb[0] = -1; }
  }
  __syncthreads();
  if (E > 0 && tb[0] < 0) return;
  const float g = *g_ptr;
  const int64_t bpr = K >> 4;
  const int64_t total = rows * bpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t ncg = K >> 6;
  const int32_t nroutes = off[E];
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t r = i / bpr, b = i - r * bpr;
    const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + b * 16);
    const Block16 q = quantize_block(__ldg(src), __ldg(src + 1), g);
    for (int j = 0; j < fanout; ++j) {
      const int32_t p = route_pos ? route_pos[r * fanout + j] : static_cast<int32_t>(r);
      if (p < 0 || p >= nroutes) continue;          // dropped route
      *reinterpret_cast<uint2*>(packed + static_cast<int64_t>(p) * (K >> 1) + b * 8) = q.packed;
      const int e = find_expert(off, E, p);
      const int64_t prow = static_cast<int64_t>(tb[e]) * 128 + (p - off[e]);
      scales[atom_offset(prow, b, ncg)] = static_cast<uint8_t>(q.sf);
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

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float* g,
                        int sms, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(g, 0, sizeof(float), s);
  if (err != cudaSuccess) return err;
  if (rows == 0 || cols == 0) return cudaSuccess;
  amax_kernel<<<grid_for(rows * cols / 8, sms), 256, 0, s>>>(x, rows, cols, ld, g);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                            uint8_t* packed, uint8_t* scales, int sf_atoms, const float* g,
                            int sms, cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  quantize_kernel<<<grid_for(rows * (cols >> 4), sms), 256, 0, s>>>(x, rows, cols, ld, packed,
                                                                   scales, sf_atoms, g);
  return cudaGetLastError();
}

cudaError_t launch_quantize_dispatch(const uint16_t* x, int64_t rows, int64_t K, int64_t ld,
                                     const int32_t* route_pos, int fanout,
                                     const int32_t* expert_offsets, int E, int64_t R,
                                     uint8_t* packed, uint8_t* scales, const float* g,
                                     int* status, int sms, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const size_t shmem = sizeof(int32_t) * (2 * static_cast<size_t>(E) + 1);
  quantize_dispatch_kernel<<<grid_for(rows * (K >> 4), sms), 256, shmem, s>>>(
      x, rows, K, ld, route_pos, fanout, expert_offsets, E, R, packed, scales, g, status);
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
