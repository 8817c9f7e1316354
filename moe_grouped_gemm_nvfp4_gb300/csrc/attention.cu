// Decode attention over an NVFP4 KV cache.
//
// "The Blackwell architectural split", The Breakthrough -- The A4Q Kernel:
// keys and values stay packed in NVFP4 (E2M1 values, an E4M3 scale per 16
// numbers along the head dimension, one FP32 global for K and one for V,
// "Preserving precision -- dual-tier scale handling") and are dequantised in
// registers inside the attention loop, never staged as wider copies.  One
// query token per sequence: every cache byte is read once and each element
// feeds G = Hq / Hkv multiply-adds, so for the grouped-query ratios of
// decode the work is bound by HBM and runs on the CUDA cores.
//
// Split-KV: CTA (split, kv head j, sequence b) covers the `chunk` tokens
// [split * chunk, ...) of that sequence for the G query heads of KV head j
// and leaves an unnormalised partial (running max, sum, weighted values) in
// the workspace; a second kernel merges the splits and writes BF16.
//
// Per warp, blocks of 32 tokens: every load of the block is issued first
// (lane l reads token l's key and value rows, 16 bytes at a time, coalesced
// across the warp: one memory round trip per block); scores lane-per-token;
// an online softmax update per block (base-2 exponentials with log2(e)
// folded into q); the value rows go through a per-warp shared-memory stage
// and are accumulated lane-per-dimension (lane owns D / 32 consecutive
// dimensions of every token's value row).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "attention.h"

namespace nvfp4 {

namespace {

constexpr int kAttnWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

// Two E2M1 codes (low nibble first) -> two floats, exactly.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h) : "r"(byte & 0xFFu));
  const __half2 v = *reinterpret_cast<const __half2*>(&h);
  return __half22float2(v);
}

// One E4M3 scale byte -> float, exactly.
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h) : "r"(byte & 0xFFu));
  const __half2 v = *reinterpret_cast<const __half2*>(&h);
  return __low2float(v);
}

// Two FP32 fused multiply-adds in one instruction: (a.x b.x + c.x, a.y b.y + c.y).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\tmov.b64 pc, {%6, %7};\n\t"
      "fma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

template <int D, int G>
__global__ void __launch_bounds__(kAttnWarps * 32) decode_attention_kernel(const AttnArgs a) {
  constexpr int DL = D / 32;          // value dimensions per lane
  constexpr int KB = D / 2;           // code bytes per token row
  constexpr int SB = D / 16;          // scale bytes per token row
  constexpr int KC = KB / 16;         // 16-byte chunks per row
  // staged value row: codes, then scales, padded to 16 bytes so that the
  // 16-byte stores of every lane's row stay aligned
  constexpr int kVRow = (KB + SB + 15) / 16 * 16;
  constexpr int kStageBytes = 32 * kVRow;                       // one warp's block
  constexpr int kOBytes = kAttnWarps * G * D * 4;               // merge buffer
  constexpr int kUnion = kAttnWarps * kStageBytes > kOBytes ? kAttnWarps * kStageBytes : kOBytes;
  __shared__ __align__(16) float q_s[G][D];
  __shared__ float m_s[kAttnWarps][G], l_s[kAttnWarps][G];
  // value blocks staged per warp during the loop; the warps' partials after it
  __shared__ __align__(16) uint8_t u_s[kUnion];

  const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n = a.seq_lens[b];
  if (n < 0 || n > a.L_max) {
    if (threadIdx.x == 0) raise_status(a.status, NVFP4_ERR_DEVICE_CHECK);
    n = 0;
  }
  const int64_t t0 = static_cast<int64_t>(split) * a.chunk;
  const int64_t t1 = min(static_cast<int64_t>(n), t0 + a.chunk);
  const int64_t row0 = (static_cast<int64_t>(b) * a.Hkv + j) * a.L_max;   // cache row of token 0

  // q of the group's heads, times scale * gk * log2(e)
  const float qmul = a.scale * (*a.gk) * kLog2e;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int g = i / D, d = i - g * D;
    const int64_t qi = (static_cast<int64_t>(b) * a.Hq + j * G + g) * D + d;
    q_s[g][d] = bf16_bits_to_f32(a.q[qi]) * qmul;
  }
  __syncthreads();

  float m[G], l[G], o[G][DL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.0f;
#pragma unroll
    for (int i = 0; i < DL; ++i) o[g][i] = 0.0f;
  }
  uint8_t* vstage = u_s + warp * kStageBytes;

  for (int64_t blk = t0 + 32 * warp; blk < t1; blk += 32 * kAttnWarps) {
    const int64_t t = blk + lane;
    const bool valid = t < t1;
    // every load of the block first (one memory round trip): this lane's
    // token's key row and scales, and its value row and scales (staged below)
    uint4 kr[KC], vr[KC];
    uint32_t ks[(SB + 3) / 4], vs[(SB + 3) / 4];
    if (valid) {
      const uint8_t* krow = a.k_packed + (row0 + t) * KB;
      const uint8_t* vrow = a.v_packed + (row0 + t) * KB;
#pragma unroll
      for (int c = 0; c < KC; ++c) {
        kr[c] = *reinterpret_cast<const uint4*>(krow + 16 * c);
        vr[c] = *reinterpret_cast<const uint4*>(vrow + 16 * c);
      }
      const uint8_t* ksrow = a.k_scales + (row0 + t) * SB;
      const uint8_t* vsrow = a.v_scales + (row0 + t) * SB;
#pragma unroll
      for (int i = 0; i < (SB + 3) / 4; ++i) {
        if constexpr (SB >= 4) {
          ks[i] = *reinterpret_cast<const uint32_t*>(ksrow + 4 * i);
          vs[i] = *reinterpret_cast<const uint32_t*>(vsrow + 4 * i);
        }
      }
    }
    // ---- scores, lane-per-token
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = valid ? 0.0f : -INFINITY;
    if (valid) {
#pragma unroll
      for (int c = 0; c < KC; ++c) {                 // 32 elements = two scale blocks
        const uint32_t w[4] = {kr[c].x, kr[c].y, kr[c].z, kr[c].w};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float2 part[G];                            // even / odd elements' partial sums
#pragma unroll
          for (int g = 0; g < G; ++g) part[g] = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int wi = 0; wi < 2; ++wi) {
            const uint32_t word = w[2 * half + wi];
#pragma unroll
            for (int by = 0; by < 4; ++by) {
              const float2 e = e2m1x2_to_float2(word >> (8 * by));
              const int d = 32 * c + 16 * half + 8 * wi + 2 * by;
#pragma unroll
              for (int g = 0; g < G; ++g)
                part[g] = ffma2(*reinterpret_cast<const float2*>(&q_s[g][d]), e, part[g]);
            }
          }
          const int blk16 = 2 * c + half;            // scale block of these 16 elements
          const float sf = e4m3_to_float(ks[blk16 / 4] >> (8 * (blk16 % 4)));
#pragma unroll
          for (int g = 0; g < G; ++g) s[g] = fmaf(part[g].x + part[g].y, sf, s[g]);
        }
      }
    }
    // ---- stage the value rows: row `lane` of the block at lane * kVRow
    __syncwarp();                                    // the previous block's reads are done
    if (valid) {
#pragma unroll
      for (int c = 0; c < KC; ++c) *reinterpret_cast<uint4*>(vstage + lane * kVRow + 16 * c) = vr[c];
#pragma unroll
      for (int i = 0; i < SB / 4; ++i)
        *reinterpret_cast<uint32_t*>(vstage + lane * kVRow + KB + 4 * i) = vs[i];
    }
    // ---- online softmax over the block (base 2)
    float p[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mn = fmaxf(m[g], warp_max(s[g]));    // finite: lane 0 is valid
      const float corr = (m[g] == -INFINITY) ? 0.0f : exp2f(m[g] - mn);
      p[g] = valid ? exp2f(s[g] - mn) : 0.0f;
      l[g] = fmaf(l[g], corr, warp_sum(p[g]));
#pragma unroll
      for (int i = 0; i < DL; ++i) o[g][i] *= corr;
      m[g] = mn;
    }
    __syncwarp();                                    // the staged rows are visible
    // ---- values, lane-per-dimension, from the staged rows
    const int nt = static_cast<int>(min(static_cast<int64_t>(32), t1 - blk));
    for (int tt = 0; tt < nt; ++tt) {
      const uint8_t* vrow = vstage + tt * kVRow;
      const float sf = e4m3_to_float(vrow[KB + (lane * DL) / 16]);
      const uint8_t* vc = vrow + lane * (DL / 2);
      uint32_t codes[(DL / 2 + 3) / 4];
      if constexpr (DL / 2 == 1) codes[0] = *vc;
      else if constexpr (DL / 2 == 2) codes[0] = *reinterpret_cast<const uint16_t*>(vc);
      else if constexpr (DL / 2 == 4) codes[0] = *reinterpret_cast<const uint32_t*>(vc);
      else {
        const uint2 c2 = *reinterpret_cast<const uint2*>(vc);
        codes[0] = c2.x;
        codes[1] = c2.y;
      }
      float2 wgt[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float w1 = __shfl_sync(0xFFFFFFFFu, p[g], tt) * sf;
        wgt[g] = make_float2(w1, w1);
      }
#pragma unroll
      for (int i = 0; i < DL / 2; ++i) {
        const float2 e = e2m1x2_to_float2(codes[i / 4] >> (8 * (i % 4)));
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 r = ffma2(wgt[g], e, make_float2(o[g][2 * i], o[g][2 * i + 1]));
          o[g][2 * i] = r.x;
          o[g][2 * i + 1] = r.y;
        }
      }
    }
  }

  // ---- merge the warps, write this split's partial
  __syncthreads();                                   // staging space becomes the merge buffer
  float (*o_s)[G][D] = reinterpret_cast<float (*)[G][D]>(u_s);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      m_s[warp][g] = m[g];
      l_s[warp][g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < DL; ++i) o_s[warp][g][lane * DL + i] = o[g][i];
  }
  __syncthreads();
  const int64_t nsplit = a.splits;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int g = i / D, d = i - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w)
      if (l_s[w][g] > 0.0f) M = fmaxf(M, m_s[w][g]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      if (l_s[w][g] > 0.0f) {
        const float f = exp2f(m_s[w][g] - M);
        L = fmaf(l_s[w][g], f, L);
        O = fmaf(o_s[w][g][d], f, O);
      }
    }
    const int64_t part = (static_cast<int64_t>(b) * a.Hq + j * G + g) * nsplit + split;
    a.ws_o[part * D + d] = O;
    if (d == 0) {
      a.ws_ml[2 * part] = M;
      a.ws_ml[2 * part + 1] = L;
    }
  }
}

// Merges the splits of (sequence b, query head h) for dimensions 128 y ..
// 128 y + 127 (blockIdx.y = y): out = gv * sum_s O_s 2^(m_s - M) / sum_s l_s
// 2^(m_s - M) in BF16 over the splits with l_s > 0; zeros for an empty
// sequence.  The split weights 2^(m_s - M) are computed once per CTA into
// shared memory (1024 splits at a time); warp c of the eight sums the splits
// c, c + 8, ... for four dimensions per lane (16-byte loads, four in flight),
// and the eight partial sums are added in warp order.
constexpr int kCombineThreads = 256, kCombineChunk = 1024;

__global__ void __launch_bounds__(kCombineThreads) decode_attention_combine_kernel(
    const AttnArgs a, int D) {
  __shared__ float wsh[kCombineChunk];
  __shared__ float4 part[8][32];
  __shared__ float red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t bh = blockIdx.x;
  const int64_t nsplit = a.splits;
  const int64_t base = bh * nsplit;
  const float* ml = a.ws_ml + 2 * base;
  float m = -INFINITY;
  for (int64_t s = tid; s < nsplit; s += kCombineThreads)
    if (ml[2 * s + 1] > 0.0f) m = fmaxf(m, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  float l = 0.0f;
  for (int64_t s = tid; s < nsplit; s += kCombineThreads) {
    const float ls = ml[2 * s + 1];
    if (ls > 0.0f) l = fmaf(ls, exp2f(ml[2 * s] - M), l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
  if (lane == 0) red[warp] = l;
  __syncthreads();
  float L = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) L += red[w];
  const int d0 = static_cast<int>(blockIdx.y) * 128 + 4 * lane;
  const bool active = d0 < D;
  const float* op = a.ws_o + base * D + d0;
  float ox = 0.0f, oy = 0.0f, oz = 0.0f, ow = 0.0f;
  for (int64_t s0 = 0; s0 < nsplit; s0 += kCombineChunk) {
    const int n = static_cast<int>(nsplit - s0 < kCombineChunk ? nsplit - s0 : kCombineChunk);
    __syncthreads();                                   // the last chunk's weights are used
    for (int k = tid; k < n; k += kCombineThreads) {
      const float ls = ml[2 * (s0 + k) + 1];
      wsh[k] = ls > 0.0f ? exp2f(ml[2 * (s0 + k)] - M) : 0.0f;
    }
    __syncthreads();
    if (active) {
      int k = warp;
      for (; k + 24 < n; k += 32) {
        float4 v[4];
        float w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          w[u] = wsh[k + 8 * u];
          v[u] = w[u] != 0.0f ? *reinterpret_cast<const float4*>(op + (s0 + k + 8 * u) * D)
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (w[u] != 0.0f) {
            ox = fmaf(v[u].x, w[u], ox);
            oy = fmaf(v[u].y, w[u], oy);
            oz = fmaf(v[u].z, w[u], oz);
            ow = fmaf(v[u].w, w[u], ow);
          }
      }
      for (; k < n; k += 8) {
        const float w = wsh[k];
        if (w != 0.0f) {
          const float4 v = *reinterpret_cast<const float4*>(op + (s0 + k) * D);
          ox = fmaf(v.x, w, ox);
          oy = fmaf(v.y, w, oy);
          oz = fmaf(v.z, w, oz);
          ow = fmaf(v.w, w, ow);
        }
      }
    }
  }
  part[warp][lane] = make_float4(ox, oy, oz, ow);
  __syncthreads();
  if (warp == 0 && active) {
    float4 t = part[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
      const float4 u = part[w][lane];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const float gv = *a.gv;
    uint32_t h[4];
    const float x[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      h[u] = f32_to_bf16_rn(L > 0.0f ? __fmul_rn(gv, __fdiv_rn(x[u], L)) : 0.0f);
    *reinterpret_cast<uint2*>(a.out + bh * D + d0) = make_uint2(h[0] | (h[1] << 16),
                                                                h[2] | (h[3] << 16));
  }
}

// the merge: one CTA per (sequence, query head, 128 dimensions)
dim3 combine_grid(const AttnArgs& a, int D) {
  return dim3(static_cast<unsigned>(static_cast<int64_t>(a.B) * a.Hq),
              static_cast<unsigned>((D + 127) / 128));
}

template <int D, int G>
cudaError_t launch_d_g(const AttnArgs& a, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(a.splits), static_cast<unsigned>(a.Hkv),
                  static_cast<unsigned>(a.B));
  decode_attention_kernel<D, G><<<grid, kAttnWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, int G, cudaStream_t s) {
  switch (G) {
    case 1: return launch_d_g<D, 1>(a, s);
    case 2: return launch_d_g<D, 2>(a, s);
    case 4: return launch_d_g<D, 4>(a, s);
    default:
      if constexpr (D <= 256) return launch_d_g<D, 8>(a, s);
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_attention(const AttnArgs& a, int D, const AttnMaps* maps,
                                    cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  cudaError_t e = cudaSuccess;
  if (a.splits == 0) {             // empty cache: the merge writes zeros
    decode_attention_combine_kernel<<<combine_grid(a, D), kCombineThreads, 0, s>>>(a, D);
    return cudaGetLastError();
  }
  // groups of 2-8 query heads over 128-wide heads and 4-8 over 64-wide heads:
  // the tensor-core kernel (attention_tc.cu); single heads (and pairs over
  // 64-wide heads), where the multiply-adds cost less than the FP16
  // expansion, and wider heads: the kernel above
  if (maps && decode_attention_tc_applies(a, D)) {
    e = launch_decode_attention_tc(a, D, *maps, s);
  } else {
    switch (D) {
      case 64: e = launch_d<64>(a, G, s); break;
      case 128: e = launch_d<128>(a, G, s); break;
      case 256: e = launch_d<256>(a, G, s); break;
      default: e = launch_d<512>(a, G, s); break;
    }
  }
  if (e != cudaSuccess) return e;
  decode_attention_combine_kernel<<<combine_grid(a, D), kCombineThreads, 0, s>>>(a, D);
  return cudaGetLastError();
}

}  // namespace nvfp4
