// NVFP4 number formats and the 16-element block quantiser, shared by the
// quantiser kernels and the GEMM epilogue that quantises its own output.
//
// Format: "The Blackwell architectural split", Preserving precision --
// dual-tier scale handling (E2M1 elements, a global tensor scale and one
// block scale per 16 values).  Recipe: g = amax / (6 * 448),
// s = (amax_b / 6) / g, each step binary32 round-to-nearest-even.
#pragma once

#include "common.cuh"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Number formats (implemented from the format definitions)
// ---------------------------------------------------------------------------

// binary32 (s >= 0) -> E4M3 code, round to nearest even, saturating at 448
// (0x7E): the hardware conversion rounds once to nearest even over the whole
// E4M3 range (subnormals included, quantum 2^-9 below 2^-6) and, with
// .satfinite, clamps what lies beyond the largest finite value to 448.
__device__ __forceinline__ uint32_t e4m3_from_f32(float s) {
  if (!(s < 448.0f)) return 0x7Eu;
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
  return r & 0xFFu;
}

// E4M3 code (never NaN here) -> binary32, exact.
__device__ __forceinline__ float f32_from_e4m3(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu;
  const uint32_t m = c & 7u;
  const float mag = (e == 0u) ? static_cast<float>(m) * 0.001953125f
                              : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -mag : mag;
}

// Two binary32 products in one instruction, each rounded to nearest even:
// (a.x * b.x, a.y * b.y).
__device__ __forceinline__ float2 fmul2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "mul.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

struct Block16 {
  uint2 packed;     // 16 codes, low nibble = lower K index
  uint32_t sf;      // E4M3 code
};

// Eight binary32 values -> eight E2M1 codes in one word (value 2i in the low
// nibble of byte i, value 2i+1 in its high nibble), each rounded to nearest
// even and saturated to +-6 by the hardware conversion.
__device__ __forceinline__ uint32_t e2m1x8_rn_satfinite(const float* q) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

// Per-tensor constants of the block quantiser: the global scale g and, for
// the fast path of the block scale, c = RN(1 / RN(6 g)) (fast only while g is
// a normal number well inside the binary32 range).
struct ScaleK {
  float g;
  float c;
  bool fast;
};

__device__ __forceinline__ ScaleK scale_consts(float g) {
  ScaleK k;
  k.g = g;
  k.fast = g >= 7.52316384526264e-37f && g <= 1.0e35f;   // [2^-120, 1e35]
  k.c = k.fast ? __frcp_rn(__fmul_rn(6.0f, g)) : 0.0f;
  return k;
}

// E4M3 code of the block scale: sf = E4M3(RN(RN(amax_b / 6) / g)), 0 when
// g == 0.  s1 = RN(amax_b * c) is within 5 * 2^-24 (relative) of that exact
// two-rounding chain s, i.e. within 10 units in the last place of s; E4M3
// rounding tells two nearby values apart only across a midpoint between E4M3
// values, which in the normal range (s >= 2^-6) has binary32 mantissa bits
// 19..0 equal to 0x80000.  So when s1 is normal for E4M3, below 448 and more
// than 16 units in the last place from such a midpoint, E4M3(s1) = E4M3(s);
// at or above 448 both saturate.  Everything else takes the exact chain.
__device__ __forceinline__ uint32_t block_scale_code(float amax_b, const ScaleK& k) {
  if (!(k.g > 0.0f)) return 0u;
  if (k.fast) {
    const float s1 = __fmul_rn(amax_b, k.c);
    if (s1 >= 448.0f) return 0x7Eu;
    const uint32_t low = __float_as_uint(s1) & 0xFFFFFu;
    if (s1 >= 0.015625f && low - 0x7FFF0u > 32u) return e4m3_from_f32(s1);
  }
  return e4m3_from_f32(__fdiv_rn(__fdiv_rn(amax_b, 6.0f), k.g));
}

// Exact element codes of a block with decode scale d > 0 (or d == 0): code =
// E2M1(RN(v / d)), the signed zero code when d == 0; the sign bit of every
// code is set from v itself.
template <typename Get>
__device__ __forceinline__ uint2 codes_exact(float d, Get get) {
  uint32_t sgn[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e) sgn[e >> 3] |= (__float_as_uint(get(e)) >> 31) << (4 * (e & 7) + 3);
  float q[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float v = get(e);
    q[e] = (d != 0.0f) ? __fdiv_rn(v, d) : __fmul_rn(v, 0.0f);
  }
  return make_uint2(e2m1x8_rn_satfinite(q) | sgn[0], e2m1x8_rn_satfinite(q + 8) | sgn[1]);
}

// Bracketing multipliers of 1/d: with inv = RN(1/d), ilo = RN(inv (1 - 2^-20))
// and ihi = RN(inv (1 + 2^-20)) satisfy, for every v, |v ilo| < |RN(v/d)| <
// |v ihi| after rounding (the combined relative error of the roundings is
// below 4 * 2^-24, far inside the 2^-20 margin; products that underflow are
// below every E2M1 rounding boundary).  E2M1 rounding is monotone, so when
// RN(v ilo) and RN(v ihi) give the same code, so does RN(v/d).
struct Bracket {
  float lo, hi;
  bool ok;
};

__device__ __forceinline__ Bracket bracket_of(float d) {
  Bracket b;
  const float inv = __frcp_rn(d);
  b.ok = d != 0.0f && inv < 3.0e38f && inv > 2.4e-38f;   // 1/d normal: relative bounds hold
  b.lo = __fmul_rn(inv, 0.99999904632568359375f);   // 1 - 2^-20
  b.hi = __fmul_rn(inv, 1.00000095367431640625f);   // 1 + 2^-20
  return b;
}

// The elements of a block whose bracketing products gave different codes
// (diff: the XOR of the two code words, kBase: the block index of the word's
// first value) get the exact code E2M1(RN(v / d)) in place; every other code
// is already exact.  Typically one element or none: only a quotient within
// 2^-19 of an E2M1 rounding boundary lands here.
template <int kBase, typename Get>
__device__ __forceinline__ uint32_t fix_codes(uint32_t c, uint32_t diff, float d, Get get) {
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const uint32_t mask = 0xFu << (4 * n);
    if (diff & mask) {
      const float q = __fdiv_rn(get(kBase + n), d);
      uint32_t code;
      asm("{\n\t.reg .b8 t;\n\t"
          "cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\t"
          "cvt.u32.u8 %0, t;\n\t}"
          : "=r"(code) : "f"(q), "f"(0.0f));
      c = (c & ~mask) | ((code & 0xFu) << (4 * n));
    }
  }
  return c;
}

// One block from its magnitude maximum and an accessor for its 16 finite
// binary32 values: s = (amax_b / 6) / g (0 when g == 0), sf = E4M3(s),
// d = e4m3(sf) * g, code = E2M1(v / d), or the signed zero code when d == 0.
template <typename Get>
__device__ __forceinline__ Block16 quantize16_with(float amax_b, const ScaleK& k, Get get) {
  Block16 b;
  b.sf = block_scale_code(amax_b, k);
  const float d = __fmul_rn(f32_from_e4m3(b.sf), k.g);
  const Bracket br = bracket_of(d);
  if (br.ok) {
    uint32_t sgn[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 16; ++e)
      sgn[e >> 3] |= (__float_as_uint(get(e)) >> 31) << (4 * (e & 7) + 3);
    float lo[16], hi[16];
    const float2 l2 = make_float2(br.lo, br.lo), h2 = make_float2(br.hi, br.hi);
#pragma unroll
    for (int e = 0; e < 16; e += 2) {        // two roundings per instruction
      const float2 v = make_float2(get(e), get(e + 1));
      const float2 l = fmul2_rn(v, l2), h = fmul2_rn(v, h2);
      lo[e] = l.x;
      lo[e + 1] = l.y;
      hi[e] = h.x;
      hi[e + 1] = h.y;
    }
    uint32_t c0 = e2m1x8_rn_satfinite(lo), c1 = e2m1x8_rn_satfinite(lo + 8);
    const uint32_t x0 = c0 ^ e2m1x8_rn_satfinite(hi), x1 = c1 ^ e2m1x8_rn_satfinite(hi + 8);
    if ((x0 | x1) != 0u) {
      c0 = fix_codes<0>(c0, x0, d, get);
      c1 = fix_codes<8>(c1, x1, d, get);
    }
    b.packed = make_uint2(c0 | sgn[0], c1 | sgn[1]);
    return b;
  }
  b.packed = codes_exact(d, get);
  return b;
}

// Element constants of one block-scale code c under a global scale g,
// gathered per tensor into a table of 128 entries (E4M3 codes 0..0x7F) so
// that a block looks up, instead of computing, its bracket: {lo, hi, d}
// with d = e4m3(c) * g.  A zero d (g == 0 or c == 0) gets lo = hi = 0, whose
// products are the signed zeros the exact path gives; a d whose reciprocal
// leaves the normal range gets lo = -1, which sends its blocks to the exact
// path.
__device__ __forceinline__ float4 elem_consts(uint32_t c, float g) {
  const float d = __fmul_rn(f32_from_e4m3(c), g);
  const Bracket br = bracket_of(d);
  if (br.ok) return make_float4(br.lo, br.hi, d, 0.0f);
  return make_float4(d == 0.0f ? 0.0f : -1.0f, 0.0f, d, 0.0f);
}

constexpr int kElemTable = 128;

// Fills a block's shared table of element constants (every thread of the
// block calls it; the caller synchronises before the first lookup).
__device__ __forceinline__ void fill_elem_table(float4* t, float g) {
  for (int c = threadIdx.x; c < kElemTable; c += blockDim.x) t[c] = elem_consts(c, g);
}

// Codes of one code word (values kBase..kBase+7 of the block: words
// kBase/2..kBase/2+3 of w) whose bracketing products disagreed (diff: the
// XOR of the two code words) replaced by the exact code E2M1(RN(v / d));
// only the disagreeing values are visited, typically one.
template <int kBase>
__device__ __forceinline__ uint32_t fix_codes_bf16(uint32_t c, uint32_t diff, float d,
                                                   const uint32_t (&w)[8]) {
  while (diff != 0u) {
    const int n = (__ffs(diff) - 1) >> 2;           // first disagreeing value
    const uint32_t mask = 0xFu << (4 * n);
    diff &= ~mask;
    const int i = n >> 1;
    const uint32_t word = i == 0 ? w[kBase / 2] : i == 1 ? w[kBase / 2 + 1]
                        : i == 2 ? w[kBase / 2 + 2] : w[kBase / 2 + 3];
    const float v = __uint_as_float((n & 1) ? (word & 0xFFFF0000u) : (word << 16));
    const float q = __fdiv_rn(v, d);
    uint32_t code;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(code) : "f"(q), "f"(0.0f));
    c = (c & ~mask) | ((code & 0xFu) << (4 * n));
  }
  return c;
}

// Per half: max(|a|, |b|) of two BF16 pairs, with the XOR of the signs in
// the sign bit (which the caller drops).
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Sixteen BF16 values as eight words (value 2i in the low half of word i),
// with the tensor's table of element constants.  The block maximum takes
// BF16 magnitudes two per instruction (finite inputs); the
// element codes take their sign from the conversion of the bracketing
// products, which carry the sign of v (E2M1 rounding is symmetric, and a
// product that rounds to zero keeps its sign).
__device__ __forceinline__ Block16 quantize_bf16x16(const uint32_t (&w)[8], const ScaleK& k,
                                                    const float4* table) {
  const uint32_t m = bf16x2_max_abs(bf16x2_max_abs(bf16x2_max_abs(w[0], w[1]), bf16x2_max_abs(w[2], w[3])),
                                     bf16x2_max_abs(bf16x2_max_abs(w[4], w[5]), bf16x2_max_abs(w[6], w[7])));
  const uint32_t amax_bits = bf16x2_max_abs(m, m >> 16) & 0x7FFFu;
  Block16 b;
  b.sf = block_scale_code(__uint_as_float(amax_bits << 16), k);
  const float4 t = table[b.sf];
  if (t.x >= 0.0f) {
    float lo[16], hi[16];
    const float2 l2 = make_float2(t.x, t.x), h2 = make_float2(t.y, t.y);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 v = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
      const float2 l = fmul2_rn(v, l2), h = fmul2_rn(v, h2);
      lo[2 * i] = l.x;
      lo[2 * i + 1] = l.y;
      hi[2 * i] = h.x;
      hi[2 * i + 1] = h.y;
    }
    uint32_t c0 = e2m1x8_rn_satfinite(lo), c1 = e2m1x8_rn_satfinite(lo + 8);
    const uint32_t x0 = c0 ^ e2m1x8_rn_satfinite(hi), x1 = c1 ^ e2m1x8_rn_satfinite(hi + 8);
    if ((x0 | x1) != 0u) {
      c0 = fix_codes_bf16<0>(c0, x0, t.z, w);
      c1 = fix_codes_bf16<8>(c1, x1, t.z, w);
    }
    b.packed = make_uint2(c0, c1);
    return b;
  }
  b.packed = codes_exact(t.z, [&](int e) {
    return __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
  });
  return b;
}

// Sixteen finite binary32 values (amax_b = max |v|).
__device__ __forceinline__ Block16 quantize16(const float* v, const ScaleK& k) {
  float amax_b = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e) amax_b = fmaxf(amax_b, fabsf(v[e]));
  return quantize16_with(amax_b, k, [&](int e) { return v[e]; });
}

}  // namespace nvfp4
