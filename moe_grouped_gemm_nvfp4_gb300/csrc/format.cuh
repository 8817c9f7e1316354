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

// One block from its magnitude maximum and an accessor for its 16 finite
// binary32 values: s = (amax_b / 6) / g (0 when g == 0), sf = E4M3(s),
// d = e4m3(sf) * g, code = E2M1(v / d), or the signed zero code when d == 0.
// The sign bit of every code is set from v itself, so values that round to
// zero keep their sign whatever the conversion does with negative zeros.
template <typename Get>
__device__ __forceinline__ Block16 quantize16_with(float amax_b, float g, Get get) {
  const float s = (g > 0.0f) ? __fdiv_rn(__fdiv_rn(amax_b, 6.0f), g) : 0.0f;
  const uint32_t sf = e4m3_from_f32(s);
  const float d = __fmul_rn(f32_from_e4m3(sf), g);
  uint32_t sgn[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e) sgn[e >> 3] |= (__float_as_uint(get(e)) >> 31) << (4 * (e & 7) + 3);
  Block16 b;
  b.sf = sf;
  // Fast path: q1 = v * RN(1/d) is within 2^-23 (relative) of v / d, and the
  // correctly rounded quotient within 2^-24 of that, so both lie between
  // q1 (1 - 2^-20) and q1 (1 + 2^-20).  The E2M1 conversion is monotone, so
  // when the two bounds give the same codes those are the codes of the
  // rounded quotient.  Otherwise (a quotient within ~2^-20 of a rounding
  // boundary, or 1/d out of range) every code comes from the exact division.
  const float inv = __frcp_rn(d);
  if (d != 0.0f && inv < 3.0e38f) {
    float lo[16], hi[16];
    const float2 inv2 = make_float2(inv, inv);
    const float2 dn = make_float2(0.99999904632568359375f, 0.99999904632568359375f);  // 1 - 2^-20
    const float2 up = make_float2(1.00000095367431640625f, 1.00000095367431640625f);  // 1 + 2^-20
#pragma unroll
    for (int e = 0; e < 16; e += 2) {        // the same roundings, two per instruction
      const float2 q1 = fmul2_rn(make_float2(get(e), get(e + 1)), inv2);
      const float2 l = fmul2_rn(q1, dn), h = fmul2_rn(q1, up);
      lo[e] = l.x;
      lo[e + 1] = l.y;
      hi[e] = h.x;
      hi[e + 1] = h.y;
    }
    const uint32_t c0 = e2m1x8_rn_satfinite(lo), c1 = e2m1x8_rn_satfinite(lo + 8);
    if (c0 == e2m1x8_rn_satfinite(hi) && c1 == e2m1x8_rn_satfinite(hi + 8)) {
      b.packed = make_uint2(c0 | sgn[0], c1 | sgn[1]);
      return b;
    }
  }
  float q[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float v = get(e);
    q[e] = (d != 0.0f) ? __fdiv_rn(v, d) : __fmul_rn(v, 0.0f);
  }
  b.packed = make_uint2(e2m1x8_rn_satfinite(q) | sgn[0], e2m1x8_rn_satfinite(q + 8) | sgn[1]);
  return b;
}

// Sixteen finite binary32 values (amax_b = max |v|).
__device__ __forceinline__ Block16 quantize16(const float* v, float g) {
  float amax_b = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e) amax_b = fmaxf(amax_b, fabsf(v[e]));
  return quantize16_with(amax_b, g, [&](int e) { return v[e]; });
}

}  // namespace nvfp4
