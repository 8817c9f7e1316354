// Launch arguments of the decode-attention kernels, shared between
// attention.cu and the C ABI layer.  Not part of the public interface.
#pragma once

#include <cuda.h>

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

struct AttnArgs {
  const uint16_t* q;               // BF16 [B, Hq, D]
  const uint8_t* k_packed;         // [B, Hkv, L_max, D/2]
  const uint8_t* k_scales;         // [B, Hkv, L_max, D/16] E4M3
  const uint8_t* v_packed;
  const uint8_t* v_scales;
  const float* gk;                 // device globals of the K and V caches
  const float* gv;
  const int32_t* seq_lens;         // [B]
  int32_t B, Hq, Hkv;
  int64_t L_max;
  int32_t chunk;                   // tokens per split
  int32_t splits;                  // ceil(L_max / chunk)
  float scale;                     // softmax scale
  uint16_t* out;                   // BF16 [B, Hq, D]
  float* ws_o;                     // [B, Hq, splits, D] partial weighted values
  float* ws_ml;                    // [B, Hq, splits, 2] partial max (base 2) and sum
  float* ws_s;                     // [B, Hq, L_max] base-2 scores (heads of 256 and 512)
  int* status;
  uint64_t timeout_ns;             // bounded waits of the tensor-core kernel
  uint32_t debug_flags;            // kDebugSkipFirstStage: test hook, see nvfp4.h
};

// Tokens per split of the decode attention: the smallest power of two from
// 128 up to 4096 that leaves about a thousand (sequence, KV head, split) work
// items at most.  A function of the shape only, so that the workspace size
// is.  The CUDA-core kernel launches one CTA per item; the tensor-core kernels
// (one CTA per SM for heads of 64 and 128, two for the wider heads' two
// passes) walk several items per CTA.  (Splits half as long for the wider
// heads, for an evener share over 304 CTAs, measured slower: each item's q,
// partials and merge cost more than the balance gained.)
inline int attention_chunk(int64_t L_max, int64_t B, int64_t Hkv) {
  const int64_t want = (L_max * B * Hkv + 1023) / 1024;
  int ch = 128;
  while (ch < want && ch < 4096) ch <<= 1;
  return ch;
}
// The tensor-core kernels' copies: 2-D maps over the K and V code arrays
// (rows of D/2 bytes, 128-row boxes, the row-width swizzle; for heads of 256
// and 512, boxes of 64 bytes = 128 dimensions with the 64-byte swizzle) and
// over the scale arrays (viewed as 16-byte rows, boxes of 128 cache rows; for
// heads of 256 and 512, rows of D/16 bytes and boxes of 16 bytes x 128 rows).
struct AttnMaps {
  CUtensorMap k_codes, v_codes, k_scales, v_scales;
};

// maps: null when decode_attention_tc_applies is false.
cudaError_t launch_decode_attention(const AttnArgs& a, int D, const AttnMaps* maps,
                                    cudaStream_t s);
// The pipelined split kernels with both contractions on the tensor cores
// (attention_tc.cu for heads of 64 and 128, attention_tc_wide.cu for heads of
// 256 and 512): heads of 128 and wider in groups of 2, 4 or 8 query heads and
// heads of 64 in groups of 4 or 8, both scale arrays 16-byte aligned (and for
// heads of 64 and 128, L_max * D / 16 a multiple of 16), and fewer than 2^31
// cache rows (the copies' row coordinate).
bool decode_attention_tc_applies(const AttnArgs& a, int D);
cudaError_t launch_decode_attention_tc(const AttnArgs& a, int D, const AttnMaps& m,
                                       cudaStream_t s);
cudaError_t launch_decode_attention_tc_wide(const AttnArgs& a, int D, const AttnMaps& m,
                                            cudaStream_t s);
cudaError_t init_attention_tc_attributes();
cudaError_t init_attention_tc_wide_attributes();

}  // namespace nvfp4
