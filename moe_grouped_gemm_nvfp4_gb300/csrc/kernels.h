// Internal launchers shared between the kernel translation units and the
// C ABI layer.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4 {

// quantize.cu
cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float* g,
                        int sms, cudaStream_t s);
cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                            uint8_t* packed, uint8_t* scales, int sf_atoms, const float* g,
                            int sms, cudaStream_t s);
// Per-block maxima of |x| (magnitude bits) into partials[0, count) for a
// later quantize_dispatch launch to reduce.
int amax_partials_count(int64_t rows, int64_t cols, int sms);
cudaError_t launch_amax_partials(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                 uint32_t* partials, int sms, cudaStream_t s);
// With partials, every block derives g from them and block 0 stores it in
// *g; without, g is read from *g.
cudaError_t launch_quantize_dispatch(const uint16_t* x, int64_t rows, int64_t K, int64_t ld,
                                     const int32_t* route_pos, int fanout,
                                     const int32_t* expert_offsets, int E, int64_t R,
                                     int chunk_rows, uint8_t* tiles, float* g,
                                     const uint32_t* partials, int n_partials, int* status,
                                     int sms, cudaStream_t s);
// Copies already-quantised rows (packed + row-major scales) into the grouped
// operand tiles of route order; route p reads row route_token[p] (or p).
cudaError_t launch_gather_dispatch(const uint8_t* packed, const uint8_t* sf, int64_t rows,
                                   int64_t K, const int32_t* route_token,
                                   const int32_t* expert_offsets, int E, int64_t R, int chunk_rows,
                                   uint8_t* tiles, int* status, int sms, cudaStream_t s);
cudaError_t launch_prepack_tiles(const uint8_t* packed, const uint8_t* sf, int64_t rows,
                                 int64_t K, uint8_t* tiles, int sms, cudaStream_t s);
cudaError_t launch_prepack(const uint8_t* src, int64_t rows, int64_t kblk, uint8_t* dst,
                           int sms, cudaStream_t s);

// sparse.cu
cudaError_t launch_prune_2of4(const uint16_t* w, int64_t rows, int64_t cols, int64_t ld,
                              uint16_t* out, int64_t ld_out, int sms, cudaStream_t s);
cudaError_t launch_prepack_sparse_tiles(const uint8_t* packed, const uint8_t* sf, int64_t rows,
                                        int64_t K, uint8_t* tiles, int* status, int sms,
                                        cudaStream_t s);

// route.cu
cudaError_t init_route_attributes();
cudaError_t launch_route(const int32_t* ids, int64_t T, int topk, int E, int32_t* offsets,
                         int32_t* route_token, int32_t* route_slot, int32_t* route_pos,
                         int* status, cudaStream_t s);

// gemm.cu
enum GemmMode : int {
  kDenseRowsX = 0,      // C[x][y]: X = A (M side), Y = B
  kDenseRowsY = 1,      // C[y][x]: X = B, Y = A (small M)
  kGrouped = 2,         // out[route][n]
  kGroupedCombine = 3,  // ws[token][n] += w * y
  kGroupedSiluMul = 4,  // h[route][f] = SiLU(gate) * up, quantised into h_tiles
  kGroupedSiluBf16 = 5, // h[route][f] = SiLU(gate) * up, BF16 into out (two-phase form)
  kMlpFused = 6,        // the SiLU-mul units, then the down projection's combine units over
                        // h in the same launch (each token tile's down units wait on a
                        // ready count its gate_up units raise)
};

struct GemmArgs {
  const uint8_t* sfx;              // dense: X scales, atom layout; grouped: X operand tiles
  const uint8_t* sfy;              // dense: Y scales, atom layout; grouped: Y operand tiles
  const float* gx;                 // X global (grouped: per expert [E])
  const float* gy;                 // Y global
  int64_t K;
  int32_t rows_x;                  // dense: rows of X
  int32_t rows_y;                  // dense: rows of Y; grouped: R (rows of A)
  const int32_t* expert_offsets;   // grouped
  int32_t E;
  int32_t n_out;                   // grouped: rows of each expert's W
  void* out;                       // BF16
  int64_t ldc;
  int32_t vec_store;               // rows of C are 16-byte aligned (ldc % 8 == 0)
  int32_t ybox_rows;               // dense: rows per TMA box of Y (16 or 128)
  const int32_t* route_token;      // combine
  const int32_t* route_slot;
  const float* topk_w;
  int32_t topk;
  int32_t n_tokens;                // combine: T, the rows of ws (route_token must be < T)
  float* ws;                       // combine: FP32 [T, n_out]
  int* status;
  uint64_t timeout_ns;
  uint32_t debug_flags;            // kDebugSkipFirstStage: test hook, see nvfp4.h
  uint8_t* h_tiles;                // SiLU-mul: NVFP4 operand tiles of h (K = n_out / 2)
  const float* g_h;                // SiLU-mul: global scale of h (given)
  int32_t h_nkb;                   // SiLU-mul: 256-element K blocks of h
  int32_t sparse_w;                // grouped: X operand tiles are 2:4-sparse tiles
  const uint8_t* sfx2;             // fused MLP: operand tiles of the down projection [E * n_out2, K2]
  const float* gx2;                // fused MLP: down projection globals [E]
  int64_t K2;                      // fused MLP: depth of the down projection (= n_out / 2)
  int32_t n_out2;                  // fused MLP: rows of each expert's down weight
  uint32_t* ready;                 // fused MLP: per token tile, gate_up units done
  int32_t x_map;                   // grouped: X codes through the tensor map tmx (row-major
                                   // [E * n_out, K/2]) and X scales in the atom layout at sfx,
                                   // instead of operand tiles
};

// Test hook: the producer of every CTA leaves its first pipeline stage
// unfilled, so the first MMA wait can only end by its time limit.
constexpr uint32_t kDebugSkipFirstStage = 1u;

constexpr int kGroupedMaxExperts = 256;

// Token-tile width of the grouped GEMM (32, 64 or 128 routes), a function of
// the route and expert counts only.  With want = ~1.6x the mean routes per
// expert: 32 when the widest experts of a balanced routing fit 32 rows, 64 up
// to want = 80 (a mean of ~50 routes), else 128.  Past that point too many
// experts need a second 64-row tile, whose unit streams the weight tile again
// and pays a second epilogue (at a mean of 64 routes, 128-row tiles took the
// down projection from 0.239 to 0.197 ms).  The grouped
// activation layout cuts each expert's routes into chunks of this width.
inline int grouped_chunk_rows(int64_t routes, int experts) {
  const int64_t want = experts > 0 ? (routes * 8 + experts * 5 - 1) / (experts * 5) : 128;
  return want <= 32 ? 32 : (want <= 80 ? 64 : 128);
}

// Token-tile width of the grouped GEMM itself: the chunk width, or 256 when
// experts average well over 160 routes (prefill).  A 256-row token tile spans
// two consecutive 128-row operand tiles of the layout above.
inline int grouped_tile_width(int64_t routes, int experts) {
  const int64_t want = experts > 0 ? (routes * 8 + experts * 5 - 1) / (experts * 5) : 128;
  return want > 256 ? 256 : grouped_chunk_rows(routes, experts);
}
constexpr int64_t kOperandTileBytes = 16384 + 2048;   // 128 rows x 256 K: codes + scale atoms
// 2:4-sparse weight tile, same 128 rows x 256 K: kept bytes (four 64-K slices
// of 16 bytes per row), 4-bit combination indices (two 128-K halves of 8
// bytes per row), scale atoms as in the dense tile
constexpr int64_t kSparseTileBytes = 8192 + 2048 + 2048;
constexpr int kSparseComboOffset = 8192;
constexpr int kSparseScaleOffset = 10240;

cudaError_t init_gemm_attributes();
cudaError_t launch_gemm(const CUtensorMap& tmx, const CUtensorMap& tmy, const GemmArgs& a,
                        int mode, int sms, cudaStream_t s);
// gemm_pair.cu: the single GEMM on CTA pairs (cta_group::2, 256 x 256 tiles);
// tmx / tmy: A and B codes (128-row boxes, 128-byte swizzle), tsx / tsy: their
// atom-layout scales as rows of 512 bytes (boxes of four atoms).
cudaError_t init_gemm_pair_attributes();
cudaError_t launch_gemm_pair(const CUtensorMap& tmx, const CUtensorMap& tmy,
                             const CUtensorMap& tsx, const CUtensorMap& tsy, const GemmArgs& a,
                             cudaStream_t s);
// gemm_pair_grouped.cu: the grouped GEMM on CTA pairs for 256-route token
// tiles with BF16 output (prefill shapes), dense operand tiles only.  Maps
// over the tile buffers viewed as rows of 128 bytes (an operand tile is 144
// such rows: 128 of codes, 16 of scale atoms), no swizzle: the weight tiles
// with boxes of 144 rows, the token tiles with boxes of 128 rows (codes) and
// of 16 rows (scales).
struct GroupedPairMaps {
  CUtensorMap x_codes, x_scales, y_codes, y_scales;
};
cudaError_t init_grouped_pair_attributes();
// 256 when the pair kernel takes this launch, else 0
int grouped_pair_width(const GemmArgs& a, int mode);
cudaError_t launch_grouped_pair(const GroupedPairMaps& m, const GemmArgs& a, int mode,
                                cudaStream_t s);
// Fused expert MLP in one cooperative persistent launch (mode kMlpFused).
cudaError_t launch_mlp_fused(const GemmArgs& a, int sms, cudaStream_t s);
cudaError_t launch_combine_finalize(const float* ws, int64_t T, int64_t N, void* out, int sms,
                                    cudaStream_t s);

}  // namespace nvfp4
