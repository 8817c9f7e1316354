/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 block-scaled GEMM library.
 *
 * NVFP4: E2M1 4-bit values (1 sign, 2 exponent, 1 mantissa bit), two per
 * byte with the lower K index in the low nibble, one FP8-E4M3 block scale per
 * 16 consecutive K elements and one FP32 global scale per tensor
 * ("The Blackwell architectural split", Preserving precision -- dual-tier
 * scale handling).  Dequantised value: x = e2m1 * e4m3(block) * global.
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers to caller-owned memory unless stated.
 *     The library never allocates or frees memory; it keeps only a per-device
 *     cache of launch attributes and a per-device status word.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it.
 *   - Global scales are device floats, so no call forces a host sync.
 *   - Host-side argument errors return immediately and enqueue nothing:
 *       NVFP4_ERR_INVALID_ARG  null pointer, negative size;
 *       NVFP4_ERR_UNSUPPORTED  shape/alignment/device outside what the
 *                              kernels implement (K % 64, 16-byte alignment,
 *                              device not sm_103, workspace too small ...);
 *       NVFP4_ERR_CUDA         a CUDA call failed (launch error).
 *   - Device-side failures (a bounded pipeline wait that expired, routing
 *     offsets that are not monotone, expert ids out of range) are recorded in
 *     the per-device status word read by nvfp4_device_status(); the kernels
 *     return early instead of trapping.  No failure leaves an output
 *     silently unwritten without a non-OK status somewhere: this is the
 *     lesson of the all-zeros backend in "The SM120 FP4 GEMM Kernel
 *     Investigation" (The Breaking Point: FlashInfer #2577).
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,
  NVFP4_ERR_UNSUPPORTED = 2,
  NVFP4_ERR_CUDA = 3,
  NVFP4_ERR_TIMEOUT = 4,       /* a bounded device wait expired            */
  NVFP4_ERR_DEVICE_CHECK = 5   /* a device-side input check failed         */
} nvfp4_status;

/* Flags of the quantiser entry points. */
#define NVFP4_SF_ROWMAJOR   0u  /* scales as uint8 [rows, cols/16]               */
#define NVFP4_SF_ATOMS      1u  /* scales in the tensor-core atom layout         */
#define NVFP4_GLOBAL_GIVEN  2u  /* read *global_scale instead of computing it    */
#define NVFP4_AMAX_DONE     4u  /* dispatch: amax maxima already in the tiles'   */
                                /* scratch (nvfp4_amax_partials)                 */

/* Human-readable name of a status code (static string, never NULL). */
const char* nvfp4_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int nvfp4_version(void);

/*
 * Reads the status word of the current device after synchronising `stream`.
 * *status_out receives the first device-side error recorded since the last
 * reset (NVFP4_OK if none).  reset != 0 clears the word afterwards.
 */
nvfp4_status nvfp4_device_status(void* stream, int reset, int* status_out);

/*
 * Reads the calling device's status word without clearing it, after
 * synchronising `stream`: NVFP4_OK, or the first device-side error recorded
 * since the last reset (or an error of the read itself).  The same word as
 * nvfp4_device_status(stream, 0, &status).
 */
nvfp4_status nvfp4_last_device_status(void* stream);

/* Bounded-wait limit of the pipeline kernels in nanoseconds (default 1 s,
 * or NVFP4_TIMEOUT_NS from the environment at the first call). */
nvfp4_status nvfp4_set_timeout_ns(uint64_t ns);

/*
 * Test hook for the failure path of the GEMM kernels and of the tensor-core
 * decode attention (0 = off, the default).  Flag 1: the producer of every CTA
 * leaves its first pipeline stage unfilled, so the first wait on it can only
 * end by its time limit; the kernel then records NVFP4_ERR_TIMEOUT, drains its
 * own copies and MMAs, frees tensor memory and returns, and the output is
 * incomplete.  Meant for tests, with a short nvfp4_set_timeout_ns.  Other bits
 * return NVFP4_ERR_INVALID_ARG.
 */
nvfp4_status nvfp4_debug_set_flags(uint32_t flags);

/*
 * Scale bytes of a [rows, cols] matrix in the tensor-core atom layout:
 * 512-byte atoms of 128 rows x 4 scale columns (64 K elements), byte
 * (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4), atoms ordered row-tile
 * major; rows are padded to a multiple of 128.  cols % 64 == 0.
 */
size_t nvfp4_atom_scales_bytes(int64_t rows, int64_t cols);

/*
 * Bytes of the atom-layout scales for rows x kblk row-major scales (kblk =
 * K/16): what nvfp4_prepack_weights writes, rows padded to 128 and kblk to 4.
 */
size_t nvfp4_prepacked_scales_bytes(int64_t rows, int64_t kblk);

/*
 * BF16 -> NVFP4 quantiser (per-16 amax, E4M3 block scale, E2M1 round to
 * nearest even, pack): the dual-tier scaling of "The Blackwell architectural
 * split", Preserving precision -- one FP32 global scale per tensor and one
 * block scale per 16 values -- applied to activations as they arrive in BF16
 * ("The SM120 FP4 GEMM Kernel Investigation", The Context).
 *   x        BF16 [rows, cols], row stride `ld` elements (ld >= cols);
 *            cols % 16 == 0 (cols % 64 == 0 with NVFP4_SF_ATOMS).
 *   packed   uint8 [rows, cols/2] out, row-major, dense.
 *   scales   uint8 out: [rows, cols/16] row-major, or the atom layout of
 *            nvfp4_atom_scales_bytes(rows, cols) bytes with NVFP4_SF_ATOMS
 *            (then 4-byte aligned; padding rows are left unwritten).
 *   global_scale  device float: written with g = amax|x| / (6 * 448), or read
 *            as the global scale when NVFP4_GLOBAL_GIVEN is set.
 * Every step is IEEE binary32 round-to-nearest-even: s = (amax_b / 6) / g
 * (0 when g == 0), sf = E4M3_satfinite(s), d = e4m3(sf) * g, and code =
 * E2M1_satfinite(x / d), or the signed zero code when d == 0.
 */
nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                            uint8_t* packed, uint8_t* scales, float* global_scale,
                            uint32_t flags, void* stream);

/*
 * Rewrites row-major E4M3 scales [rows, kblk] (kblk = K/16, kblk % 4 == 0)
 * into the atom layout (nvfp4_atom_scales_bytes(rows, 16 * kblk) bytes);
 * padding rows are written as zero.  Offline step for weights: the block
 * scales of "The Blackwell architectural split", Preserving precision, staged
 * as the scale-factor tiles the block-scaled MMA reads ("The SM120 FP4 GEMM
 * Kernel Investigation", The Comprehensive Synthesis: scale-factor tiles
 * beside the A/B FP4 tiles).
 */
nvfp4_status nvfp4_prepack_weights(const uint8_t* scales_rowmajor, int64_t rows,
                                   int64_t kblk, uint8_t* scales_atoms, void* stream);

/*
 * Single NVFP4 GEMM: C[M, N] (BF16, row stride ldc elements) =
 * (*gA) * (*gB) * A_hat . B_hat^T, FP32 accumulation in tensor memory,
 * BF16 round-to-nearest-even output.  A_hat = e2m1 * e4m3 * global, the
 * dual-tier dequantisation of "The Blackwell architectural split",
 * Preserving precision; the large-GEMM case is the one "The Tile That Didn't
 * Fit", The Core Finding, measures against the FP4 tensor peak.
 *   A  packed [M, K/2], sfA atom layout for [M, K];
 *   B  packed [N, K/2], sfB atom layout for [N, K];
 *   K % 64 == 0, M, N >= 1, ldc >= N; A, B, sfA, sfB 16-byte aligned, C
 *   2-byte aligned (rows that are 16-byte aligned get vector stores).  Small
 *   M runs with the operands swapped (weights on the MMA's M side); the
 *   result is the same.
 */
nvfp4_status nvfp4_gemm(const uint8_t* A, const uint8_t* sfA, const float* gA,
                        const uint8_t* B, const uint8_t* sfB, const float* gB,
                        void* C, int64_t M, int64_t N, int64_t K, int64_t ldc,
                        void* stream);

/*
 * MoE routing prep ("The FP4 Frontier", Finding 5: grouped GEMM batching all
 * experts): counting sort of the T*topk routes by expert, stable by token.
 *   topk_ids        int32 [T, topk], values in [0, E)
 *   expert_offsets  int32 [E+1] out: routes of expert e are positions
 *                   expert_offsets[e] .. expert_offsets[e+1]-1
 *   route_token     int32 [T*topk] out: token of each sorted route
 *   route_slot      int32 [T*topk] out: top-k slot of each sorted route
 *   route_pos       int32 [T*topk] out (may be NULL): sorted position of the
 *                   route t*topk + slot
 * E <= 1024.  An id out of range sets NVFP4_ERR_DEVICE_CHECK on the device
 * and the route is dropped: expert_offsets[E] < T*topk then, route_token and
 * route_slot past expert_offsets[E] are left unwritten (undefined), and
 * route_pos of the dropped route is -1.  Every consumer in this library
 * reads only positions below expert_offsets[E].
 */
nvfp4_status nvfp4_moe_route(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                             int32_t* expert_offsets, int32_t* route_token,
                             int32_t* route_slot, int32_t* route_pos, void* stream);

/*
 * Operand tiles: the layout the grouped GEMM copies one pipeline stage from.
 * A tile covers 128 rows x 256 K elements and is 18432 bytes: 16384 bytes of
 * packed codes, row r at r * 128 with its 16-byte chunk j stored at chunk
 * position j ^ (r % 8) (the tensor cores' 128-byte shared-memory swizzle),
 * then 2048 bytes of scales as four atoms (one per 64 K elements, atom
 * layout as above).  Tiles are ordered row-tile major, then K block.  Rows
 * are padded to a multiple of 128 and K to a multiple of 256.
 */
size_t nvfp4_operand_tiles_bytes(int64_t rows, int64_t K);

/*
 * Offline weight prepack: packed codes [rows, K/2] and row-major scales
 * [rows, K/16] (as written by nvfp4_quantize) -> operand tiles
 * (nvfp4_operand_tiles_bytes(rows, K) bytes, padding zero).  For expert
 * weights [E, N, K] pass rows = E * N with N % 128 == 0, so that every tile
 * belongs to one expert.  K % 64 == 0; packed and tiles 16-byte aligned.
 */
nvfp4_status nvfp4_prepack_weight_tiles(const uint8_t* packed, const uint8_t* scales_rowmajor,
                                        int64_t rows, int64_t K, uint8_t* tiles, void* stream);

/*
 * Chunk width (32, 64 or 128 routes) of the grouped activation tiles for R
 * routes over E experts: with want = ceil(1.6 x R / E), 32 if want <= 32, 64 if
 * want <= 80, else 128.  It is also the grouped GEMM's token-tile width, so
 * that narrow decode tiles leave shared memory for a deeper pipeline.
 */
int nvfp4_grouped_chunk_rows(int64_t R, int32_t E);

/*
 * Bytes of the grouped activation tile buffer for R routes over E experts:
 * an upper bound on the tiles (every expert's routes are cut into chunks of
 * nvfp4_grouped_chunk_rows(R, E) rows and each chunk fills its own tile),
 * plus 16 KiB of scratch at the end in which nvfp4_quantize_dispatch keeps
 * the tensor amax's per-block maxima between its two kernels.
 */
size_t nvfp4_grouped_tiles_bytes(int64_t R, int32_t E, int64_t K);

/*
 * Quantise activations straight into route order for the grouped GEMM
 * ("The FP4 Frontier", Finding 5: grouped GEMM, token counts padded for TMA).
 *   x           BF16 [rows, K], row stride ld (elements), 16-byte aligned.
 *   route_pos   int32 [rows * fanout]: destination route of source row i,
 *               copy j is route_pos[i * fanout + j] (the route_pos output of
 *               nvfp4_moe_route with fanout = topk); negative = dropped.
 *               NULL means the rows are already in route order (rows == R,
 *               fanout == 1).
 *   expert_offsets  int32 [E+1] (device), as from nvfp4_moe_route.
 *   tiles       operand tiles out (nvfp4_grouped_tiles_bytes(R, E, K) bytes):
 *               with c = nvfp4_grouped_chunk_rows(R, E), route p of expert e,
 *               j = p - expert_offsets[e], is row j % c of tile
 *               tb[e] + j / c, tb[e] = sum over e' < e of ceil(count_e' / c).
 *               Rows past a chunk's routes are left unwritten (they only ever
 *               feed output columns the GEMM does not store).
 *   global_scale  as in nvfp4_quantize (one g over the whole of x).
 *   flags       NVFP4_GLOBAL_GIVEN: use *global_scale; NVFP4_AMAX_DONE: the
 *               tensor amax's per-block maxima of this x are already in the
 *               tiles' scratch (nvfp4_amax_partials, same x, rows, K, R, E and
 *               device), so only the quantise-and-dispatch kernel runs.
 * K % 64 == 0, E <= 1024.  Offsets that are not monotone or exceed R set
 * NVFP4_ERR_DEVICE_CHECK and nothing is written.
 */
nvfp4_status nvfp4_quantize_dispatch(const void* x, int64_t rows, int64_t K, int64_t ld,
                                     const int32_t* route_pos, int32_t fanout,
                                     const int32_t* expert_offsets, int32_t E, int64_t R,
                                     uint8_t* tiles, float* global_scale, uint32_t flags,
                                     void* stream);

/*
 * The first half of nvfp4_quantize_dispatch: the tensor amax of x as
 * per-block maxima in the scratch at the end of `tiles` (sized by
 * nvfp4_grouped_tiles_bytes(R, E, K)).  It needs no routing, so it can run
 * on another stream while nvfp4_moe_route runs; then call
 * nvfp4_quantize_dispatch with NVFP4_AMAX_DONE after both.
 */
nvfp4_status nvfp4_amax_partials(const void* x, int64_t rows, int64_t K, int64_t ld, int64_t R,
                                 int32_t E, uint8_t* tiles, void* stream);

/* Bytes of the FP32 combine workspace for T tokens and N outputs. */
size_t nvfp4_combine_workspace_bytes(int64_t T, int64_t N);

/*
 * Workspace bytes of nvfp4_grouped_gemm for T tokens, top-k, E experts, N
 * outputs and depth K: the activation operand tiles of the R = T * topk
 * routes (nvfp4_grouped_tiles_bytes without its scratch), plus, when combine
 * != 0 (topk_weights given), the FP32 sums [T, N].
 */
size_t nvfp4_grouped_gemm_workspace_bytes(int64_t T, int32_t topk, int32_t E, int64_t N,
                                          int64_t K, int32_t combine);

/*
 * MoE expert grouped GEMM ("The FP4 Frontier", Finding 5: one persistent
 * grouped GEMM over all experts, token counts padded for TMA; Finding 7:
 * small-batch decode is bound by streaming the expert weights), on
 * already-quantised operands in their plain layouts.
 *   A, sfA, gA   NVFP4 activations: packed codes uint8 [rows, K/2] and
 *                row-major E4M3 scales uint8 [rows, K/16] (nvfp4_quantize with
 *                NVFP4_SF_ROWMAJOR), device float global.  Without
 *                topk_weights: rows = T token rows gathered by route_token
 *                (route p reads row route_token[p]), or, with route_token
 *                NULL, rows = R = T * topk already in route order.  With
 *                topk_weights (the combine): rows = R in route order (the
 *                experts' intermediate), route_token then places outputs.
 *   W, sfW_tc, gW  expert weights: packed codes [E * N, K/2] (expert e's
 *                rows e * N .. e * N + N - 1), their scales in the
 *                tensor-core atom layout (nvfp4_prepack_weights over E * N
 *                rows), device float [E], one global per expert.
 *   expert_offsets, route_token, route_slot  int32, from nvfp4_moe_route.
 *   topk_weights NULL: out = BF16 [R, N] in route order, out[p, n] = gA *
 *                gW[e] * sum_k A_hat[src(p), k] W_hat[e, n, k].  FP32 [T, topk]:
 *                out = BF16 [T, N], out[t] = sum over the routes p of t of
 *                w[t, slot(p)] * y[p].
 *   workspace    caller-owned, >= nvfp4_grouped_gemm_workspace_bytes(T, topk, E,
 *                N, K, topk_weights != NULL) bytes, 16-byte aligned: the call
 *                first copies the activation rows into grouped operand tiles
 *                there (one pass over R rows), then runs the persistent GEMM.
 * N % 128 == 0, K % 64 == 0, E <= 256; A, W, sfW_tc, out 16-byte aligned.  A
 * gathered row index outside [0, rows), a token outside [0, T) or a slot
 * outside [0, topk) sets NVFP4_ERR_DEVICE_CHECK and the route is skipped.
 */
nvfp4_status nvfp4_grouped_gemm(const uint8_t* A, const uint8_t* sfA, const float* gA,
                                const uint8_t* W, const uint8_t* sfW_tc, const float* gW,
                                const int32_t* expert_offsets, int32_t E,
                                const int32_t* route_token, const float* topk_weights,
                                const int32_t* route_slot, int64_t T, int32_t topk, int64_t N,
                                int64_t K, void* out, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * The same grouped GEMM on operand tiles: the form the decode step uses,
 * with the activations quantised straight into route order by
 * nvfp4_quantize_dispatch (no separate copy pass) and the weights in one
 * contiguous tile per pipeline stage.
 *   A_tiles, gA  route-ordered activation tiles from nvfp4_quantize_dispatch
 *                and their device float global scale.
 *   W_tiles      expert weights as operand tiles over [E * N, K]
 *                (nvfp4_prepack_weight_tiles); gW device float [E], one
 *                global per expert.
 *   expert_offsets  int32 [E+1] (device), R = T * topk routes.
 *   topk_weights == NULL:  out = BF16 [R, N] in route order,
 *       out[p, n] = gA * gW[e] * sum_k A_hat[p, k] W_hat[e, n, k].
 *   topk_weights != NULL (FP32 [T, topk]):  out = BF16 [T, N],
 *       out[t] = sum over the routes p of t of w[t, slot(p)] * y[p], with
 *       route_token / route_slot from nvfp4_moe_route and an FP32 workspace
 *       of nvfp4_combine_workspace_bytes(T, N) bytes (zeroed here).  The FP32
 *       additions run in no fixed order.  A token outside [0, T) or a slot
 *       outside [0, topk) sets NVFP4_ERR_DEVICE_CHECK and that route adds
 *       nothing.
 * N % 128 == 0, K % 64 == 0, E <= 256; all buffers 16-byte aligned.
 */
nvfp4_status nvfp4_grouped_gemm_tiles(const uint8_t* A_tiles, const float* gA,
                                      const uint8_t* W_tiles, const float* gW,
                                      const int32_t* expert_offsets, int32_t E,
                                      int64_t T, int32_t topk, int64_t N, int64_t K,
                                      const int32_t* route_token, const int32_t* route_slot,
                                      const float* topk_weights,
                                      void* out, float* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * Fused expert MLP front half: the gate_up grouped GEMM, SiLU(gate) * up,
 * and the NVFP4 quantisation of the product, in one launch ("The FP4
 * Frontier", Finding 5: persistent grouped GEMM; the activation between the
 * two projections never goes to memory in BF16).
 *   A_tiles, gA, W_tiles, gW, expert_offsets, E, T, topk, K  as in
 *       nvfp4_grouped_gemm_tiles (gather orientation: A in route order).
 *   N         rows of each expert's W: rows [0, N/2) are the gate projection,
 *             rows [N/2, N) the up projection of the same N/2 features.
 *   g_h       device float: the global scale of h (given, for instance
 *             calibrated offline as amax(h) / (6 * 448)).
 *   h_tiles   out: h = SiLU(g) * u per route and feature, with
 *             g = gA * gW[e] * sum_k A_hat W_hat[e, f, :] and u the same for row
 *             N/2 + f, SiLU(z) = z / (1 + exp(-z)), all in binary32; quantised
 *             per 16 features with g_h exactly as nvfp4_quantize does, into the
 *             grouped tile layout nvfp4_quantize_dispatch writes for R routes,
 *             E experts and K = N/2 (nvfp4_grouped_tiles_bytes(R, E, N/2)
 *             bytes).  Feed it to nvfp4_grouped_gemm_tiles as A_tiles with gA = g_h.
 * N % 256 == 0, K % 64 == 0, E <= 256.  A unit holds a gate tile and its up
 * tile against one token tile of nvfp4_grouped_chunk_rows(R, E) routes (32,
 * 64 or 128).
 */
nvfp4_status nvfp4_moe_gate_up_silu(const uint8_t* A_tiles, const float* gA,
                                    const uint8_t* W_tiles, const float* gW,
                                    const int32_t* expert_offsets, int32_t E, int64_t T,
                                    int32_t topk, int64_t N, int64_t K, const float* g_h,
                                    uint8_t* h_tiles, void* stream);

/*
 * The whole expert MLP in one persistent launch ("The FP4 Frontier",
 * Finding 5: a persistent kernel over all experts; the MLP's intermediate
 * stays NVFP4 between the projections): the gate_up units of
 * nvfp4_moe_gate_up_silu (h = SiLU(g) * u quantised with the given g_h into
 * h_tiles), then in the same launch the down projection's units over h with
 * the weighted combine of nvfp4_grouped_gemm_tiles, then the BF16 rounding of
 * the sums.  A down unit starts once every gate_up unit of its token tile has
 * written its features of h (a count per token tile in the workspace, waited
 * on with the bounded wait: NVFP4_ERR_TIMEOUT on expiry).  The launch is
 * cooperative (all CTAs resident at once), so those waits always end.
 *   A_tiles, gA, W1_tiles, gW1, expert_offsets, E, T, topk, N1, K1, g_h,
 *       h_tiles  as in nvfp4_moe_gate_up_silu (N = N1).
 *   W2_tiles, gW2  down weights as operand tiles over [E * N2, N1 / 2], one
 *       global per expert.
 *   route_token, route_slot, topk_weights, out  as in nvfp4_grouped_gemm_tiles
 *       with the combine: out = BF16 [T, N2].
 *   workspace  nvfp4_moe_mlp_workspace_bytes(T, topk, E, N2) bytes, 16-byte
 *       aligned, caller-owned: the FP32 sums [T, N2] and the ready counts,
 *       cleared by the call.
 * N1 % 256 == 0, N2 % 256 == 0, K1 % 64 == 0, E <= 256.
 */
size_t nvfp4_moe_mlp_workspace_bytes(int64_t T, int32_t topk, int32_t E, int64_t N2);

nvfp4_status nvfp4_moe_mlp(const uint8_t* A_tiles, const float* gA, const uint8_t* W1_tiles,
                           const float* gW1, const uint8_t* W2_tiles, const float* gW2,
                           const int32_t* expert_offsets, int32_t E, int64_t T, int32_t topk,
                           int64_t N1, int64_t K1, int64_t N2, const float* g_h, uint8_t* h_tiles,
                           const int32_t* route_token, const int32_t* route_slot,
                           const float* topk_weights, void* out, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * Two-phase form of the fused gate_up epilogue, for callers that do not have
 * the global scale of h in advance: the same grouped GEMM and h = SiLU(g) * u
 * (binary32), written as BF16 (round to nearest even) in route order,
 * h_out[p, f] for route p and feature f < N/2 (row stride N/2 elements,
 * 16-byte aligned).  Then nvfp4_quantize_dispatch over h_out (rows = R,
 * route_pos NULL, fanout 1) finds the global of h from its amax and writes
 * the operand tiles of the down projection.  Same arguments and limits as
 * nvfp4_moe_gate_up_silu otherwise.
 */
nvfp4_status nvfp4_moe_gate_up_silu_bf16(const uint8_t* A_tiles, const float* gA,
                                         const uint8_t* W_tiles, const float* gW,
                                         const int32_t* expert_offsets, int32_t E, int64_t T,
                                         int32_t topk, int64_t N, int64_t K, void* h_out,
                                         void* stream);

/*
 * Allocation-free weighted-combine grouped GEMM.  (This entry point is a
 * library convenience; the pages have no counterpart.)
 *
 * Same operation and arguments as nvfp4_grouped_gemm_tiles with topk_weights given
 * (out = BF16 [T, N], out[t] = sum over the routes p of token t of
 * w[t, slot(p)] * y[p]), except that there is no workspace argument: the FP32
 * sums go to a fixed workspace inside the library, a device array of
 * nvfp4_noalloc_workspace_floats() floats (16 MiB) that every GPU loading
 * the library holds until the process exits.  It serves callers that cannot
 * allocate device memory at call time and have no workspace to lend: plugin
 * interfaces that hand a kernel only its inputs and outputs, and serving
 * loops that forbid the CUDA allocator after start-up (cudaMalloc may
 * synchronise the device and can fail under memory pressure).  The call
 * allocates and frees nothing.
 *
 *   - T * N must not exceed nvfp4_noalloc_workspace_floats(); larger shapes
 *     return NVFP4_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on a device looks up the workspace's device address
 *     (once per device, with that device current); make that first call
 *     before any stream capture.
 *   - Every call clears the part of the workspace it uses, then accumulates
 *     into it.  All calls on a device share the one workspace, so calls that
 *     overlap on the GPU (different streams without ordering between them)
 *     race and give wrong sums; serialise them.
 */
size_t nvfp4_noalloc_workspace_floats(void);

nvfp4_status nvfp4_grouped_gemm_combine_noalloc(const uint8_t* A_tiles, const float* gA,
                                                const uint8_t* W_tiles, const float* gW,
                                                const int32_t* expert_offsets, int32_t E,
                                                int64_t T, int32_t topk, int64_t N, int64_t K,
                                                const int32_t* route_token,
                                                const int32_t* route_slot,
                                                const float* topk_weights, void* out,
                                                void* stream);

/*
 * 2:4-sparse NVFP4 weights ("The FP4 Frontier", Finding 6: structured 2:4
 * sparsity halves the bits of an NVFP4 weight; the experts of an MoE model
 * can be pruned independently).  The unit of sparsity is the packed byte,
 * i.e. the pair of E2M1 values at K = 2i, 2i+1: in every aligned group of
 * four bytes (eight K elements) at most two bytes are non-zero.  Preparing
 * weights: nvfp4_prune_2of4 on the BF16 weights, nvfp4_quantize of the pruned
 * tensor (one global per expert, as for dense weights), then
 * nvfp4_prepack_sparse_weight_tiles; multiply with nvfp4_grouped_gemm_sparse.
 */

/*
 * Magnitude pruning of BF16 weights [rows, cols] (row stride ld elements) to
 * 2:4 over element pairs.  In each group of four pairs, pair i scores
 * |w[2i]| + |w[2i+1]| (one binary32 addition); the two highest scores stay,
 * equal scores favouring the lower position; the other two pairs are written
 * as +0.  out [rows, cols] (row stride ld_out) may be w itself (ld_out == ld).
 * cols, ld and ld_out % 8 == 0; both buffers 16-byte aligned.
 */
nvfp4_status nvfp4_prune_2of4(const void* w, int64_t rows, int64_t cols, int64_t ld, void* out,
                              int64_t ld_out, void* stream);

/* Bytes of the sparse operand tiles of rows x K weights:
 * ceil(rows / 128) x ceil(K / 256) tiles of 12288 bytes. */
size_t nvfp4_sparse_tiles_bytes(int64_t rows, int64_t K);

/*
 * Packed codes [rows, K/2] (2:4 over bytes) + row-major E4M3 scales
 * [rows, K/16] -> sparse operand tiles (nvfp4_sparse_tiles_bytes(rows, K)
 * bytes, caller-owned).  Tile (rt, kb) covers rows 128 rt .. 128 rt + 127 and
 * K 256 kb .. 256 kb + 255, at byte (rt * ceil(K / 256) + kb) * 12288:
 *   [0, 8192)       kept bytes: per group the two kept bytes in position
 *                   order; 64-K slice j of row r at j * 2048 + r * 16;
 *   [8192, 10240)   combination indices, 4 bits per group, numbering the
 *                   kept positions (i0 < i1) lexicographically: (0,1) (0,2)
 *                   (0,3) (1,2) (1,3) (2,3) -> 0..5; a group with fewer than
 *                   two non-zero bytes keeps the lowest zero positions; the 16
 *                   groups of 128-K half h of row r at 8192 + h * 1024 + r * 8,
 *                   group g in byte g / 2, low nibble for even g;
 *   [10240, 12288)  the scales as four 512-byte atoms, as in the dense tile.
 * Padding rows and K are zero.  A group with more than two non-zero bytes
 * sets NVFP4_ERR_DEVICE_CHECK in the device status word (the tile is then
 * not a faithful copy).  K % 64 == 0; packed and tiles 16-byte aligned,
 * scales 4-byte aligned.
 */
nvfp4_status nvfp4_prepack_sparse_weight_tiles(const uint8_t* packed,
                                               const uint8_t* scales_rowmajor, int64_t rows,
                                               int64_t K, uint8_t* tiles, void* stream);

/*
 * nvfp4_grouped_gemm_tiles over 2:4-sparse expert weights: the same operation,
 * arguments, orientations (route-ordered out or weighted combine), limits
 * and errors, with W_sparse_tiles = nvfp4_prepack_sparse_weight_tiles over
 * [E * N, K].  The result equals that of nvfp4_grouped_gemm_tiles on the dense
 * tiles of the same pruned weights: the kernel streams the sparse tiles (two
 * thirds of the dense bytes) and expands them in shared memory before the
 * block-scaled MMAs.
 */
nvfp4_status nvfp4_grouped_gemm_sparse(const uint8_t* A_tiles, const float* gA,
                                       const uint8_t* W_sparse_tiles, const float* gW,
                                       const int32_t* expert_offsets, int32_t E,
                                       int64_t T, int32_t topk, int64_t N, int64_t K,
                                       const int32_t* route_token, const int32_t* route_slot,
                                       const float* topk_weights,
                                       void* out, float* workspace, size_t workspace_bytes,
                                       void* stream);

/*
 * Decode attention over an NVFP4 KV cache ("The Blackwell architectural
 * split", The Breakthrough -- The A4Q Kernel, and Preserving precision --
 * dual-tier scale handling): the cache stays packed in memory and is expanded
 * on chip inside the attention loop.  One query token per sequence.  Groups of
 * 2, 4 or 8 query heads over heads of 128 and 256, of 2 or 4 over 512-wide
 * heads and of 4 or 8 over 64-wide heads run both contractions as tcgen05
 * MMAs on exact FP16 expansions of the cache (when both scale arrays are
 * 16-byte aligned, for heads of 64 and 128 L_max * D / 16 is a multiple of
 * 16, and B * Hkv * L_max < 2^31): one pipelined kernel for heads of 64 and
 * 128, a scores pass and a values pass for the wider heads.  Other shapes
 * multiply-add on the CUDA cores.  Both give the result defined below.
 *   q          BF16 [B, Hq, D].
 *   k_packed   NVFP4 codes [B, Hkv, L_max, D/2] (token rows of sequence b and
 *              KV head j contiguous), k_scales E4M3 [B, Hkv, L_max, D/16]
 *              (row-major, 16-element blocks along D), gk device float: the
 *              K cache's global.  nvfp4_quantize of the BF16 cache viewed as
 *              [B * Hkv * L_max, D] rows, with NVFP4_GLOBAL_GIVEN, writes
 *              exactly this layout.  v_packed, v_scales, gv likewise for V.
 *   seq_lens   int32 [B] (device): tokens of each sequence, 0 <= n <= L_max
 *              (others set NVFP4_ERR_DEVICE_CHECK and count as 0).
 *   scale      softmax scale (e.g. 1 / sqrt(D)).
 *   out        BF16 [B, Hq, D]: query head h reads KV head h / (Hq / Hkv);
 *              out = sum_t p_t v_hat_t, p = softmax over t < n of
 *              scale * q . k_hat_t, with k_hat = e2m1 * e4m3 * gk (likewise
 *              v_hat); FP32 arithmetic, BF16 round to nearest even; an empty
 *              sequence gives zeros.
 *   workspace  FP32, nvfp4_decode_attention_workspace_bytes(B, Hq, Hkv, L_max,
 *              D) bytes, caller-owned (per-split partials and, for heads of
 *              256 and 512, every cached token's score per query head;
 *              overwritten).
 * D in {64, 128, 256, 512}; Hq / Hkv in {1, 2, 4, 8} (at most 4 for D = 512);
 * q, out, workspace and the code arrays 16-byte aligned, the scale arrays
 * 4-byte aligned.  The tensor-core kernel's waits are bounded: a wait that
 * runs out records NVFP4_ERR_TIMEOUT in the device status word.
 */
size_t nvfp4_decode_attention_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int64_t L_max,
                                              int32_t D);

nvfp4_status nvfp4_decode_attention(const void* q, const uint8_t* k_packed,
                                    const uint8_t* k_scales, const float* gk,
                                    const uint8_t* v_packed, const uint8_t* v_scales,
                                    const float* gv, const int32_t* seq_lens, int32_t B,
                                    int32_t Hq, int32_t Hkv, int64_t L_max, int32_t D, float scale,
                                    void* out, float* workspace, size_t workspace_bytes,
                                    void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* NVFP4_GB300_H */
