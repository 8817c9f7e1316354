// NVFP4 block-scaled GEMM and MoE grouped GEMM on 5th-generation tensor cores.
//
// One persistent, warp-specialised kernel serves the single GEMM and the
// grouped GEMM ("The FP4 Frontier", Finding 5: a persistent grouped GEMM over
// all experts to avoid launch overhead; "The SM120 FP4 GEMM Kernel
// Investigation", The Comprehensive Synthesis: A/B FP4 tiles plus their
// scale-factor tiles staged through shared memory over several stages).
//
// Roles of the warps of a CTA (one CTA per SM; 224 threads for dense weights
// and token tiles up to 128 wide):
//   warp 0      TMA producer: operand tiles (128-byte swizzle) and scale
//               atoms into a ring of shared-memory stages;
//   warp 1      tensor-memory allocation; lane 0 issues tcgen05.cp (scales
//               -> tensor memory) and tcgen05.mma kind::mxf4nvf4 into a
//               double-buffered FP32 accumulator in tensor memory;
//   warp 6      second MMA issuer for narrow token tiles (odd K steps, own
//               accumulator): each tcgen05 instruction holds its issuing
//               thread for ~60-110 cycles, so one thread cannot issue the
//               12 instructions of a decode stage as fast as HBM delivers it;
//   warps 2-5   epilogue: tcgen05.ld, global-scale multiply, BF16 store or
//               weighted FP32 scatter-add (MoE combine);
//   warps 7-14  (2:4-sparse weights only) expansion of each stage's sparse
//               weight tiles into dense tiles in shared memory, with byte
//               permutes ("The FP4 Frontier", Finding 6: 2:4 sparsity halves
//               the weight bits; decode is bound by the weight bytes);
//   warp 15     (sparse 32-route units) scale warp.
// Wider tiles add a second epilogue group and a scale warp (see Cfg).
// A work unit is one 128-row tile of operand X (the MMA's M side) against up
// to BN rows of operand Y (the MMA's N side).  For the grouped GEMM, X is an
// expert's weights and Y its routed tokens, so a decode step streams every
// weight tile exactly once ("The FP4 Frontier", Finding 7: small-batch
// decode is bound by memory bandwidth).
//
// Every wait is bounded; on expiry the CTA records NVFP4_ERR_TIMEOUT, drains
// its own copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "kernels.h"
#include "format.cuh"

namespace nvfp4 {

namespace {

// 7 warps (11 for 256-wide tiles: Cfg::kThreads), roles below
constexpr int kRowBytes = 128;                 // 256 FP4 values = one swizzle row
constexpr int kBK = 256;                       // K elements per stage
constexpr int kXTileBytes = 128 * kRowBytes;   // 16 KB
constexpr int kSFStageBytes = 4 * 512;         // four scale atoms (K = 256)
constexpr int kTmemCols = 512;

// Pipeline configuration per token-tile width BN (rows of operand Y, the
// MMA's N).  Narrow tiles leave shared memory for more stages, i.e. more
// weight bytes in flight per SM, which is what the decode shapes need: each
// stage stays occupied for a memory round trip plus the tensor-pipe latency
// of its scale copies and MMAs.
template <int BN, int MT = 1, bool SP = false>
struct Cfg {
  static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 256, "tile width");
  // MT 128-row X tiles per unit (2 only for 32-row token tiles: two MMAs per
  // K step share the token operand, halving the units, the token re-reads
  // and the scale copies of Y per weight byte)
  // (64-row tiles with two X tiles serve the fused SiLU-mul epilogue and
  // sparse weights)
  // (128-row token tiles with two X tiles: the fused SiLU-mul epilogue of the
  // gate_up projection at wide token tiles)
  static_assert(MT == 1 || (MT == 2 && (BN == 32 || BN == 64 || (BN == 128 && !SP))),
                "unit height");
  // SP: X (the weights) arrives as 2:4-sparse tiles and is expanded in shared
  // memory by the decompression warps before the MMAs read it
  static_assert(!SP || (BN <= 128 && (MT == 1 || BN <= 64)),
                "sparse weights: token tiles <= 128, two X tiles only for 32/64-route tiles");
  static constexpr int kYTileBytes = BN * kRowBytes;
  static constexpr int kSfyAtomsPerStep = BN == 256 ? 2 : 1;   // 128-row scale atoms of Y
  // rows of one grouped operand tile / layout chunk: a 256-row token tile
  // spans two consecutive 128-row operand tiles
  static constexpr int kLayoutRows = BN < 128 ? BN : 128;
  static constexpr int kSfyStageBytes = kSfyAtomsPerStep * kSFStageBytes;
  // stage: [X part][Y codes][Y scales]; the X part has the operand-tile
  // layout (dense: codes 16 KB + scales 2 KB; sparse: kept bytes 8 KB +
  // combination indices 2 KB + scales 2 KB), so a tile K block lands with
  // one copy
  static constexpr int kXPartBytes = SP ? static_cast<int>(kSparseTileBytes)
                                        : kXTileBytes + kSFStageBytes;
  static constexpr int kXsfOffset = SP ? kSparseScaleOffset : kXTileBytes;  // X scales in the part
  static constexpr int kYOffset = MT * kXPartBytes;
  static constexpr int kStageBytes = kYOffset + kYTileBytes + kSfyStageBytes;
  static_assert(kYOffset % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle alignment");
  static constexpr int kStages = SP ? (MT == 2 ? (BN == 32 ? 4 : 3) : (BN == 32 ? 7 : (BN == 64 ? 6 : 5)))
                                    : MT == 2 ? (BN == 32 ? 5 : 4)
                                              : (BN == 32 ? 9 : (BN == 256 ? 4 : 6));
  // sparse: ring of expanded (dense) X code tiles, written by the
  // decompression warps, read by the MMAs.  A slot stays taken from its
  // expansion until the MMAs reading it complete (~4000 cycles at decode
  // rates, half of it the commit latency).  (Six slots for the one-tile
  // units of 64 and 128 routes, at the cost of compressed stages, measured
  // slightly slower than three.)
  static constexpr int kDStages = SP ? (BN == 32 && MT == 1 ? 4 : 3) : 0;   // slots of MT tiles
  static constexpr int kDecWarps = SP ? 8 : 0;
  // Stages are released to the producer in groups with one tcgen05.commit
  // per group.  One stage per group: a commit completes ~1000 cycles after it
  // is issued, and releasing stages one by one keeps more of the ring in
  // flight across that latency than saving the commits does.
  static constexpr int kGroup = 1;
  static constexpr int kGroups = kStages / kGroup;
  static_assert(kStages % kGroup == 0, "stage groups");
  // MMA-issuing warps: two for narrow tiles, except the fused two-tile units
  // of 64 routes, whose accumulators (gate and up) then fit twice in tensor
  // memory so the epilogue overlaps the next unit
  static constexpr int kIssuers = (BN <= 64 && !(MT == 2 && BN == 64)) ? 2 : 1;
  // With one MMA warp, warp 6 becomes a scale warp: it copies the stage's Y
  // scales (and for 128-wide tiles the X scales too) into tensor memory and
  // signals the MMA warp, so the two warps issue tcgen05 instructions in
  // parallel (each warp's issue rate, not the tensor pipe, bounds a stage).
  static constexpr bool kSplit = kIssuers == 1;
  // Sparse two-tile units: the two MMA warps issue only MMAs and commits; a
  // scale warp of its own (after the decompression warps) copies all of the
  // stage's scale atoms.
  // (64-route two-tile units have one MMA warp, so warp 6 is the scale warp)
  static constexpr bool kSpScaleWarp = SP && MT == 2 && !kSplit;
  static constexpr bool kScaleWarp = kSplit || kSpScaleWarp;
  static constexpr bool kXsfOnScaleWarp = kScaleWarp && (BN == 128 || MT == 2);
  // accumulator buffers: two (the epilogue of one tile overlaps the next
  // tile's MMAs), except for 256-wide tiles, whose one accumulator already
  // takes half of tensor memory
  // (and for the two 128-column accumulators of a 128-row two-tile unit)
  static constexpr int kAccBufs = (BN == 256 || (MT == 2 && BN == 128)) ? 1 : 2;
  static constexpr int kAccCols = BN;                  // one accumulator
  // Epilogue warp groups: 256-wide tiles hold their single accumulator until
  // the epilogue has read it, so a second group of four warps (warps 7-10)
  // takes the upper half of its columns and halves that wait.
  static constexpr int kEpiGroups = BN == 256 ? 2 : 1;
  // decompression warps (sparse) follow the epilogue warps: warps 7-14
  static constexpr int kDecWarp0 = 7 + 4 * (kEpiGroups - 1);
  static constexpr int kScaleWarpId = kSplit ? 6 : kDecWarp0 + kDecWarps;
  static constexpr int kThreads = (kDecWarp0 + kDecWarps + (kSpScaleWarp ? 1 : 0)) * 32;
  // accumulator (buffer b, X tile x, issuer j) at column ((b * MT + x) *
  // kIssuers + j) * BN; scale columns follow the accumulators: per stage 16
  // for each X tile, 16 or 32 for Y
  static constexpr int kSfColBase = kAccBufs * MT * kIssuers * BN;
  static constexpr int kSfyColsPerStep = 4 * kSfyAtomsPerStep;
  static constexpr int kSfColsPerStage = 16 * MT + 4 * kSfyColsPerStep;
  static_assert(kSfColBase + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
  static constexpr int kDenseOffset = kStages * kStageBytes;     // expanded X ring (sparse)
  // barriers: full[S], empty[S / G], acc_full[2], acc_empty[2], drain,
  // scales_ready[S] (split issue only), dense_ready[D] and dense_free[D]
  // (sparse only)
  static constexpr int kBarOffset = kDenseOffset + kDStages * MT * kXTileBytes;
  static constexpr int kBarBytes =
      8 * (kStages + kGroups + 5 + (kScaleWarp ? kStages : 0) + 2 * kDStages);
  static constexpr int kTableInts = 3 * (kGroupedMaxExperts + 1);
  static constexpr int kCtlOffset = kBarOffset + kBarBytes;
  // ring of per-unit token-row counts published by the producer (see below)
  static constexpr int kUnitRing = 16;
  static_assert(kUnitRing > kStages + 1, "unit ring depth");
  static constexpr int kRingOffset = kCtlOffset + 32;
  static constexpr int kTablesOffset = kRingOffset + 4 * kUnitRing;
  // combine epilogue: 512 bytes per epilogue warp, where its 32 features x 4
  // tokens of FP32 products are regrouped so that each reduction covers 16
  // bytes of four features and a warp's reduction four whole 128-byte rows
  static constexpr int kXchgOffset = (kTablesOffset + 4 * kTableInts + 15) & ~15;
  static constexpr int kXchgBytes = 512 * 4 * kEpiGroups;
  static constexpr int kSmemBytes = kXchgOffset + kXchgBytes + 1024;  // + align slack
  static_assert(kSmemBytes <= 232448 - 64, "shared memory budget");
};

struct Unit {
  int32_t x_row0;     // dense: tensor-map row of the X tile
  int32_t y_row0;     // dense: tensor-map row of the Y tile; grouped: first route
  int32_t y_rows;     // valid Y rows (1..BN)
  int32_t x_local0;   // first output feature (grouped) / first X row (dense)
  int32_t e;          // expert (grouped)
  int64_t sfx_off;    // dense: X scale atoms at k-block 0; grouped: X operand tile
  int64_t sfy_off;    // dense: Y scale atoms at k-block 0; grouped: Y operand tile
  int32_t x_reused;   // grouped: the expert has more than one token tile, so its
                      // weight tiles are read again by other units
  int32_t x_pair;     // grouped, MT == 2: row tiles from the first X tile to the second
  int32_t y_tile;     // grouped: first operand tile of the unit's token tile
  // per-unit phase of the fused MLP (the other modes: one phase, these are
  // the launch's own values)
  int32_t emode;      // epilogue mode of the unit
  int32_t k64;        // K / 64 of the unit's GEMM
  int32_t n_out;      // rows of each expert's X (output features)
  const uint8_t* xsrc;  // X operand tiles (or X scales)
  const uint8_t* ysrc;  // Y operand tiles (or Y scales)
  const float* gxp;     // X globals
};

struct Tables {
  int32_t* up;        // [E+1] unit prefix
  int32_t* off;       // [E+1] expert offsets
  int32_t* tb;        // [E+1] scale-tile prefix
};

template <int BN, int MT, bool SP = false>
__device__ __forceinline__ Unit get_unit(int u, int mode, const GemmArgs& a, const Tables& t,
                                         int tiles_x, int64_t atoms_per_rowtile) {
  Unit un;
  un.emode = mode;
  un.k64 = static_cast<int32_t>(a.K >> 6);
  un.n_out = a.n_out;
  un.xsrc = a.sfx;
  un.ysrc = a.sfy;
  un.gxp = a.gx;
  if (mode == kMlpFused && u >= t.up[a.E]) {
    // down projection unit: token tile tt (every expert's token tiles in
    // order), X tiles m and m + 1 of the expert's down weight, Y = h tiles
    const int munits1 = (a.n_out >> 7) / 2;       // gate_up units per token tile
    const int mtiles2 = a.n_out2 >> 7;
    const int munits2 = mtiles2 / MT;
    const int u2 = u - t.up[a.E];
    const int tt = u2 / munits2;
    const int mt = (u2 % munits2) * MT;
    int lo = 0, hi = a.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (t.up[mid] <= tt * munits1) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int nt = tt - t.up[e] / munits1;
    const int cnt = t.off[e + 1] - t.off[e];
    const int64_t n_kb2 = (a.K2 + kBK - 1) / kBK;
    un.emode = kGroupedCombine;
    un.k64 = static_cast<int32_t>(a.K2 >> 6);
    un.n_out = a.n_out2;
    un.xsrc = a.sfx2;
    un.ysrc = a.h_tiles;
    un.gxp = a.gx2;
    un.e = e;
    un.x_row0 = e * a.n_out2 + mt * 128;
    un.x_local0 = mt * 128;
    un.y_row0 = t.off[e] + nt * BN;
    un.y_rows = min(BN, cnt - nt * BN);
    un.sfx_off = static_cast<int64_t>(e * mtiles2 + mt) * n_kb2 * kOperandTileBytes;
    un.y_tile = tt;
    un.sfy_off = static_cast<int64_t>(tt) * n_kb2 * kOperandTileBytes;
    un.x_reused = cnt > BN;
    un.x_pair = 1;
    return un;
  }
  if (mode == kGrouped || mode == kGroupedCombine || mode == kGroupedSiluMul ||
      mode == kGroupedSiluBf16 || mode == kMlpFused) {
    if (mode == kMlpFused) un.emode = kGroupedSiluMul;
    int lo = 0, hi = a.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (t.up[mid] <= u) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int mtiles = a.n_out >> 7;
    const int munits = mtiles / MT;               // units per token tile
    const int local = u - t.up[e];
    // SiLU-mul: X tile m (gate rows) pairs with X tile m + mtiles / 2 (the
    // up rows of the same features); otherwise a unit's X tiles are adjacent
    const bool glu = mode == kGroupedSiluMul || mode == kGroupedSiluBf16 || mode == kMlpFused;
    const int mt = glu ? (local % munits) : (local % munits) * MT;   // first X tile
    const int nt = local / munits;
    const int cnt = t.off[e + 1] - t.off[e];
    un.e = e;
    un.x_row0 = e * a.n_out + mt * 128;
    un.x_local0 = mt * 128;
    un.y_row0 = t.off[e] + nt * BN;
    un.y_rows = min(BN, cnt - nt * BN);
    const int64_t n_kb = (a.K + kBK - 1) / kBK;
    // X from operand tiles: the unit's first tile; X from the tensor map: its
    // row tile's scale atoms (the codes come by TMA at row x_row0)
    un.sfx_off = a.x_map ? static_cast<int64_t>(e * mtiles + mt) * atoms_per_rowtile * 512
                         : static_cast<int64_t>(e * mtiles + mt) * n_kb *
                               (SP ? kSparseTileBytes : kOperandTileBytes);
    un.y_tile = t.tb[e] + nt * (BN / Cfg<BN, MT>::kLayoutRows);
    un.sfy_off = static_cast<int64_t>(un.y_tile) * n_kb * kOperandTileBytes;
    un.x_reused = cnt > BN;
    un.x_pair = glu ? mtiles / 2 : 1;
  } else {
    const int tx = u % tiles_x;
    const int ty = u / tiles_x;
    un.e = 0;
    un.x_row0 = tx * 128;
    un.x_local0 = tx * 128;
    un.y_row0 = ty * BN;
    un.y_rows = min(BN, a.rows_y - ty * BN);
    un.sfx_off = static_cast<int64_t>(tx) * atoms_per_rowtile * 512;
    un.sfy_off = static_cast<int64_t>(ty * (BN / 128)) * atoms_per_rowtile * 512;
    un.x_reused = 1;
    un.x_pair = 1;
    un.y_tile = 0;
  }
  return un;
}

// In-register transpose of a 32 x 32 block held by one warp: lane l's r[i]
// becomes the value lane i held in r[l].  Five butterfly stages; every
// register index is a compile-time constant, so r stays in registers.
__device__ __forceinline__ void warp_transpose32(uint32_t (&r)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & s) == 0) {
        const uint32_t send = upper ? r[i] : r[i + s];
        const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, s);
        if (upper) r[i] = recv; else r[i + s] = recv;
      }
    }
  }
}

// ---------------------------------------------------------------- 2:4 sparse
// A sparse weight group is four packed bytes (eight K elements) of which two
// are kept; its 4-bit combination index c numbers the kept positions
// (i0 < i1) in lexicographic order: (0,1) (0,2) (0,3) (1,2) (1,3) (2,3).
// Expanding a group is one byte permute of the word holding its two kept
// bytes (in bytes 0 and 1) and a zero word: output byte p takes byte 0 if
// p == i0, byte 1 if p == i1, else byte 4 (zero).  sp_selector(c) is that
// 16-bit permute selector; indices 6 and 7 never occur (all-zero selector).
__host__ __device__ constexpr uint32_t sp_selector(int c) {
  int i0 = 0, i1 = 1, n = 0;
  for (int x = 0; x < 4; ++x)
    for (int y = x + 1; y < 4; ++y) {
      if (n == c) { i0 = x; i1 = y; }
      ++n;
    }
  if (c >= 6) return 0x4444u;
  uint32_t sel = 0;
  for (int p = 0; p < 4; ++p) sel |= (p == i0 ? 0u : (p == i1 ? 1u : 4u)) << (4 * p);
  return sel;
}
// Byte-permute lookup tables: byte b of word (lo, 0) / (lo, 1) is the low
// selector byte of combination b / 4 + b, likewise (hi, *) the high byte, so
// one permute turns four combination nibbles into four selector bytes.
__host__ __device__ constexpr uint32_t sp_table(int hi, int upper) {
  uint32_t w = 0;
  for (int b = 0; b < 4; ++b) w |= ((sp_selector(4 * upper + b) >> (8 * hi)) & 0xFFu) << (8 * b);
  return w;
}

// Expands K elements 128h .. 128h + 127 of row r of one sparse X tile at
// `sp` (shared memory, the sparse tile layout: kept bytes of 64-K slice j of
// row r at j * 2048 + r * 16, combination nibbles of 128-K half h at 8192 +
// h * 1024 + r * 8) into the dense code tile at `dn` (row r at r * 128,
// 16-byte chunk c at position c ^ (r % 8)): four 16-byte chunks.
__device__ __forceinline__ void sp_expand_row_half(const uint8_t* sp, uint8_t* dn, int r, int h) {
  constexpr uint32_t kLoA = sp_table(0, 0), kLoB = sp_table(0, 1);
  constexpr uint32_t kHiA = sp_table(1, 0), kHiB = sp_table(1, 1);
  const uint4 k0 = *reinterpret_cast<const uint4*>(sp + (2 * h) * 2048 + r * 16);
  const uint4 k1 = *reinterpret_cast<const uint4*>(sp + (2 * h + 1) * 2048 + r * 16);
  const uint2 m = *reinterpret_cast<const uint2*>(sp + kSparseComboOffset + h * 1024 + r * 8);
  // word k holds the kept bytes of groups 2k and 2k + 1 of the half
  const uint32_t w[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {                  // dense chunk 4h + q: groups 4q .. 4q + 3
    const uint32_t mw = q < 2 ? m.x : m.y;
    const uint32_t m16 = (q & 1) ? (mw >> 16) : mw;   // the permutes read 16 selector bits
    const uint32_t lo = __byte_perm(kLoA, kLoB, m16);
    const uint32_t hi = __byte_perm(kHiA, kHiB, m16);
    const uint32_t s01 = __byte_perm(lo, hi, 0x5140);  // selectors of groups 4q, 4q + 1
    const uint32_t s23 = __byte_perm(lo, hi, 0x7362);  // groups 4q + 2, 4q + 3
    uint4 d;
    d.x = __byte_perm(w[2 * q], 0u, s01);
    d.y = __byte_perm(w[2 * q] >> 16, 0u, s01 >> 16);
    d.z = __byte_perm(w[2 * q + 1], 0u, s23);
    d.w = __byte_perm(w[2 * q + 1] >> 16, 0u, s23 >> 16);
    const int c = 4 * h + q;
    *reinterpret_cast<uint4*>(dn + r * kRowBytes + ((c ^ (r & 7)) << 4)) = d;
  }
}

// Four FP32 additions into global memory in one reduction (16-byte aligned).
__device__ __forceinline__ void red_add_v4(float* dst, float4 v) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
               :: "l"(dst), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}

// Generic-proxy global accesses of this thread ordered with its async-proxy
// (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Adds 1 to a counter in global memory with release semantics at GPU scope.
__device__ __forceinline__ void red_release_add1(uint32_t* p) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(p) : "memory");
}

// Waits (acquire at GPU scope) until *p >= target.  Gives up when the CTA
// has aborted or after the time limit, recording NVFP4_ERR_TIMEOUT.
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t target, CtaCtl* ctl,
                                           int* status) {
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 0; i < 0x7FFFFFFFu; ++i) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if (*reinterpret_cast<volatile uint32_t*>(&ctl->abort)) return false;
    if (globaltimer() - t0 > ctl->timeout_ns) {
      *reinterpret_cast<volatile uint32_t*>(&ctl->abort) = 1u;
      raise_status(status, NVFP4_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  *reinterpret_cast<volatile uint32_t*>(&ctl->abort) = 1u;
  raise_status(status, NVFP4_ERR_TIMEOUT);
  return false;
}

// Waits for a phase regardless of the abort flag (used only to drain copies
// and MMAs already in flight); bounded by the timeout.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1; i < 0x7FFFFFFFu; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0 && globaltimer() - t0 > timeout) return false;
  }
  return false;
}

template <int BN, int MT, bool SP>
__global__ void __launch_bounds__(Cfg<BN, MT, SP>::kThreads, 1)
nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                  const GemmArgs a, int mode) {
  using C = Cfg<BN, MT, SP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kBarOffset;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int g) { return bar0 + 8u * (C::kStages + g); };   // per stage group
  auto accf_bar = [&](int b) { return bar0 + 8u * (C::kStages + C::kGroups + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (C::kStages + C::kGroups + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (C::kStages + C::kGroups + 4);
  auto sfr_bar = [&](int s) { return bar0 + 8u * (C::kStages + C::kGroups + 5 + s); };
  // sparse: an expanded X tile is ready for the MMAs / free for the next expansion
  constexpr int kDBar0 = C::kStages + C::kGroups + 5 + (C::kScaleWarp ? C::kStages : 0);
  auto dready_bar = [&](int d) { return bar0 + 8u * (kDBar0 + d); };
  auto dfree_bar = [&](int d) { return bar0 + 8u * (kDBar0 + C::kDStages + d); };
  CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + C::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kCtlOffset + 16);
  int32_t* tab = reinterpret_cast<int32_t*>(smem + C::kTablesOffset);
  // The producer decodes every unit anyway; it publishes the unit's token-row
  // count here before arriving on the unit's first full barrier, and the MMA
  // issuers read it after waiting on that barrier, which keeps the unit
  // decoding (binary search, divisions) off their critical path.  The
  // producer runs at most kStages stages ahead, so a slot is never rewritten
  // before it is read.
  volatile int32_t* unit_rows = reinterpret_cast<volatile int32_t*>(smem + C::kRingOffset);
  Tables t{tab, tab + (kGroupedMaxExperts + 1), tab + 2 * (kGroupedMaxExperts + 1)};
  __shared__ int32_t s_units;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool grouped = (mode == kGrouped || mode == kGroupedCombine || mode == kGroupedSiluMul ||
                        mode == kGroupedSiluBf16 || mode == kMlpFused);
  const int64_t atoms_per_rowtile = a.K >> 6;
  // K / 64 of unit u: the fused MLP's down units (u at or past the gate_up
  // units) have the down projection's depth
  auto unit_k64 = [&](int u) {
    return static_cast<int>(((mode == kMlpFused && u >= t.up[a.E]) ? a.K2 : a.K) >> 6);
  };
  const int tiles_x = (a.rows_x + 127) >> 7;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) mbar_init(full_bar(s), 1);
    for (int g = 0; g < C::kGroups; ++g) mbar_init(empty_bar(g), C::kIssuers);
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), C::kIssuers);
      mbar_init(acce_bar(b), 128 * C::kEpiGroups);
    }
    mbar_init(drain_bar, C::kIssuers + (C::kScaleWarp ? 1 : 0));
    if (C::kScaleWarp)
      for (int s = 0; s < C::kStages; ++s) mbar_init(sfr_bar(s), 1);
    for (int d = 0; d < C::kDStages; ++d) {
      mbar_init(dready_bar(d), C::kDecWarps);
      mbar_init(dfree_bar(d), C::kIssuers);
    }

    ctl->abort = 0;
    ctl->timeout_ns = a.timeout_ns;
    fence_mbar_init();
  }
  // Work list.  Grouped: per-expert unit and scale-tile prefixes, built by
  // warp 2 from the device-side offsets (validated: monotone, within R).
  if (grouped) {
    if (warp == 2) {
      const int E = a.E;
      const int per = (E + 31) / 32;
      const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
      const int mtiles = (a.n_out >> 7) / MT;       // units per token tile
      // the offsets arrive with coalesced loads (all in flight at once);
      // the scan below reads them from shared memory
#pragma unroll 4
      for (int i = lane; i <= E; i += 32) t.off[i] = a.expert_offsets[i];
      __syncwarp();
      int32_t su = 0, st = 0;
      bool ok = true;
      for (int e = e0; e < e1; ++e) {
        const int32_t c = t.off[e + 1] - t.off[e];
        ok = ok && (c >= 0);
        su += mtiles * ((c + BN - 1) / BN);
        st += (c + C::kLayoutRows - 1) / C::kLayoutRows;
      }
      int32_t iu = su, it = st;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t vu = __shfl_up_sync(0xFFFFFFFFu, iu, o);
        const int32_t vt = __shfl_up_sync(0xFFFFFFFFu, it, o);
        if (lane >= o) { iu += vu; it += vt; }
      }
      int32_t pu = iu - su, pt = it - st;
      for (int e = e0; e < e1; ++e) {
        const int32_t c = t.off[e + 1] - t.off[e];
        t.up[e] = pu; t.tb[e] = pt;
        pu += mtiles * ((c + BN - 1) / BN);
        pt += (c + C::kLayoutRows - 1) / C::kLayoutRows;
      }
      const bool all_ok = __all_sync(0xFFFFFFFFu, ok);
      if (lane == 31) {
        const int32_t oE = t.off[E];
        t.up[E] = iu;
        t.tb[E] = it;
        const bool good = all_ok && t.off[0] == 0 && oE <= a.rows_y;
        if (!good) raise_status(a.status, NVFP4_ERR_DEVICE_CHECK);
        // fused MLP: the down units follow, munits2 per token tile
        const int32_t all = mode == kMlpFused
                                ? iu + iu / ((a.n_out >> 7) / 2) * ((a.n_out2 >> 7) / MT)
                                : iu;
        s_units = good ? all : 0;
      }
    }
  } else if (threadIdx.x == 0) {
    s_units = tiles_x * ((a.rows_y + BN - 1) / BN);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int units = s_units;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (uniform control flow); one elected lane
    // issues each copy, as in the MMA warp.
    // Weights read by a single unit stream through L2 (evict first); weights
    // that other token tiles of the same expert read again stay (normal).
    const uint64_t pol_once = l2_policy_evict_first();
    const uint64_t pol_again = grouped ? l2_policy_evict_normal() : l2_policy_evict_last();
    const uint64_t pol_y = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool alive = true;
    int uidx = 0;
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x, ++uidx) {
      const Unit un = get_unit<BN, MT, SP>(u, mode, a, t, tiles_x, atoms_per_rowtile);
      if (lane == 0) unit_rows[uidx & (C::kUnitRing - 1)] = un.y_rows;
      __syncwarp();
      const uint64_t pol_x = un.x_reused ? pol_again : pol_once;
      const int ybox = (un.y_rows + 15) >> 4;                  // 16-row groups
      const int ny_loads = (un.y_rows + a.ybox_rows - 1) / a.ybox_rows;
      const int k64 = unit_k64(u);
      const int nkb = (k64 + 3) >> 2;
      if (mode == kMlpFused && un.emode == kGroupedCombine) {
        // a down unit reads h of its token tile: wait until every gate_up
        // unit of that token tile has written its features (bounded), then
        // order those generic-proxy stores before this warp's bulk copies
        bool ok = true;
        if (lane == 0)
          ok = wait_count(a.ready + un.y_tile, static_cast<uint32_t>((a.n_out >> 7) / 2) * 4u,
                          ctl, a.status);
        if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) {
          alive = false;
          break;
        }
        fence_proxy_async_global();
      }
      for (int kb = 0; kb < nkb; ++kb) {
        // a group of stages is refilled once the MMAs of its previous round completed
        if (stage % C::kGroup == 0 &&
            !__all_sync(0xFFFFFFFFu, mbar_wait(empty_bar(stage / C::kGroup), phase ^ 1u, ctl,
                                               a.status))) {
          alive = false;
          break;
        }
        const int ksteps = min(4, k64 - 4 * kb);
        const uint32_t sx = sbase + stage * C::kStageBytes;
        const uint32_t ssfx = sx + kXTileBytes;
        const uint32_t sy = sx + C::kYOffset;
        const uint32_t ssfy = sy + C::kYTileBytes;
        if ((a.debug_flags & kDebugSkipFirstStage) && issued == 0 && stage == 0 && kb == 0 &&
            u == static_cast<int>(blockIdx.x)) {
          // test hook: leave stage 0 empty; its consumers' bounded waits expire.
          // Counted as issued so the drain below keeps stage numbers aligned
          // (its wait on this stage ends by the time limit too).
          ++issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
          continue;
        }
        const uint32_t ybytes = grouped ? ybox * 16 * kRowBytes : ny_loads * a.ybox_rows * kRowBytes;
        // the second 128-row scale group of a 256-wide Y tile exists only when
        // the tile has more than 128 rows
        const int sfy_groups = (C::kSfyAtomsPerStep == 2 && un.y_rows > 128) ? 2 : 1;
        // grouped 256-row tiles: codes of rows 0-127 and 128+ come from two tiles
        const int ybox_lo = min(ybox, 8), ybox_hi = ybox - ybox_lo;
        // X part: codes (dense) or kept bytes + combination indices (sparse),
        // then the scale atoms of the block's K steps
        const uint32_t xbytes = C::kXsfOffset + ksteps * 512;
        const uint32_t bytes = MT * xbytes + ybytes + sfy_groups * ksteps * 512;
        mbar_arrive_expect_tx_elect(full_bar(stage), bytes);
        if (grouped) {
          // operand tiles: X codes + scales in one contiguous copy, Y codes
          // (only the unit's rows) and Y scales in two more
          const uint8_t* yt = un.ysrc + un.sfy_off + kb * kOperandTileBytes;
          if (!SP && a.x_map) {
            // X as row-major codes (TMA, 128-byte swizzle: the layout the
            // operand tiles store) and atom-layout scales (one bulk copy)
            for (int x = 0; x < MT; ++x) {
              const int xo = x * un.x_pair;            // row tiles to the unit's tile x
              tma_load_2d_elect(sx + x * C::kXPartBytes, &tmx, full_bar(stage), kb * kRowBytes,
                                un.x_row0 + 128 * xo, pol_x);
              bulk_load_elect(sx + x * C::kXPartBytes + kXTileBytes,
                              a.sfx + un.sfx_off + xo * atoms_per_rowtile * 512 +
                                  kb * kSFStageBytes,
                              ksteps * 512, full_bar(stage), pol_x);
            }
          } else {
            const uint8_t* xt =
                un.xsrc + un.sfx_off + kb * (SP ? kSparseTileBytes : kOperandTileBytes);
            bulk_load_elect(sx, xt, xbytes, full_bar(stage), pol_x);
            if (MT == 2)                 // the unit's second weight tile
              bulk_load_elect(sx + C::kXPartBytes,
                              xt + static_cast<int64_t>(un.x_pair) * nkb *
                                       (SP ? kSparseTileBytes : kOperandTileBytes),
                              xbytes, full_bar(stage), pol_x);
          }
          bulk_load_elect(sy, yt, ybox_lo * 16 * kRowBytes, full_bar(stage), pol_y);
          bulk_load_elect(ssfy, yt + kXTileBytes, ksteps * 512, full_bar(stage), pol_y);
          if (ybox_hi > 0) {               // second operand tile of a 256-row token tile
            const uint8_t* yt2 = yt + static_cast<int64_t>(nkb) * kOperandTileBytes;
            bulk_load_elect(sy + 128 * kRowBytes, yt2, ybox_hi * 16 * kRowBytes, full_bar(stage),
                            pol_y);
            bulk_load_elect(ssfy + kSFStageBytes, yt2 + kXTileBytes, ksteps * 512, full_bar(stage),
                            pol_y);
          }
        } else {
          tma_load_2d_elect(sx, &tmx, full_bar(stage), kb * kRowBytes, un.x_row0, pol_x);
          for (int j = 0; j < ny_loads; ++j)
            tma_load_2d_elect(sy + j * a.ybox_rows * kRowBytes, &tmy, full_bar(stage),
                              kb * kRowBytes, un.y_row0 + a.ybox_rows * j, pol_y);
          bulk_load_elect(ssfx, a.sfx + un.sfx_off + kb * kSFStageBytes, ksteps * 512,
                          full_bar(stage), pol_x);
          bulk_load_elect(ssfy, a.sfy + un.sfy_off + kb * kSFStageBytes, ksteps * 512,
                          full_bar(stage), pol_y);
          if (sfy_groups == 2)
            bulk_load_elect(ssfy + kSFStageBytes,
                            a.sfy + un.sfy_off + atoms_per_rowtile * 512 + kb * kSFStageBytes,
                            ksteps * 512, full_bar(stage), pol_y);
        }
        ++issued;
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
    }
    // Drain: every copy this warp issued must land before the CTA exits.
    if (lane == 0) {
      const int64_t first = issued > C::kStages ? issued - C::kStages : 0;
      for (int64_t n = first; n < issued; ++n)
        mbar_wait_drain(full_bar(static_cast<int>(n % C::kStages)),
                        static_cast<uint32_t>((n / C::kStages) & 1), ctl->timeout_ns);
    }
    __syncwarp();
  } else if (C::kScaleWarp && warp == C::kScaleWarpId) {
    // ---------------------------------------------------------- scale warp
    // Copies each stage's Y scale atoms (and X's for 128-wide tiles) into the
    // stage's tensor-memory columns once the stage has landed, then arrives
    // on the stage's scales-ready barrier, on which the MMA warp waits.  A
    // stage's columns are rewritten only after its refill, which follows the
    // completion of the MMAs that read them.
    int stage = 0;
    uint32_t phase = 0;
    bool alive = true;
    int uidx = 0;
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x, ++uidx) {
      int y_rows = 0;
      const int k64 = unit_k64(u);
      const int nkb = (k64 + 3) >> 2;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_bar(stage), phase, ctl, a.status))) {
          alive = false;
          break;
        }
        if (kb == 0) y_rows = unit_rows[uidx & (C::kUnitRing - 1)];
        const int ksteps = min(4, k64 - 4 * kb);
        const uint32_t sx = sbase + stage * C::kStageBytes;
        const uint32_t ssfx = sx + C::kXsfOffset;
        const uint32_t ssfy = sx + C::kYOffset + C::kYTileBytes;
        const uint32_t tsfx = tmem + C::kSfColBase + stage * C::kSfColsPerStage;
        const uint32_t tsfy = tsfx + 16 * MT;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (C::kXsfOnScaleWarp) {
            tc_cp_sf_atom_elect(tsfx + 4 * ks, sdesc_sf_atom(ssfx + 512 * ks));
            if (MT == 2)                 // the unit's second X tile
              tc_cp_sf_atom_elect(tsfx + 16 + 4 * ks,
                                  sdesc_sf_atom(ssfx + C::kXPartBytes + 512 * ks));
          }
          tc_cp_sf_atom_elect(tsfy + C::kSfyColsPerStep * ks, sdesc_sf_atom(ssfy + 512 * ks));
          if (C::kSfyAtomsPerStep == 2 && y_rows > 128)
            tc_cp_sf_atom_elect(tsfy + C::kSfyColsPerStep * ks + 4,
                                sdesc_sf_atom(ssfy + kSFStageBytes + 512 * ks));
        }
        // The MMA warp issues after this arrive and its after-sync fence, and
        // copies followed by MMAs that read their columns execute in that
        // order, so no commit (and its completion latency) is needed here.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfr_bar(stage));
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
    }
    tc_commit_elect(drain_bar);
    if (lane == 0) mbar_wait_drain(drain_bar, 0, ctl->timeout_ns);
    __syncwarp();
  } else if (warp == 1 || (C::kIssuers == 2 && warp == 6)) {
    // ---------------------------------------------------------------- MMA
    // Issuer j takes the K steps with ks % kIssuers == j of every stage.  The
    // whole warp runs the loop (every lane waits on the barriers, so the
    // control flow stays converged and uniform); one elected lane issues each
    // tcgen05 instruction.
    const int j = (warp == 6) ? 1 : 0;
    int stage = 0;
    uint32_t phase = 0;
    int dstage = 0;                     // sparse: expanded X tile ring
    uint32_t dphase = 0;
    int abuf = 0;
    uint32_t aphase = 0;
    bool alive = true;
    int uidx = 0;
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x, ++uidx) {
      int y_rows = 0;
      uint32_t idesc = 0;
      const int k64 = unit_k64(u);
      const int nkb = (k64 + 3) >> 2;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(acce_bar(abuf), aphase ^ 1u, ctl, a.status))) break;
      tc_fence_after();
      // accumulator of X tile x: column ((abuf * MT + x) * kIssuers + j) * BN
      const uint32_t d_tmem = tmem + (abuf * MT * C::kIssuers + j) * C::kAccCols;
      for (int kb = 0; kb < nkb; ++kb) {
        // The stage's operands arrive by TMA / bulk copy, completing on the
        // mbarrier; the MMAs read them through the same async proxy, so the
        // wait alone orders them.  (A tcgen05 thread-sync fence here would
        // wait for this thread's earlier MMAs and serialise the stages.)
        // split issue: the scales-ready barrier completes after the stage
        // landed (the scale warp waited for it) and its scale copies were
        // issued; the fence orders these MMAs after those copies
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(C::kScaleWarp ? sfr_bar(stage) : full_bar(stage),
                                               phase, ctl, a.status))) {
          alive = false;
          break;
        }
        // sparse: the decompression warps expanded this stage's X tile (they
        // waited for the stage too; their proxy fence orders their writes
        // before these MMAs' operand reads)
        if (SP && !__all_sync(0xFFFFFFFFu, mbar_wait(dready_bar(dstage), dphase, ctl, a.status))) {
          alive = false;
          break;
        }
        if (C::kScaleWarp) tc_fence_after();
        if (kb == 0) {
          y_rows = unit_rows[uidx & (C::kUnitRing - 1)];
          idesc = idesc_nvf4(static_cast<uint32_t>((y_rows + 15) & ~15));
        }
        const int ksteps = min(4, k64 - 4 * kb);
        const uint32_t sx = sbase + stage * C::kStageBytes;
        const uint32_t ssfx = sx + C::kXsfOffset;
        const uint32_t sy = sx + C::kYOffset;
        const uint32_t ssfy = sy + C::kYTileBytes;
        const uint32_t tsfx = tmem + C::kSfColBase + stage * C::kSfColsPerStage;
        const uint32_t tsfy = tsfx + 16 * MT;
        // X tile x: the stage's dense X part, or slot x of the expanded ring
        const uint32_t sx_tile0 = SP ? sbase + C::kDenseOffset + dstage * MT * kXTileBytes : sx;
        const uint32_t x_tile_step = SP ? kXTileBytes : C::kXPartBytes;
        const uint64_t dx = sdesc_sw128(sx_tile0);
        const uint64_t dy = sdesc_sw128(sy);
        // Every token tile starts at row 0 of its operand tile, so every
        // scale address handed to the MMA is a multiple of 4 columns (an
        // address inside an atom's column group faults as misaligned).
        for (int ks = j; ks < ksteps; ks += C::kIssuers) {
          const uint32_t tsfy_ks = tsfy + C::kSfyColsPerStep * ks;
          if (!C::kXsfOnScaleWarp)
            tc_cp_sf_atom_elect(tsfx + 4 * ks, sdesc_sf_atom(ssfx + 512 * ks));
          if (!C::kScaleWarp) {
            tc_cp_sf_atom_elect(tsfy_ks, sdesc_sf_atom(ssfy + 512 * ks));
            // rows 128-255 of a 256-wide Y tile: the next 4 columns (the MMA
            // reads the scales of row n from column base + n / 32)
            if (C::kSfyAtomsPerStep == 2 && y_rows > 128)
              tc_cp_sf_atom_elect(tsfy_ks + 4, sdesc_sf_atom(ssfy + kSFStageBytes + 512 * ks));
          }
          tc_mma_nvf4_elect(d_tmem, dx + 2 * ks, dy + 2 * ks, idesc, tsfx + 4 * ks, tsfy_ks,
                            (kb > 0 || ks >= C::kIssuers) ? 1u : 0u);
          if (MT == 2) {                 // second weight tile, same token operand
            if (!C::kXsfOnScaleWarp)
              tc_cp_sf_atom_elect(tsfx + 16 + 4 * ks,
                                  sdesc_sf_atom(ssfx + C::kXPartBytes + 512 * ks));
            tc_mma_nvf4_elect(d_tmem + C::kIssuers * C::kAccCols,
                              sdesc_sw128(sx_tile0 + x_tile_step) + 2 * ks, dy + 2 * ks, idesc,
                              tsfx + 16 + 4 * ks, tsfy_ks,
                              (kb > 0 || ks >= C::kIssuers) ? 1u : 0u);
          }
        }
        if (stage % C::kGroup == C::kGroup - 1) tc_commit_elect(empty_bar(stage / C::kGroup));
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        if (SP) {                        // the expanded tile is free once these MMAs complete
          tc_commit_elect(dfree_bar(dstage));
          if (++dstage == C::kDStages) { dstage = 0; dphase ^= 1u; }
        }
      }
      if (!alive) break;
      tc_commit_elect(accf_bar(abuf));
      if (++abuf == C::kAccBufs) { abuf = 0; aphase ^= 1u; }
    }
    // Drain: wait for every MMA and copy issued above before teardown.
    tc_commit_elect(drain_bar);
    if (lane == 0) mbar_wait_drain(drain_bar, 0, ctl->timeout_ns);
    __syncwarp();
  } else if (SP && warp >= C::kDecWarp0) {
    // ------------------------------------------------------- decompression
    // Eight warps; thread (row r, half h) expands K elements 128h .. 128h +
    // 127 of row r of each of the stage's MT sparse X tiles into the next
    // free slot of the expanded ring, then the warp hands the slot to the MMA
    // warps.  (Spreading the stage's scale copies over these warps instead
    // was measured slower: tcgen05 work issued from ten warps backed up the
    // tensor pipe.)
    static_assert(!SP || C::kDecWarps == 8, "one thread per row half");
    const int dt = threadIdx.x - C::kDecWarp0 * 32;
    const int r = dt & 127, h = dt >> 7;
    int stage = 0, dstage = 0;
    uint32_t phase = 0, dphase = 0;
    bool alive = true;
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
      const int nkb = (unit_k64(u) + 3) >> 2;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_bar(stage), phase, ctl, a.status)) ||
            !__all_sync(0xFFFFFFFFu,
                        mbar_wait(dfree_bar(dstage), dphase ^ 1u, ctl, a.status))) {
          alive = false;
          break;
        }
#pragma unroll
        for (int x = 0; x < MT; ++x)
          sp_expand_row_half(smem + stage * C::kStageBytes + x * C::kXPartBytes,
                             smem + C::kDenseOffset + (dstage * MT + x) * kXTileBytes, r, h);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(dready_bar(dstage));
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        if (++dstage == C::kDStages) { dstage = 0; dphase ^= 1u; }
      }
    }
  } else if ((warp >= 2 && warp <= 5) || (C::kEpiGroups == 2 && warp >= 7)) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // tensor-memory lane quarter
    // columns of the accumulator this warp's group reads
    const int grp = warp >= 7 ? 1 : 0;
    constexpr int kGrpCols = BN / C::kEpiGroups;
    const int gc0 = grp * kGrpCols;
    const int row = q * 32 + lane;                // row of the X tile
    int abuf = 0;
    uint32_t aphase = 0;
    const float gy = *a.gy;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit un = get_unit<BN, MT, SP>(u, mode, a, t, tiles_x, atoms_per_rowtile);
      const int emode = un.emode;
      // accumulators that received at least one K step (issuer j's first is ks = j)
      const int n_acc = un.k64 < C::kIssuers ? un.k64 : C::kIssuers;
      // the fused MLP's down units scale by the global of h
      const float gy_u = (mode == kMlpFused && emode == kGroupedCombine) ? *a.g_h : gy;
      // Combine: fetch this lane's tokens and routing weights (one token per
      // lane per 32-column chunk) before waiting, so the dependent L2 round
      // trips overlap the MMAs instead of following them.  A token outside
      // [0, T) or a slot outside [0, topk) is a device-side input error: the
      // route is skipped (c_tok = -1) and the status word records it.
      int c_tok[BN / 32];
      float c_w[BN / 32];
      if (emode == kGroupedCombine) {
#pragma unroll
        for (int ci = 0; ci < BN / 32; ++ci) {
          const int col = ci * 32 + lane;
          c_tok[ci] = -1;
          c_w[ci] = 0.0f;
          if (col < un.y_rows) {
            const int p = un.y_row0 + col;
            const int tok = a.route_token[p];
            const int slot = a.route_slot[p];
            if (tok >= 0 && tok < a.n_tokens && slot >= 0 && slot < a.topk) {
              c_tok[ci] = tok;
              c_w[ci] = a.topk_w[static_cast<int64_t>(tok) * a.topk + slot];
            } else {
              raise_status(a.status, NVFP4_ERR_DEVICE_CHECK);
            }
          }
        }
      }
      // all lanes wait (sleeping between polls, see mbar_wait_sleepy), then
      // agree, so the warp-collective loads below stay converged
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_sleepy(accf_bar(abuf), aphase, ctl, a.status)))
        break;
      tc_fence_after();
      const float alpha = __fmul_rn(grouped ? un.gxp[un.e] : a.gx[0], gy_u);
      const int n_valid = un.y_rows;
      if (!SP && MT == 2 && (emode == kGroupedSiluMul || emode == kGroupedSiluBf16)) {
        // (sparse weights: not fused)
        // Gate (X tile 0) and up (X tile 1) accumulators of the same 128
        // features: h = SiLU(alpha * gate) * (alpha * up) in FP32, quantised
        // per 16 features with the given global of h and written as NVFP4
        // into h's operand tiles (the layout the dispatch quantiser writes
        // for K = n_out / 2), row = the route's row in its token tile.
        const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                            abuf * MT * C::kIssuers * C::kAccCols;
        // one X tile's accumulator, the two MMA warps' partial sums added
        auto load_acc = [&](uint32_t ta, uint32_t (&r)[32]) {
          uint32_t r2[32];
          tmem_ld32(ta, r);
          if (n_acc == 2) tmem_ld32(ta + C::kAccCols, r2);
          tmem_ld_wait();
          if (n_acc == 2) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              r[i] = __float_as_uint(__fadd_rn(__uint_as_float(r[i]), __uint_as_float(r2[i])));
          }
        };
        // one 32-token chunk at a time; the accumulator buffer goes back to
        // the MMA warps after the last chunk (the other buffer keeps them busy)
        // (one accumulator buffer for 128-row units: the next unit's MMAs
        // wait for this epilogue)
#pragma unroll 1
        for (int ci = 0; ci < BN / 32; ++ci) {
        if (ci * 32 >= n_valid) break;
        uint32_t rg[32], ru[32];
        load_acc(tq + ci * 32, rg);
        load_acc(tq + C::kIssuers * C::kAccCols + ci * 32, ru);
        warp_transpose32(rg, lane);                // lane = token, 32 features of quarter q
        warp_transpose32(ru, lane);
        if (ci * 32 + lane < n_valid) {
          const ScaleK gh = scale_consts(emode == kGroupedSiluMul ? *a.g_h : 0.0f);
          float h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float gz = __fmul_rn(__uint_as_float(rg[i]), alpha);
            const float uz = __fmul_rn(__uint_as_float(ru[i]), alpha);
            h[i] = __fmul_rn(__fdiv_rn(gz, __fadd_rn(1.0f, expf(-gz))), uz);
          }
          const int f0 = un.x_local0 + q * 32;     // first feature of h in this lane
          if (emode == kGroupedSiluBf16) {
            // two-phase form: h in BF16, route order, 32 consecutive features
            uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) +
                            static_cast<int64_t>(un.y_row0 + ci * 32 + lane) * a.ldc + f0;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w4[4];
#pragma unroll
              for (int hh = 0; hh < 4; ++hh)
                w4[hh] = static_cast<uint32_t>(f32_to_bf16_rn(h[8 * v + 2 * hh])) |
                         (static_cast<uint32_t>(f32_to_bf16_rn(h[8 * v + 2 * hh + 1])) << 16);
              reinterpret_cast<uint4*>(dst)[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            continue;
          }
          const Block16 b0 = quantize16(h, gh);
          const Block16 b1 = quantize16(h + 16, gh);
          const int row = ci * 32 + lane;          // token tile = one layout chunk (BN <= 128)
          const int64_t tile = (static_cast<int64_t>(un.y_tile) * a.h_nkb + (f0 >> 8)) *
                               kOperandTileBytes;
          const int chunk = (f0 & 255) >> 5;       // 16-byte chunk of the 128-byte row
          *reinterpret_cast<uint4*>(a.h_tiles + tile + row * 128 + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(b0.packed.x, b0.packed.y, b1.packed.x, b1.packed.y);
          const int sc = (f0 & 255) >> 4;          // scale column (even)
          *reinterpret_cast<uint16_t*>(a.h_tiles + tile + kXTileBytes + (sc >> 2) * 512 +
                                       (row & 31) * 16 + ((row >> 5) & 3) * 4 + (sc & 3)) =
              static_cast<uint16_t>(b0.sf | (b1.sf << 8));
        }
        }
        tc_fence_before();
        mbar_arrive(acce_bar(abuf));               // both accumulators have been read
        if (++abuf == C::kAccBufs) { abuf = 0; aphase ^= 1u; }
        if (mode == kMlpFused) {
          // this warp's 32 features of h for the unit's tokens are written:
          // count them for the token tile (each lane orders its stores, the
          // warp meets, one lane releases); a token tile is complete at 4
          // counts per gate_up unit.  No wait here: a warp that gave up
          // above never blocks the others.
          fence_proxy_async_global();
          __threadfence();
          __syncwarp();
          if (lane == 0) red_release_add1(a.ready + un.y_tile);
        }
        continue;
      }
      if (C::kAccBufs == 1 && emode != kGroupedCombine && emode != kGroupedSiluMul &&
          emode != kGroupedSiluBf16) {
        // One accumulator: the next unit's MMAs wait for it.  Read all of it
        // into registers as BF16 first, hand it back, then store, so the
        // stores overlap the next unit's MMAs.
        uint32_t pk[kGrpCols / 32][16];           // BF16 pairs of alpha * acc
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + gc0;
        // two 32-column loads in flight per wait (the load latency, not the
        // conversion, sets the drain time)
#pragma unroll
        for (int cp2 = 0; cp2 < kGrpCols / 64; ++cp2) {
          if (gc0 + cp2 * 64 < n_valid) {
            uint32_t r[2][32];
            tmem_ld32(taddr + cp2 * 64, r[0]);
            tmem_ld32(taddr + cp2 * 64 + 32, r[1]);
            tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int ci = 2 * cp2 + hh;
              if (mode != kDenseRowsX) warp_transpose32(r[hh], lane);
#pragma unroll
              for (int h = 0; h < 16; ++h)
                pk[ci][h] = static_cast<uint32_t>(
                                f32_to_bf16_rn(__fmul_rn(__uint_as_float(r[hh][2 * h]), alpha))) |
                            (static_cast<uint32_t>(f32_to_bf16_rn(
                                 __fmul_rn(__uint_as_float(r[hh][2 * h + 1]), alpha))) << 16);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(acce_bar(abuf));
        if (++abuf == C::kAccBufs) { abuf = 0; aphase ^= 1u; }
#pragma unroll
        for (int ci = 0; ci < kGrpCols / 32; ++ci) {
          const int c0 = gc0 + ci * 32;
          if (c0 >= n_valid) continue;
          uint16_t* dst;
          bool vec;
          int lim;                                 // valid elements of this lane's 32
          if (mode == kDenseRowsX) {
            const int xr = un.x_local0 + row;
            if (xr >= a.rows_x) continue;
            dst = reinterpret_cast<uint16_t*>(a.out) + static_cast<int64_t>(xr) * a.ldc +
                  un.y_row0 + c0;
            lim = min(32, n_valid - c0);
          } else {
            const int col = c0 + lane;
            if (col >= n_valid) continue;
            const int f0 = un.x_local0 + q * 32;
            dst = reinterpret_cast<uint16_t*>(a.out) + (un.y_row0 + col) * a.ldc + f0;
            lim = (mode == kGrouped) ? 32 : min(32, a.rows_x - f0);
          }
          vec = (lim == 32) && a.vec_store;
          if (vec) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              reinterpret_cast<uint4*>(dst)[v] =
                  make_uint4(pk[ci][4 * v], pk[ci][4 * v + 1], pk[ci][4 * v + 2], pk[ci][4 * v + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < lim) dst[i] = static_cast<uint16_t>(pk[ci][i >> 1] >> (16 * (i & 1)));
          }
        }
        continue;
      }
#pragma unroll 1
      for (int xt = 0; xt < MT; ++xt) {           // the unit's X tiles
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                             (abuf * MT + xt) * C::kIssuers * C::kAccCols;
      const int xr = un.x_local0 + xt * 128 + row;  // output feature / X row
      for (int c0 = gc0; c0 < min(n_valid, gc0 + kGrpCols); c0 += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        if (n_acc == 2) {                 // the second issuer's partial sums
          uint32_t r2[32];
          tmem_ld32(taddr + C::kAccCols + c0, r2);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            r[i] = __float_as_uint(__fadd_rn(__uint_as_float(r[i]), __uint_as_float(r2[i])));
        } else {
          tmem_ld_wait();
        }
        const int nc = min(32, n_valid - c0);
        if (mode == kDenseRowsX) {
          if (xr < a.rows_x) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + static_cast<int64_t>(xr) * a.ldc +
                            un.y_row0 + c0;
            if (nc == 32 && a.vec_store) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float f0 = __fmul_rn(__uint_as_float(r[8 * v + 2 * h]), alpha);
                  const float f1 = __fmul_rn(__uint_as_float(r[8 * v + 2 * h + 1]), alpha);
                  w[h] = static_cast<uint32_t>(f32_to_bf16_rn(f0)) |
                         (static_cast<uint32_t>(f32_to_bf16_rn(f1)) << 16);
                }
                reinterpret_cast<uint4*>(dst)[v] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < nc) dst[j] = f32_to_bf16_rn(__fmul_rn(__uint_as_float(r[j]), alpha));
            }
          }
        } else if (emode == kGroupedCombine) {
          // Combine.  Lane = feature f0 + lane, r[j] = token column c0 + j.
          // Four token columns at a time go through this warp's 512 bytes of
          // shared memory (feature fastest) and come back as lane = (token
          // column lane / 8 of the four, features 4 (lane % 8) .. + 3), so
          // each 16-byte reduction carries four consecutive features of one
          // token and a warp's reduction instruction covers four whole
          // 128-byte rows of the FP32 output (lanes on tokens would touch 32
          // rows, 16 bytes each).
          const int f0 = un.x_local0 + xt * 128 + q * 32;  // first feature of this warp
          float* xb = reinterpret_cast<float*>(smem + C::kXchgOffset) + (grp * 4 + q) * 128;
          int tok_l = c_tok[0];
          float w_l = c_w[0];
#pragma unroll
          for (int ci = 1; ci < BN / 32; ++ci)
            if (c0 == ci * 32) { tok_l = c_tok[ci]; w_l = c_w[ci]; }
#pragma unroll
          for (int sc = 0; sc < 8; ++sc) {
            if (4 * sc >= nc) break;                 // uniform
            __syncwarp();                            // the previous group's reads are done
#pragma unroll
            for (int jl = 0; jl < 4; ++jl)
              xb[jl * 32 + lane] = __fmul_rn(__uint_as_float(r[4 * sc + jl]), alpha);
            __syncwarp();
            const int jc = 4 * sc + (lane >> 3);     // token column in the chunk
            const float4 v =
                *reinterpret_cast<const float4*>(xb + (lane >> 3) * 32 + 4 * (lane & 7));
            const int tok = __shfl_sync(0xFFFFFFFFu, tok_l, jc);
            const float w = __shfl_sync(0xFFFFFFFFu, w_l, jc);
            if (jc < nc && tok >= 0) {               // (a rejected route has tok < 0)
              float4 acc4;
              acc4.x = __fmul_rn(w, v.x);
              acc4.y = __fmul_rn(w, v.y);
              acc4.z = __fmul_rn(w, v.z);
              acc4.w = __fmul_rn(w, v.w);
              red_add_v4(a.ws + static_cast<int64_t>(tok) * un.n_out + f0 + 4 * (lane & 7), acc4);
            }
          }
        } else {
          // Transposed orientations: lane l takes token column c0 + l and the
          // 32 features of this warp, so stores are vectors.
          warp_transpose32(r, lane);
          const int col = c0 + lane;
          const int f0 = un.x_local0 + xt * 128 + q * 32;  // first feature of this warp
          if (col < n_valid) {
            const int64_t y = un.y_row0 + col;
            uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + y * a.ldc + f0;
            const bool full = (mode == kGrouped) || (f0 + 32 <= a.rows_x);
            if (full && a.vec_store) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float v0 = __fmul_rn(__uint_as_float(r[8 * v + 2 * h]), alpha);
                  const float v1 = __fmul_rn(__uint_as_float(r[8 * v + 2 * h + 1]), alpha);
                  w[h] = static_cast<uint32_t>(f32_to_bf16_rn(v0)) |
                         (static_cast<uint32_t>(f32_to_bf16_rn(v1)) << 16);
                }
                reinterpret_cast<uint4*>(dst)[v] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (mode == kGrouped || f0 + i < a.rows_x)
                  dst[i] = f32_to_bf16_rn(__fmul_rn(__uint_as_float(r[i]), alpha));
            }
          }
        }
      }
      }  // X tiles
      tc_fence_before();
      mbar_arrive(acce_bar(abuf));
      if (++abuf == C::kAccBufs) { abuf = 0; aphase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// FP32 [T, N] -> BF16 [T, N], round to nearest even.
__global__ void __launch_bounds__(256) combine_finalize_kernel(const float* __restrict__ ws,
                                                               int64_t n4, uint16_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += stride) {
    const float4 v = reinterpret_cast<const float4*>(ws)[i];
    uint2 o;
    o.x = static_cast<uint32_t>(f32_to_bf16_rn(v.x)) | (static_cast<uint32_t>(f32_to_bf16_rn(v.y)) << 16);
    o.y = static_cast<uint32_t>(f32_to_bf16_rn(v.z)) | (static_cast<uint32_t>(f32_to_bf16_rn(v.w)) << 16);
    reinterpret_cast<uint2*>(out)[i] = o;
  }
}

}  // namespace

template <int BN, int MT = 1, bool SP = false>
static cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(nvfp4_gemm_kernel<BN, MT, SP>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<BN, MT, SP>::kSmemBytes);
}

cudaError_t init_gemm_attributes() {
  cudaError_t e = set_smem_attr<32>();
  if (e == cudaSuccess) e = set_smem_attr<32, 2>();
  if (e == cudaSuccess) e = set_smem_attr<64, 2>();
  if (e == cudaSuccess) e = set_smem_attr<128, 2>();
  if (e == cudaSuccess) e = set_smem_attr<64>();
  if (e == cudaSuccess) e = set_smem_attr<128>();
  if (e == cudaSuccess) e = set_smem_attr<256>();
  if (e == cudaSuccess) e = set_smem_attr<32, 1, true>();
  if (e == cudaSuccess) e = set_smem_attr<32, 2, true>();
  if (e == cudaSuccess) e = set_smem_attr<64, 2, true>();
  if (e == cudaSuccess) e = set_smem_attr<64, 1, true>();
  if (e == cudaSuccess) e = set_smem_attr<128, 1, true>();
  return e;
}

template <int BN, int MT = 1, bool SP = false>
static cudaError_t launch_bn(const CUtensorMap& tmx, const CUtensorMap& tmy, const GemmArgs& a,
                             int mode, int grid, cudaStream_t s) {
  nvfp4_gemm_kernel<BN, MT, SP>
      <<<grid, Cfg<BN, MT, SP>::kThreads, Cfg<BN, MT, SP>::kSmemBytes, s>>>(tmx, tmy, a, mode);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const CUtensorMap& tmx, const CUtensorMap& tmy, const GemmArgs& a,
                        int mode, int sms, cudaStream_t s) {
  int grid = sms;
  if (mode == kDenseRowsX || mode == kDenseRowsY) {
    // 256-wide Y tiles when Y is large: each MMA instruction then covers
    // 128 x 256 x 64 and a K block moves 1.33x fewer bytes per FLOP
    const int bn = (mode == kDenseRowsX && a.rows_y >= 256) ? 256 : 128;
    const int64_t units = ((a.rows_x + 127) / 128) * ((a.rows_y + bn - 1) / bn);
    if (units < grid) grid = static_cast<int>(units);
    if (grid < 1) return cudaSuccess;
    return bn == 256 ? launch_bn<256>(tmx, tmy, a, mode, grid, s)
                     : launch_bn<128>(tmx, tmy, a, mode, grid, s);
  }
  // 2:4-sparse weights (gather or combine): token tiles of the activation
  // layout's chunk width (128 for prefill shapes)
  if (a.sparse_w) {
    switch (grouped_chunk_rows(a.rows_y, a.E)) {
      case 32:   // two weight tiles per unit when the expert's rows pair up
        return (a.n_out / 128) % 2 == 0 ? launch_bn<32, 2, true>(tmx, tmy, a, mode, grid, s)
                                         : launch_bn<32, 1, true>(tmx, tmy, a, mode, grid, s);
      case 64:
        return (a.n_out / 128) % 2 == 0 ? launch_bn<64, 2, true>(tmx, tmy, a, mode, grid, s)
                                         : launch_bn<64, 1, true>(tmx, tmy, a, mode, grid, s);
      default: return launch_bn<128, 1, true>(tmx, tmy, a, mode, grid, s);
    }
  }
  // gate and up tiles pair up in one unit of 32, 64 or 128 routes, the
  // activation layout's chunk width (with dense weights, <64, 2> and <128, 2>
  // serve only these modes)
  if (mode == kGroupedSiluMul || mode == kGroupedSiluBf16) {
    switch (grouped_chunk_rows(a.rows_y, a.E)) {
      case 32: return launch_bn<32, 2>(tmx, tmy, a, mode, grid, s);
      case 64: return launch_bn<64, 2>(tmx, tmy, a, mode, grid, s);
      default: return launch_bn<128, 2>(tmx, tmy, a, mode, grid, s);
    }
  }
  switch (grouped_tile_width(a.rows_y, a.E)) {
    case 32:   // two weight tiles per unit when the expert's rows pair up
      return (a.n_out / 128) % 2 == 0 ? launch_bn<32, 2>(tmx, tmy, a, mode, grid, s)
                                       : launch_bn<32>(tmx, tmy, a, mode, grid, s);
    case 64:
      // two weight tiles per unit when the tiles pair up: twice the weight
      // bytes in flight per stage for the same token bytes (down projection
      // at 512 tokens: 0.179 -> 0.170 ms)
      return (a.n_out / 128) % 2 == 0 ? launch_bn<64, 2>(tmx, tmy, a, mode, grid, s)
                                       : launch_bn<64>(tmx, tmy, a, mode, grid, s);
    case 128: return launch_bn<128>(tmx, tmy, a, mode, grid, s);
    default: return launch_bn<256>(tmx, tmy, a, mode, grid, s);
  }
}

template <int BN>
static cudaError_t launch_mlp_bn(const GemmArgs& a, int grid, cudaStream_t s) {
  static_assert(Cfg<BN, 2>::kEpiGroups == 1, "the ready counts assume four epilogue warps");
  CUtensorMap unused{};                          // the grouped path needs no tensor map
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // the down units wait on other CTAs' work
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(Cfg<BN, 2>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<BN, 2>::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, nvfp4_gemm_kernel<BN, 2, false>, unused, unused, a,
                            static_cast<int>(kMlpFused));
}

cudaError_t launch_mlp_fused(const GemmArgs& a, int sms, cudaStream_t s) {
  switch (grouped_chunk_rows(a.rows_y, a.E)) {
    case 32: return launch_mlp_bn<32>(a, sms, s);
    case 64: return launch_mlp_bn<64>(a, sms, s);
    default: return launch_mlp_bn<128>(a, sms, s);
  }
}

cudaError_t launch_combine_finalize(const float* ws, int64_t T, int64_t N, void* out, int sms,
                                    cudaStream_t s) {
  const int64_t n4 = T * N / 4;
  if (n4 == 0) return cudaSuccess;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  combine_finalize_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(ws, n4,
                                                                  static_cast<uint16_t*>(out));
  return cudaGetLastError();
}

}  // namespace nvfp4
