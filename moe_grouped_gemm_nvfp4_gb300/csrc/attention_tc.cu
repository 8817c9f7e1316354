// Decode attention over an NVFP4 KV cache with both contractions on the
// tensor cores (tcgen05, FP16 operands, FP32 accumulation in tensor memory),
// for heads of 128 (groups of 2, 4 or 8 query heads per KV head) and of 64
// (groups of 4 or 8).
//
// "The Blackwell architectural split", The Breakthrough -- The A4Q Kernel:
// the cache stays NVFP4 in memory (E2M1 values, an E4M3 scale per 16 numbers
// along the head dimension, one FP32 global for K and one for V) and is
// expanded on chip inside the attention loop.  Here the expansion goes to
// FP16 in shared memory, where the products E2M1 x E4M3 are exact (at most 6
// significant bits, between 2^-10 and 2688), so that the two contractions of
// a tile become tensor-core MMAs instead of per-element multiply-adds:
//
//   S[t, g]  = sum_d K^[t, d] q[g, d]          M 128 cached tokens, N 16 (heads), K = D
//   O^T[d, g] += sum_t V^[t, d] P[t, g]        M = 128 (D, padded), N 16, K 128 tokens
//
// K^ and V^ are the cache rows times their block scales (the globals are
// applied to the scores and by the split merge); q enters in FP16 scaled per
// head by a power of two (exact for its BF16 values).  V^ is written in its
// natural token-row order and read by the MMA as an MN-major operand, so no
// transpose is needed.  The split partials (unnormalised O, reference maximum
// in base 2, sum) have the layout the merge kernel of attention.cu reads.
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "attention.h"
#include "attention_tc_common.cuh"

namespace nvfp4 {

namespace {

// ---------------------------------------------------------------------------
// Pipelined form for heads of 64 and 128: one CTA per SM with specialised
// warps, so that the cache streams, the expansion to FP16, the MMAs and the
// softmax of different tiles overlap.
//
//   warps 0-3   softmax: scores from tensor memory, P^T, the split partials;
//               they also write q of the next work item
//   warps 4-11  expansion: raw tile -> K^ in tensor memory (lane = token) and
//               V^ in shared memory (MN-major)
//   warp 12     producer: TMA boxes of the raw cache tiles (codes and scales
//               of 128 tokens) into a ring
//   warp 13     score MMAs: S = K^ q^T of each tile, A from tensor memory
//   warp 14     value MMAs: O^T += V^T P^T of each tile
//
// K^, V^, P^T and S rotate through three buffers (tiles in flight between
// the roles).  O accumulates in tensor memory over the tiles of a work item
// (one buffer per item parity).  The softmax keeps a reference maximum per
// head and rescales O and the sums only when a score exceeds it by more than
// 2^8 (so p <= 256); within a tile no maximum is exchanged unless that
// happens.  P is the sum of two FP16 parts (22 significant bits) held in the
// two halves of the MMA's 16 columns: rows g (high) and 8 + g (low), so one
// MMA takes both and O = columns g + 8 + g.  S and O are each split over two
// accumulators (even and odd K steps of the MMAs).
// Every wait is bounded (CtaCtl): on expiry the kernel records
// NVFP4_ERR_TIMEOUT, every role leaves its loop, and the copies and MMAs in
// flight are waited for before the tensor memory is freed.
// ---------------------------------------------------------------------------
constexpr int kWsStages = 4;
constexpr int kSoftWarps = 4, kExpWarps = 8;
constexpr int kProdWarp = kSoftWarps + kExpWarps, kSWarp = kProdWarp + 1, kOWarp = kSWarp + 1;
constexpr int kWsThreads = (kOWarp + 1) * 32;            // 480
constexpr float kRescaleLog2 = 8.0f;                     // p <= 2^8 between rescales
constexpr int kNBuf = 3;                                 // tiles in flight between the roles
// tensor memory (512 columns): K^ of buffer b at columns 64 b (the score
// MMA's A operand: lane t = token t, two FP16 per column along D); S of
// buffer b at 192 + 32 b and O of item parity c at 288 + 32 c, each as two
// 16-column accumulators (even and odd MMA K steps) that the softmax adds
constexpr uint32_t kKCol = 0, kSCol = 192, kOCol = 288, kWsTmemCols = 512;

template <int D>
struct WsCfg {
  static constexpr int KB = D / 2;                       // code bytes per cache row
  static constexpr int SB = D / 16;                      // scale bytes per cache row
  static constexpr int kBlk = D / 64;
  static constexpr int kRawCodes = 128 * KB;
  static constexpr int kRawScales = 128 * SB;
  // a ring stage: K codes, V codes, K scales, V scales of 128 tokens
  static constexpr int kStage = 2 * kRawCodes + 2 * kRawScales;
  static constexpr int kVhBuf = 2 * 16384;               // V^: M padded to 128, MN-major
  static constexpr int kPhBuf = 4096;                    // P^T: 16 rows x 128 tokens FP16
  static constexpr int kQhBuf = kBlk * 2048;             // q: 16 rows x D FP16, K-major
  static constexpr int kVh = kWsStages * kStage;
  static constexpr int kPh = kVh + kNBuf * kVhBuf;
  static constexpr int kQh = kPh + kNBuf * kPhBuf;
  static constexpr int kRed = kQh + 2 * kQhBuf;          // [4][16] maxima
  static constexpr int kRedQ = kRed + 256;               // [4][16] q maxima
  static constexpr int kRedL = kRedQ + 256;              // [4][16] sums
  static constexpr int kCtl = kRedL + 256;
  static constexpr int kBar = kCtl + 16;
  static constexpr int kNumBars = 2 * kWsStages + 4 * kNBuf + 6;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kBytes = kSlot + 16 + 1024;       // + alignment slack
  static_assert(kStage % 1024 == 0, "layout");
  static_assert(sizeof(CtaCtl) == 16, "control block");
  static_assert(kBytes <= 232448, "shared memory");
};

template <int D, int G>
__global__ void __launch_bounds__(kWsThreads, 1)
decode_attention_ws_kernel(const __grid_constant__ CUtensorMap tmk,
                           const __grid_constant__ CUtensorMap tmv,
                           const __grid_constant__ CUtensorMap tsk,
                           const __grid_constant__ CUtensorMap tsv, const AttnArgs a) {
  static_assert(G <= 8, "P's high and low parts share the MMA's 16 columns");
  static_assert(D == 64 || D == 128, "four or eight 16-element blocks per row");
  using C = WsCfg<D>;
  constexpr int KB = C::KB, SB = C::SB, NB = D / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + C::kCtl);
  const uint32_t bars = sbase + C::kBar;
  // per-buffer barriers (kNBuf each), then the q buffers' pair and the drains
  const uint32_t op_full0 = bars + 8u * (2 * kWsStages), o_done0 = op_full0 + 8 * kNBuf,
                 s_full0 = o_done0 + 8 * kNBuf, p_full0 = s_full0 + 8 * kNBuf,
                 q_full0 = p_full0 + 8 * kNBuf, q_empty0 = q_full0 + 16, fin_s = q_empty0 + 16,
                 fin_o = fin_s + 8;
  auto raw_full = [&](uint32_t st) { return bars + 8u * st; };
  auto raw_empty = [&](uint32_t st) { return bars + 8u * (kWsStages + st); };
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + C::kSlot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    ctl->abort = 0u;
    ctl->timeout_ns = a.timeout_ns;
    for (int st = 0; st < kWsStages; ++st) {
      mbar_init(raw_full(st), 1);
      mbar_init(raw_empty(st), kExpWarps);
    }
    for (int h = 0; h < kNBuf; ++h) {
      mbar_init(op_full0 + 8 * h, kExpWarps);
      mbar_init(o_done0 + 8 * h, 1);
      mbar_init(s_full0 + 8 * h, 1);
      mbar_init(p_full0 + 8 * h, kSoftWarps);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(q_full0 + 8 * h, kSoftWarps);
      mbar_init(q_empty0 + 8 * h, 1);
    }
    mbar_init(fin_s, 1);
    mbar_init(fin_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), kWsTmemCols);
    tmem_relinquish();
  }
  // the q and P^T buffers start at zero (rows the group does not use stay
  // so); for 64-wide heads the value operands' second M block is zero padding
  for (int i = tid; i < 2 * C::kQhBuf / 16; i += kWsThreads)
    reinterpret_cast<uint4*>(smem + C::kQh)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = tid; i < kNBuf * C::kPhBuf / 16; i += kWsThreads)
    reinterpret_cast<uint4*>(smem + C::kPh)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (D < 128)
    for (int i = tid; i < kNBuf * 16384 / 16; i += kWsThreads) {
      const int h = i / (16384 / 16), r = i % (16384 / 16);
      reinterpret_cast<uint4*>(smem + C::kVh + h * C::kVhBuf + 16384)[r] =
          make_uint4(0u, 0u, 0u, 0u);
    }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const int64_t items = static_cast<int64_t>(a.splits) * a.Hkv * a.B;

  if (warp == kProdWarp) {
    // ---------------------------------------------------------------- producer
    const uint64_t policy = l2_policy_evict_first();
    uint32_t i = 0;
    bool ok = true, skipped_first = false;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile, ++i) {
        const uint32_t st = i % kWsStages;
        if (i >= kWsStages)
          ok = __all_sync(0xFFFFFFFFu, ws_wait(raw_empty(st), ((i / kWsStages) - 1) & 1u, ctl,
                                               a.status));
        if (!ok) break;
        const uint32_t dst = sbase + st * C::kStage;
        const int64_t r = it.row0 + tt;
        if (i == 0 && (a.debug_flags & kDebugSkipFirstStage)) {
          skipped_first = true;                          // test hook: this stage never fills
          continue;
        }
        // 128-row TMA boxes: the codes with the row-width swizzle, the scales
        // as 16-byte rows (16 / SB cache rows each).  Rows past the split's
        // end are read too and left unused; past the cache's end they are
        // zero-filled.
        mbar_arrive_expect_tx_elect(raw_full(st), 2 * C::kRawCodes + 2 * C::kRawScales);
        tma_load_2d_elect(dst, &tmk, raw_full(st), 0, static_cast<int32_t>(r), policy);
        tma_load_2d_elect(dst + C::kRawCodes, &tmv, raw_full(st), 0, static_cast<int32_t>(r),
                          policy);
        const int32_t rs = static_cast<int32_t>(r * SB / 16);
        tma_load_2d_elect(dst + 2 * C::kRawCodes, &tsk, raw_full(st), 0, rs, policy);
        tma_load_2d_elect(dst + 2 * C::kRawCodes + C::kRawScales, &tsv, raw_full(st), 0, rs,
                          policy);
      }
    }
    // every copy this warp issued has landed before the CTA can exit
    const uint32_t issued = i;
    for (uint32_t k = issued > kWsStages ? issued - kWsStages : 0; k < issued; ++k)
      if (k > 0 || !skipped_first) ws_drain(raw_full(k % kWsStages), (k / kWsStages) & 1u, a.timeout_ns);
  } else if (warp >= kSoftWarps && warp < kProdWarp) {
    // --------------------------------------------------------------- expansion
    // The raw code rows arrive swizzled by the TMA: 16-byte chunk c of row t
    // sits at chunk c ^ ((t >> 1) & 3) for 64-byte rows (D 128) and c ^ ((t >> 2)
    // & 1) for 32-byte rows (D 64).
    auto swz = [](int t) { return NB == 8 ? ((t >> 1) & 3) : ((t >> 2) & 1); };
    const int e = warp - kSoftWarps;
    // K: lane = token (the tensor-memory lane the score MMA reads as row t of
    // A); warp e takes the 32 tokens of its lane quarter and part pp of the
    // row's blocks (NBP of them), expands them and stores them with one
    // tcgen05.st
    constexpr int kParts = kExpWarps / 4;                // warps per lane quarter
    constexpr int NBP = NB / kParts;                     // blocks per part
    static_assert(NBP == 1 || NBP == 2 || NBP == 4, "parts of a K row");
    const int tk = (warp & 3) * 32 + lane, pp = e >> 2;
    const uint32_t kcol = static_cast<uint32_t>(pp * NBP * 8);
    // V: lanes 8m .. 8m + 7 (one pass of a 16-byte shared-memory store) take
    // four blocks of two adjacent rows, so the 128-byte swizzle of the V^
    // operand spreads each pass over all eight bank groups
    constexpr int kRowStep = kExpWarps * 32 / NB;        // rows between a thread's V units
    constexpr int kUnits = kTile / kRowStep;             // V units per thread
    const int blk = NB == 8 ? ((lane >> 3) & 1) * 4 + (lane & 3) : (lane & 3);
    const int rin = NB == 8 ? ((lane >> 4) * 2 + ((lane >> 2) & 1))
                            : ((lane >> 3) * 2 + ((lane >> 2) & 1));
    const int trow0 = e * (32 / NB) + rin;               // trow0 % 8 is the same for every unit
    const uint32_t sw = static_cast<uint32_t>(trow0 & 7);
    const uint32_t c = static_cast<uint32_t>(2 * blk) & 7u;
    const uint32_t off0 = (blk >> 2) * 16384 + (trow0 >> 3) * 1024 + sw * 128;
    const uint32_t offlo = off0 + ((c ^ sw) << 4), offhi = off0 + (((c + 1) ^ sw) << 4);
    constexpr uint32_t kUnitStride = (kRowStep / 8) * 1024;
    uint32_t i = 0;
    bool ok = true;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      for (int64_t tt = it.t0; tt < it.t1; tt += kTile, ++i) {
        const uint32_t st = i % kWsStages, ob = i % kNBuf;
        ok = __all_sync(0xFFFFFFFFu, ws_wait(raw_full(st), (i / kWsStages) & 1u, ctl, a.status));
        if (!ok) break;
        const int rows = static_cast<int>(min(static_cast<int64_t>(kTile), it.t1 - tt));
        const uint8_t* raw = smem + st * C::kStage;
        const uint8_t* ksr = raw + 2 * C::kRawCodes;    // scales, row-major [128][SB]
        const uint8_t* vsr = ksr + C::kRawScales;
        // part pp of token tk's K row: NBP blocks of 8 code bytes (whole 16-byte
        // chunks, or half of one when NBP is 1) and their NBP scale bytes
        uint32_t kw[2 * NBP];
        uint32_t ksw = 0u;
#pragma unroll
        for (int j = 0; j < 2 * NBP; ++j) kw[j] = 0u;
        if (tk < rows) {
          if constexpr (NBP >= 2) {
#pragma unroll
            for (int j = 0; j < NBP / 2; ++j) {
              const int ch = (pp * (NBP / 2) + j) ^ swz(tk);
              const uint4 q = *reinterpret_cast<const uint4*>(raw + tk * KB + ch * 16);
              kw[4 * j] = q.x; kw[4 * j + 1] = q.y; kw[4 * j + 2] = q.z; kw[4 * j + 3] = q.w;
            }
          } else {
            const int ch = (pp >> 1) ^ swz(tk);
            const uint2 q = *reinterpret_cast<const uint2*>(raw + tk * KB + ch * 16 + (pp & 1) * 8);
            kw[0] = q.x; kw[1] = q.y;
          }
          ksw = NBP == 4 ? *reinterpret_cast<const uint32_t*>(ksr + tk * SB + pp * 4)
                : NBP == 2 ? *reinterpret_cast<const uint16_t*>(ksr + tk * SB + pp * 2)
                           : ksr[tk * SB + pp];
        }
        uint2 vcode[kUnits];
        uint32_t vscale[kUnits];
#pragma unroll
        for (int k = 0; k < kUnits; ++k) {
          const int t = trow0 + k * kRowStep;
          vcode[k] = make_uint2(0u, 0u);
          vscale[k] = 0u;
          if (t < rows) {
            const int ch = (blk >> 1) ^ swz(t);
            vcode[k] = *reinterpret_cast<const uint2*>(raw + C::kRawCodes + t * KB + ch * 16 +
                                                      (blk & 1) * 8);
            vscale[k] = vsr[t * SB + blk];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty(st));       // the ring stage may be refilled
        if (i >= kNBuf)                                  // tile i - 3's MMAs are done with the buffers
          ok = __all_sync(0xFFFFFFFFu, ws_wait(o_done0 + 8 * ob, ((i / kNBuf) - 1) & 1u, ctl,
                                               a.status));
        if (!ok) break;
        // K^ -> tensor memory, row tk, columns kcol .. kcol + 8 NBP
        uint32_t kv[8 * NBP];
#pragma unroll
        for (int u = 0; u < NBP; ++u) {
          uint4 lo, hi;
          expand16(kw[2 * u], kw[2 * u + 1], (ksw >> (8 * u)) & 0xFFu, lo, hi);
          kv[8 * u + 0] = lo.x; kv[8 * u + 1] = lo.y; kv[8 * u + 2] = lo.z; kv[8 * u + 3] = lo.w;
          kv[8 * u + 4] = hi.x; kv[8 * u + 5] = hi.y; kv[8 * u + 6] = hi.z; kv[8 * u + 7] = hi.w;
        }
        const uint32_t kt = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kKCol +
                            64u * ob + kcol;
        if constexpr (NBP == 4) {
          tmem_st32(kt, kv);
        } else if constexpr (NBP == 2) {
          tmem_st16(kt, kv);
        } else {
          tmem_st8(kt, kv);
        }
        // V^ -> shared memory (MN-major operand)
        uint8_t* vh = smem + C::kVh + ob * C::kVhBuf;
#pragma unroll
        for (int k = 0; k < kUnits; ++k) {
          uint4 lo, hi;
          expand16(vcode[k].x, vcode[k].y, vscale[k], lo, hi);
          *reinterpret_cast<uint4*>(vh + offlo + k * kUnitStride) = lo;
          *reinterpret_cast<uint4*>(vh + offhi + k * kUnitStride) = hi;
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(op_full0 + 8 * ob);
      }
    }
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------- score MMAs
    const uint32_t idesc_s = idesc_f16(16, 0);
    uint32_t i = 0, k = 0;
    bool ok = true;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x, ++k) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      const uint32_t qb = k & 1u;
      ok = __all_sync(0xFFFFFFFFu, ws_wait(q_full0 + 8 * qb, (k >> 1) & 1u, ctl, a.status));
      if (!ok) break;
      if (it.t1 <= it.t0) {                              // nothing reads this q
        mbar_arrive_elect(q_empty0 + 8 * qb);
        continue;
      }
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile, ++i) {
        const uint32_t ob = i % kNBuf;
        ok = __all_sync(0xFFFFFFFFu, ws_wait(op_full0 + 8 * ob, (i / kNBuf) & 1u, ctl, a.status));
        if (!ok) break;
        tc_fence_after();
        // A = K^ in tensor memory: 16 K values (8 columns) per MMA
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_f16_ts_elect(tmem + kSCol + 32 * ob + 16 * (kk & 1),
                              tmem + kKCol + 64 * ob + 8 * kk,
                              sdesc_sw128(sbase + C::kQh + qb * C::kQhBuf + (kk >> 2) * 2048 +
                                          (kk & 3) * 32),
                              idesc_s, kk > 1 ? 1u : 0u);
        tc_commit_elect(s_full0 + 8 * ob);
      }
      if (ok) tc_commit_elect(q_empty0 + 8 * qb);        // q's buffer is free once these finish
    }
    tc_commit_elect(fin_s);                              // every MMA of this warp has completed
    ws_drain(fin_s, 0u, a.timeout_ns);
  } else if (warp == kOWarp) {
    // ------------------------------------------------------------- value MMAs
    const uint32_t idesc_o = idesc_f16(16, 1);
    uint32_t i = 0, k = 0;
    bool ok = true;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x, ++k) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      const uint32_t otm = tmem + kOCol + 32 * (k & 1u);
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile, ++i) {
        const uint32_t pb = i % kNBuf;
        ok = __all_sync(0xFFFFFFFFu, ws_wait(p_full0 + 8 * pb, (i / kNBuf) & 1u, ctl, a.status));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t va =
              sdesc_sw128_mn(sbase + C::kVh + pb * C::kVhBuf + kk * 2048, 16384, 1024);
          const uint32_t pa = sbase + C::kPh + pb * C::kPhBuf + (kk >> 2) * 2048 + (kk & 3) * 32;
          tc_mma_f16_elect(otm + 16 * (kk & 1), va, sdesc_sw128(pa), idesc_o,
                           (tt > it.t0 || kk > 1) ? 1u : 0u);
        }
        tc_commit_elect(o_done0 + 8 * pb);
      }
    }
    tc_commit_elect(fin_o);
    ws_drain(fin_o, 0u, a.timeout_ns);
  } else {
    // ----------------------------------------------------------------- softmax
    const int s = tid;                                   // token of S, dimension of O
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + C::kRed);
    float* redq = reinterpret_cast<float*>(smem + C::kRedQ);
    float* redl = reinterpret_cast<float*>(smem + C::kRedL);
    const float qmul = a.scale * (*a.gk) * kLog2eTc;
    // q of an item: thread s holds elements e = s + 128 k of the G x D values
    constexpr int QE = (G * D + 127) / 128;
    uint32_t qreg[QE];
    auto load_q = [&](int64_t w) {
      const WsIdx x = ws_idx(a, w);
      const int j = static_cast<int>(x.j), b = static_cast<int>(x.b);
      const uint16_t* qp = a.q + (static_cast<int64_t>(b) * a.Hq + j * G) * D;
#pragma unroll
      for (int k = 0; k < QE; ++k) {
        const int e = s + 128 * k;
        qreg[k] = e < G * D ? ld_prefetch_u16(qp + e) : 0u;
      }
    };
    bool ok = true;
    // q -> FP16 operand rows of buffer qb, each head scaled by the power of
    // two that puts its largest magnitude in [2^13, 2^14) (exact for BF16
    // values); qm gets each head's factor of the scores
    auto write_q = [&](uint32_t qb, float (&qm)[G]) {
      float m[G];
#pragma unroll
      for (int g = 0; g < G; ++g) m[g] = 0.0f;
#pragma unroll
      for (int k = 0; k < QE; ++k) {
        const int e = s + 128 * k;
        if (e < G * D) {
          const int g = e / D;
#pragma unroll
          for (int h = 0; h < G; ++h)
            if (h == g) m[h] = fmaxf(m[h], fabsf(bf16_bits_to_f32(qreg[k])));
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m[g] = fmaxf(m[g], __shfl_xor_sync(0xFFFFFFFFu, m[g], o));
        if (lane == 0) redq[warp * 16 + g] = m[g];
      }
      ok = softmax_bar_and(ok);
      int ex[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mg = fmaxf(fmaxf(redq[g], redq[16 + g]), fmaxf(redq[32 + g], redq[48 + g]));
        int e = 0;
        if (mg > 0.0f) e = 13 - ((__float_as_uint(mg) >> 23) & 0xFF) + 127;
        ex[g] = max(-100, min(100, e));
        qm[g] = qmul * __uint_as_float(static_cast<uint32_t>(127 - ex[g]) << 23);
      }
#pragma unroll
      for (int k = 0; k < QE; ++k) {
        const int e = s + 128 * k;
        if (e < G * D) {
          const int g = e / D, d = e - g * D;
          int eg = 0;
#pragma unroll
          for (int h = 0; h < G; ++h)
            if (h == g) eg = ex[h];
          const float up = __uint_as_float(static_cast<uint32_t>(127 + eg) << 23);
          *reinterpret_cast<__half*>(smem + C::kQh + qb * C::kQhBuf + (d >> 6) * 2048 +
                                     kmajor_chunk(g, (d & 63) >> 3) + (d & 7) * 2) =
              __float2half_rn(bf16_bits_to_f32(qreg[k]) * up);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full0 + 8 * qb);
    };

    float qm_cur[G], qm_nxt[G];
#pragma unroll
    for (int g = 0; g < G; ++g) qm_cur[g] = qm_nxt[g] = 0.0f;
    const int64_t w0 = blockIdx.x, stride = gridDim.x;
    WsItem it_nxt{};
    int n_nn = 0;
    if (w0 < items) {
      load_q(w0);
      write_q(0u, qm_cur);
      it_nxt = ws_item(a, w0, ws_len(a, w0, items));
      n_nn = ws_len(a, w0 + stride, items);
      if (w0 + stride < items) load_q(w0 + stride);
    }
    uint32_t i = 0, k = 0;
    for (int64_t w = w0; w < items && ok; w += stride, ++k) {
      const WsItem it = it_nxt;
      // q of the next item into the other buffer once the score MMAs of the
      // item before have released it, then the prefetches the items after
      // need: after this item's first tile (whose P goes first; the softmax
      // warps agree on ok there), or here when the item has no tile
      bool q_pending = w + stride < items;
      auto next_q = [&]() {
        const uint32_t nb = (k + 1) & 1u;
        if (k >= 1)
          ok = __all_sync(0xFFFFFFFFu, ok && ws_wait(q_empty0 + 8 * nb, ((k - 1) >> 1) & 1u, ctl,
                                                     a.status));
        write_q(nb, qm_nxt);
        it_nxt = ws_item(a, w + stride, n_nn);
        n_nn = ws_len(a, w + 2 * stride, items);
        if (w + 2 * stride < items) load_q(w + 2 * stride);
        q_pending = false;
      };
      if (q_pending && it.t1 <= it.t0) next_q();
      if (!ok) break;
      if (it.bad_len && s == 0) raise_status(a.status, NVFP4_ERR_DEVICE_CHECK);
      auto part_of = [&](int g) {
        return (static_cast<int64_t>(it.b) * a.Hq + it.j * G + g) * a.splits + it.split;
      };
      if (it.t1 > it.t0) {
        const uint32_t otm = tmem + lane_base + kOCol + 32 * (k & 1u);
        float m_ref[G], l_part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          m_ref[g] = -INFINITY;
          l_part[g] = 0.0f;
        }
        for (int64_t tt = it.t0; tt < it.t1; tt += kTile, ++i) {
          const uint32_t ob = i % kNBuf;
          const bool first = tt == it.t0;
          ok = __all_sync(0xFFFFFFFFu, ok && ws_wait(s_full0 + 8 * ob, (i / kNBuf) & 1u, ctl,
                                                     a.status));
          const bool valid = tt + s < it.t1;
          float x[G];
          bool need = first;
          if (ok) {
            tc_fence_after();
            uint32_t sr[16], sr2[16];
            tmem_ld16(tmem + lane_base + kSCol + 32 * ob, sr);
            tmem_ld16(tmem + lane_base + kSCol + 32 * ob + 16, sr2);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float sg = __uint_as_float(sr[g]) + __uint_as_float(sr2[g]);
              x[g] = valid ? sg * qm_cur[g] : -INFINITY;
              need = need || x[g] > m_ref[g] + kRescaleLog2;
            }
          }
          bool rescaled = false;
          if (softmax_bar_or(need || !ok)) {
            // a new reference maximum: exchange the tile's maxima
            if (ok) {
#pragma unroll
              for (int g = 0; g < G; ++g) {
                float m = x[g];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                if (lane == 0) red[warp * 16 + g] = m;
              }
            }
            ok = softmax_bar_and(ok);
            if (!ok) break;
            float corr[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float mt = fmaxf(fmaxf(red[g], red[16 + g]), fmaxf(red[32 + g], red[48 + g]));
              const float mn = fmaxf(m_ref[g], mt);
              corr[g] = m_ref[g] == -INFINITY ? 0.0f : exp2f(m_ref[g] - mn);
              l_part[g] *= corr[g];
              m_ref[g] = mn;
            }
            if (!first) {
              // O so far (through tile i - 1) times the correction
              ok = __all_sync(0xFFFFFFFFu, ws_wait(o_done0 + 8 * ((i - 1) % kNBuf), ((i - 1) / kNBuf) & 1u,
                                                   ctl, a.status));
              if (ok) {
                tc_fence_after();
                uint32_t orr[16], orr2[16];
                tmem_ld16(otm, orr);
                tmem_ld16(otm + 16, orr2);
                tmem_ld_wait();
#pragma unroll
                for (int g = 0; g < G; ++g) {
                  orr[g] = __float_as_uint(__uint_as_float(orr[g]) * corr[g]);
                  orr[8 + g] = __float_as_uint(__uint_as_float(orr[8 + g]) * corr[g]);
                  orr2[g] = __float_as_uint(__uint_as_float(orr2[g]) * corr[g]);
                  orr2[8 + g] = __float_as_uint(__uint_as_float(orr2[8 + g]) * corr[g]);
                }
                tmem_st16(otm, orr);
                tmem_st16(otm + 16, orr2);
                tmem_st_wait();
                rescaled = true;
              }
            }
            // the next exchange overwrites the maxima only after every thread read them
            ok = softmax_bar_and(ok);
            if (!ok) break;
          }
          // P^T: row g the high part, row 8 + g the low part of p for token s
          uint8_t* pt = smem + C::kPh + ob * C::kPhBuf;
          const uint32_t pc = (s >> 6) * 2048 + (s & 7) * 2;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float p = valid ? exp2f(x[g] - m_ref[g]) : 0.0f;
            const __half ph = __float2half_rn(p);
            const __half pl = __float2half_rn(p - __half2float(ph));
            l_part[g] += p;
            *reinterpret_cast<__half*>(pt + pc + kmajor_chunk(g, (s & 63) >> 3)) = ph;
            *reinterpret_cast<__half*>(pt + pc + kmajor_chunk(8 + g, (s & 63) >> 3)) = pl;
          }
          fence_proxy_async_smem();
          if (rescaled) tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full0 + 8 * ob);
          if (q_pending) next_q();
        }
        // O of the item: the value MMAs of its last tile have completed
        float o[G];
        if (ok) {
          ok = __all_sync(0xFFFFFFFFu, ws_wait(o_done0 + 8 * ((i - 1) % kNBuf), ((i - 1) / kNBuf) & 1u,
                                               ctl, a.status));
          if (ok) {
            tc_fence_after();
            uint32_t orr[16], orr2[16];
            tmem_ld16(otm, orr);
            tmem_ld16(otm + 16, orr2);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < G; ++g)
              o[g] = (__uint_as_float(orr[g]) + __uint_as_float(orr[8 + g])) +
                     (__uint_as_float(orr2[g]) + __uint_as_float(orr2[8 + g]));
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float l = l_part[g];
#pragma unroll
          for (int oo = 16; oo > 0; oo >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, oo);
          if (lane == 0) redl[warp * 16 + g] = l;
        }
        ok = softmax_bar_and(ok);
        if (!ok) break;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int64_t part = part_of(g);
          if (s < D) a.ws_o[part * D + s] = o[g];
          if (s == 0) {
            a.ws_ml[2 * part] = m_ref[g];
            a.ws_ml[2 * part + 1] = (redl[g] + redl[16 + g]) + (redl[32 + g] + redl[48 + g]);
          }
        }
      } else {                                           // no cached token in this split
        for (int e = s; e < G * D; e += 128) {
          const int g = e / D, d = e - g * D;
          a.ws_o[part_of(g) * D + d] = 0.0f;
          if (d == 0) {
            a.ws_ml[2 * part_of(g)] = -INFINITY;
            a.ws_ml[2 * part_of(g) + 1] = 0.0f;
          }
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) qm_cur[g] = qm_nxt[g];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kWsTmemCols);
  }
}

template <int D, int G>
cudaError_t set_ws_attr() {
  auto kern = decode_attention_ws_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       WsCfg<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
  return e;
}

template <int D>
cudaError_t set_ws_attrs_d() {
  cudaError_t e = set_ws_attr<D, 4>();
  if (e == cudaSuccess) e = set_ws_attr<D, 8>();
  if (D == 128 && e == cudaSuccess) e = set_ws_attr<D, 2>();
  return e;
}

// One CTA per SM (the pipeline's shared memory), or one per work item when
// there are fewer items.
template <int D, int G>
cudaError_t launch_ws_d_g(const AttnArgs& a, const AttnMaps& m, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t items = static_cast<int64_t>(a.splits) * a.Hkv * a.B;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  decode_attention_ws_kernel<D, G><<<grid, kWsThreads, WsCfg<D>::kBytes, s>>>(m.k_codes, m.v_codes,
                                                                             m.k_scales,
                                                                             m.v_scales, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_ws_d(const AttnArgs& a, int G, const AttnMaps& m, cudaStream_t s) {
  if constexpr (D == 128)
    if (G == 2) return launch_ws_d_g<D, 2>(a, m, s);
  return G == 4 ? launch_ws_d_g<D, 4>(a, m, s) : launch_ws_d_g<D, 8>(a, m, s);
}

}  // namespace

cudaError_t init_attention_tc_attributes() {
  cudaError_t e = set_ws_attrs_d<64>();
  if (e == cudaSuccess) e = set_ws_attrs_d<128>();
  if (e == cudaSuccess) e = init_attention_tc_wide_attributes();
  return e;
}

bool decode_attention_tc_applies(const AttnArgs& a, int D) {
  const int G = a.Hq / a.Hkv;
  // the pipelined kernels copy scale rows in 16-byte units: both scale
  // arrays 16-byte aligned and, for heads of 64 and 128 (scale rows of 4 and
  // 8 bytes), every (sequence, KV head) slab a whole number of units (L_max *
  // D / 16 bytes a multiple of 16)
  const bool units16 =
      ((reinterpret_cast<uintptr_t>(a.k_scales) | reinterpret_cast<uintptr_t>(a.v_scales)) &
       15u) == 0 &&
      (D >= 256 || (a.L_max * (D / 16)) % 16 == 0);
  const bool rows31 = static_cast<int64_t>(a.B) * a.Hkv * a.L_max < (int64_t{1} << 31);
  // group sizes where it beats the CUDA-core kernel (measured): 2, 4 and 8
  // query heads over heads of 128 and wider, 4 and 8 over 64-wide heads
  const bool groups = D >= 128 ? (G == 2 || G == 4 || (G == 8 && D != 512))
                              : (D == 64 && (G == 4 || G == 8));
  return groups && units16 && rows31;
}

cudaError_t launch_decode_attention_tc(const AttnArgs& a, int D, const AttnMaps& m,
                                       cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  if (!decode_attention_tc_applies(a, D)) return cudaErrorInvalidValue;
  if (D >= 256) return launch_decode_attention_tc_wide(a, D, m, s);
  return D == 64 ? launch_ws_d<64>(a, G, m, s) : launch_ws_d<128>(a, G, m, s);
}

}  // namespace nvfp4
