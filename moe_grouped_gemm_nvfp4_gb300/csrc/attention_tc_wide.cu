// Decode attention over an NVFP4 KV cache with both contractions on the
// tensor cores, for heads of 256 and 512 ("The Blackwell architectural
// split", The Breakthrough -- The A4Q Kernel: attention layers with 512-wide
// heads, the cache kept in NVFP4 and expanded on chip inside the loop).
//
// A tile of 128 cached tokens at these widths does not fit on chip at once
// (K^ and V^ of one tile are 128 KB each at D = 512), so the work runs as two
// persistent kernels that stream the rows in slices of 128 head dimensions:
//
//   scores:  S[t, g] = sum over slices of K^_s[t, :] . q_s[g, :]  (A = K^ slice
//            in tensor memory, B = q slice in shared memory), times the
//            softmax scale, the K global and log2(e), written per token to
//            the workspace (base 2);
//   values:  per split, the maximum of its scores, p = 2^(S - max) as two FP16
//            parts, and O^T_s[d, g] += sum_t V^_s[t, d] P^T[g, t] per slice
//            (A = V^ slice in shared memory, MN-major), then the same split
//            partials as the kernels for narrower heads.
//
// K^ and V^ are exact FP16 expansions (E2M1 x E4M3, see
// attention_tc_common.cuh); q enters FP16 scaled per head by a power of two,
// exact for BF16.  With the split's maximum known before its first P, no
// rescaling is needed.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "attention.h"
#include "attention_tc_common.cuh"

namespace nvfp4 {

namespace {

// raw ring stages (one slice of a tile each) and expanded slices in flight.
// Both kernels run two CTAs per SM (measured: 512-wide heads in groups of 4,
// 0.18 ms with one CTA of each per SM, 0.14 ms with two), so that twice the
// warps hide the latency of the expansion's loads, waits and stores; the
// values kernel's ring and buffers are sized to fit two CTAs.
constexpr int kScoreStages = 6, kScoreNBuf = 3;
// score tiles the MMA warp may run ahead of the front warps that read them
// (their item boundaries, where q of the next item is written, take time)
constexpr int kScoreSBuf = 4;
constexpr int kValueCtas = 2, kValueStages = 3, kValueNBuf = 2;
constexpr int kWideFrontWarps = 4, kWideExpWarps = 8;
constexpr int kWideProdWarp = kWideFrontWarps + kWideExpWarps, kWideMmaWarp = kWideProdWarp + 1;
constexpr int kWideThreads = (kWideMmaWarp + 1) * 32;   // 448

template <int D>
struct WideCfg {
  static constexpr int NS = D / 128;                     // slices of 128 dimensions
  static constexpr int kRawCodes = 128 * 64;             // a slice's codes: 64 bytes per row
  static constexpr int kRawScales = 128 * 16;            // 16 scale bytes per row (two slices)
  static constexpr int kStage = kRawCodes + kRawScales;  // 10 KB
  static constexpr int kQhBuf = (D / 64) * 2048;         // q: 16 rows x D FP16, K-major
  static constexpr int kVhBuf = 2 * 16384;               // V^ slice: 128 tokens x 128 dims
  static constexpr int kPhBuf = 4096;                    // P^T: 16 rows x 128 tokens
  // scores kernel: ring | q x 2 | reductions | control | barriers
  static constexpr int kSQh = kScoreStages * kStage;
  static constexpr int kSRed = kSQh + 2 * kQhBuf;
  // values kernel: ring | V^ buffers | P^T x 2 | reductions | control | barriers
  static constexpr int kVVh = kValueStages * kStage;
  static constexpr int kVPh = kVVh + kValueNBuf * kVhBuf;
  static constexpr int kVRed = kVPh + 2 * kPhBuf;
  static_assert(kStage % 1024 == 0 && kSQh % 1024 == 0 && kVVh % 1024 == 0, "layout");
};

// Shared memory after the layout-specific part: [4][16] reductions x 3,
// control block, barriers, tensor-memory slot.
constexpr int kWideTail = 768 + 16 + 40 * 8 + 16;

template <int D>
constexpr int wide_scores_bytes() { return WideCfg<D>::kSRed + kWideTail + 1024; }
template <int D>
constexpr int wide_values_bytes() { return WideCfg<D>::kVRed + kWideTail + 1024; }
// two scores CTAs and kValueCtas values CTAs per SM: 228 KB of shared memory
// per SM, 1 KB of it reserved per CTA
template <int D>
constexpr bool wide_fits() {
  return 2 * (wide_scores_bytes<D>() + 1024) <= 233472 &&
         kValueCtas * (wide_values_bytes<D>() + 1024) <= 233472;
}
static_assert(wide_fits<256>() && wide_fits<512>(), "CTAs per SM");

// 16-byte chunk of a 64-byte code row as the TMA's 64-byte swizzle places it
__device__ __forceinline__ int swz64(int t) { return (t >> 1) & 3; }

// q of a work item as the front warps hold it: thread tid has elements
// tid + 128 k (k < G * D / 128) of the item's G heads, two BF16 per word.
// Loaded one item ahead (the loads are issued where written and land while
// the current item's tiles go by).
template <int D, int G>
struct WideQ {
  static constexpr int kElems = G * D / 128;            // per thread
  uint32_t w[kElems / 2];
};

template <int D, int G>
__device__ __forceinline__ void wide_load_q(const AttnArgs& a, int64_t w, WideQ<D, G>& q) {
  const int tid = threadIdx.x;
  const WsIdx x = ws_idx(a, w);
  const int j = static_cast<int>(x.j), b = static_cast<int>(x.b);
  const uint16_t* qp = a.q + (static_cast<int64_t>(b) * a.Hq + j * G) * D + tid;
#pragma unroll
  for (int k = 0; k < WideQ<D, G>::kElems; k += 2)
    q.w[k / 2] = ld_prefetch_u16(qp + 128 * k) | (ld_prefetch_u16(qp + 128 * (k + 1)) << 16);
}

// q -> FP16 operand rows of buffer qh (each head scaled by the power of two
// that puts its largest magnitude in [2^13, 2^14), exact for BF16); qm[g]
// gets the factor that turns head g's MMA scores into base-2 scaled scores.
// Element k of a thread is head k / (D / 128), dimension 128 (k % (D / 128))
// + tid.  Called by the four front warps together (named-barrier reductions,
// which also make ok the same in all of them).
template <int D, int G>
__device__ __forceinline__ void wide_write_q(const AttnArgs& a, const WideQ<D, G>& q, uint8_t* qh,
                                             float* redq, float (&qm)[G], bool& ok) {
  constexpr int KE = WideQ<D, G>::kElems, KD = D / 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto val = [&](int k) {
    return bf16_bits_to_f32((q.w[k / 2] >> (16 * (k & 1))) & 0xFFFFu);
  };
  float m[G];
#pragma unroll
  for (int g = 0; g < G; ++g) m[g] = 0.0f;
#pragma unroll
  for (int k = 0; k < KE; ++k) m[k / KD] = fmaxf(m[k / KD], fabsf(val(k)));
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m[g] = fmaxf(m[g], __shfl_xor_sync(0xFFFFFFFFu, m[g], o));
    if (lane == 0) redq[warp * 16 + g] = m[g];
  }
  ok = softmax_bar_and(ok);
  const float qmul = a.scale * (*a.gk) * kLog2eTc;
  float up[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float mg = fmaxf(fmaxf(redq[g], redq[16 + g]), fmaxf(redq[32 + g], redq[48 + g]));
    int e = 0;
    if (mg > 0.0f) e = 13 - ((__float_as_uint(mg) >> 23) & 0xFF) + 127;
    e = max(-100, min(100, e));
    qm[g] = qmul * __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    up[g] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
  }
#pragma unroll
  for (int k = 0; k < KE; ++k) {
    const int g = k / KD, d = (k % KD) * 128 + tid;
    *reinterpret_cast<__half*>(qh + (d >> 6) * 2048 + kmajor_chunk(g, (d & 63) >> 3) +
                               (d & 7) * 2) = __float2half_rn(val(k) * up[g]);
  }
  // the next reduction overwrites redq only after every thread read it
  ok = softmax_bar_and(ok);
}

// ---------------------------------------------------------------------------
// Scores kernel: warps 0-3 write q and store the scores, 4-11 expand K slices
// into tensor memory (lane = token), 12 copies the raw slices, 13 issues the
// score MMAs.  Tensor memory: K^ slices at 64 b (b < 3), S of tile t at
// 192 + 16 (t % kScoreSBuf).
// ---------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(kWideThreads, 2)
decode_scores_wide_kernel(const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tsk, const AttnArgs a) {
  using C = WideCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  float* redq = reinterpret_cast<float*>(smem + C::kSRed);
  CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + C::kSRed + 768);
  const uint32_t bars = sbase + C::kSRed + 768 + 16;
  auto raw_full = [&](uint32_t st) { return bars + 8u * st; };
  auto raw_empty = [&](uint32_t st) { return bars + 8u * (kScoreStages + st); };
  const uint32_t op_full0 = bars + 8u * (2 * kScoreStages), k_free0 = op_full0 + 8 * kScoreNBuf,
                 s_full0 = k_free0 + 8 * kScoreNBuf, s_empty0 = s_full0 + 8 * kScoreSBuf,
                 q_full0 = s_empty0 + 8 * kScoreSBuf, q_empty0 = q_full0 + 16,
                 fin = q_empty0 + 16;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + C::kSRed + 768 + 16 + 40 * 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    ctl->abort = 0u;
    ctl->timeout_ns = a.timeout_ns;
    for (int st = 0; st < kScoreStages; ++st) {
      mbar_init(raw_full(st), 1);
      mbar_init(raw_empty(st), kWideExpWarps);
    }
    for (int h = 0; h < kScoreNBuf; ++h) {
      mbar_init(op_full0 + 8 * h, kWideExpWarps);
      mbar_init(k_free0 + 8 * h, 1);
    }
    for (int h = 0; h < kScoreSBuf; ++h) {
      mbar_init(s_full0 + 8 * h, 1);
      mbar_init(s_empty0 + 8 * h, kWideFrontWarps);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(q_full0 + 8 * h, kWideFrontWarps);
      mbar_init(q_empty0 + 8 * h, 1);
    }
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), 256);
    tmem_relinquish();
  }
  for (int i = tid; i < 2 * C::kQhBuf / 16; i += kWideThreads)   // q rows G..15 stay zero
    reinterpret_cast<uint4*>(smem + C::kSQh)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const int64_t items = static_cast<int64_t>(a.splits) * a.Hkv * a.B;

  if (warp == kWideProdWarp) {
    // ---------------------------------------------------------------- producer
    const uint64_t policy = l2_policy_evict_first();
    uint32_t i = 0;
    bool ok = true, skipped_first = false;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile) {
        for (int s = 0; s < NS && ok; ++s, ++i) {
          const uint32_t st = i % kScoreStages;
          if (i >= kScoreStages)
            ok = __all_sync(0xFFFFFFFFu, ws_wait(raw_empty(st), ((i / kScoreStages) - 1) & 1u,
                                                 ctl, a.status));
          if (!ok) break;
          if (i == 0 && (a.debug_flags & kDebugSkipFirstStage)) {
            skipped_first = true;                        // test hook: this stage never fills
            continue;
          }
          const uint32_t dst = sbase + st * C::kStage;
          const int32_t r = static_cast<int32_t>(it.row0 + tt);
          mbar_arrive_expect_tx_elect(raw_full(st), C::kStage);
          tma_load_2d_elect(dst, &tmk, raw_full(st), 64 * s, r, policy);
          tma_load_2d_elect(dst + C::kRawCodes, &tsk, raw_full(st), 16 * (s >> 1), r, policy);
        }
      }
    }
    const uint32_t issued = i;
    for (uint32_t k = issued > kScoreStages ? issued - kScoreStages : 0; k < issued; ++k)
      if (k > 0 || !skipped_first) ws_drain(raw_full(k % kScoreStages), (k / kScoreStages) & 1u,
                                            a.timeout_ns);
  } else if (warp >= kWideFrontWarps && warp < kWideProdWarp) {
    // ------------------------------------------------------- K expansion
    // lane = token of the warp's lane quarter; part pp of the slice's eight
    // 16-element blocks (four each)
    const int e = warp - kWideFrontWarps;
    const int tk = (warp & 3) * 32 + lane, pp = e >> 2;
    uint32_t i = 0;
    bool ok = true;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile) {
        const int rows = static_cast<int>(min(static_cast<int64_t>(kTile), it.t1 - tt));
        for (int s = 0; s < NS; ++s, ++i) {
          const uint32_t st = i % kScoreStages, ob = i % kScoreNBuf;
          ok = __all_sync(0xFFFFFFFFu, ws_wait(raw_full(st), (i / kScoreStages) & 1u, ctl,
                                               a.status));
          if (!ok) break;
          const uint8_t* raw = smem + st * C::kStage;
          uint32_t kw[8];
          uint32_t ksw = 0u;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) kw[jj] = 0u;
          if (tk < rows) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int ch = (pp * 2 + jj) ^ swz64(tk);
              const uint4 q = *reinterpret_cast<const uint4*>(raw + tk * 64 + ch * 16);
              kw[4 * jj] = q.x; kw[4 * jj + 1] = q.y; kw[4 * jj + 2] = q.z; kw[4 * jj + 3] = q.w;
            }
            ksw = *reinterpret_cast<const uint32_t*>(raw + C::kRawCodes + tk * 16 + (s & 1) * 8 +
                                                     pp * 4);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(raw_empty(st));
          if (i >= kScoreNBuf)                   // the score MMAs of the buffer's last slice are done
            ok = __all_sync(0xFFFFFFFFu, ws_wait(k_free0 + 8 * ob, ((i / kScoreNBuf) - 1) & 1u,
                                                 ctl, a.status));
          if (!ok) break;
          uint32_t kv[32];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 lo, hi;
            expand16(kw[2 * u], kw[2 * u + 1], (ksw >> (8 * u)) & 0xFFu, lo, hi);
            kv[8 * u + 0] = lo.x; kv[8 * u + 1] = lo.y; kv[8 * u + 2] = lo.z; kv[8 * u + 3] = lo.w;
            kv[8 * u + 4] = hi.x; kv[8 * u + 5] = hi.y; kv[8 * u + 6] = hi.z; kv[8 * u + 7] = hi.w;
          }
          tmem_st32(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 64u * ob + 32u * pp,
                    kv);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(op_full0 + 8 * ob);
        }
      }
    }
  } else if (warp == kWideMmaWarp) {
    // ------------------------------------------------------------- score MMAs
    const uint32_t idesc_s = idesc_f16(16, 0);
    uint32_t i = 0, k = 0, t = 0;
    bool ok = true;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x, ++k) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      const uint32_t qb = k & 1u;
      ok = __all_sync(0xFFFFFFFFu, ws_wait(q_full0 + 8 * qb, (k >> 1) & 1u, ctl, a.status));
      if (!ok) break;
      if (it.t1 <= it.t0) {
        mbar_arrive_elect(q_empty0 + 8 * qb);
        continue;
      }
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile, ++t) {
        const uint32_t sb = t % kScoreSBuf;
        if (t >= kScoreSBuf)                             // the front warps have read this S buffer
          ok = __all_sync(0xFFFFFFFFu, ws_wait(s_empty0 + 8 * sb, ((t / kScoreSBuf) - 1) & 1u,
                                               ctl, a.status));
        for (int s = 0; s < NS && ok; ++s, ++i) {
          const uint32_t ob = i % kScoreNBuf;
          ok = __all_sync(0xFFFFFFFFu, ws_wait(op_full0 + 8 * ob, (i / kScoreNBuf) & 1u, ctl,
                                               a.status));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_f16_ts_elect(tmem + 192 + 16 * sb, tmem + 64 * ob + 8 * kk,
                                sdesc_sw128(sbase + C::kSQh + qb * C::kQhBuf +
                                            (2 * s + (kk >> 2)) * 2048 + (kk & 3) * 32),
                                idesc_s, (s > 0 || kk > 0) ? 1u : 0u);
          tc_commit_elect(k_free0 + 8 * ob);
        }
        if (ok) tc_commit_elect(s_full0 + 8 * sb);
      }
      if (ok) tc_commit_elect(q_empty0 + 8 * qb);
    }
    tc_commit_elect(fin);
    ws_drain(fin, 0u, a.timeout_ns);
  } else {
    // ------------------------------------------ q, the score stores, the maxima
    // Thread tid stores token tt + tid of every tile and keeps the largest
    // score per head; at the end of the item the four warps reduce them (in
    // the buffer of the item's parity, so one barrier per item suffices) and
    // thread 0 writes the split's reference maximum.  A split without tokens
    // gets its whole partial here (O 0, maximum -inf, sum 0).  q of the next
    // item is written after the item's first tile (from registers loaded an
    // item earlier), so the scores of a tile never wait for it.
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float* redm = redq + 64;                             // [2][4][16]
    float qm_cur[G], qm_nxt[G];
#pragma unroll
    for (int g = 0; g < G; ++g) qm_cur[g] = qm_nxt[g] = 0.0f;
    bool ok = true;
    const int64_t w0 = blockIdx.x, stride = gridDim.x;
    WsItem it_nxt{};
    int n_nn = 0;
    WideQ<D, G> qr;
    if (w0 < items) {
      wide_load_q<D, G>(a, w0, qr);
      wide_write_q<D, G>(a, qr, smem + C::kSQh, redq, qm_cur, ok);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full0);
      it_nxt = ws_item(a, w0, ws_len(a, w0, items));
      n_nn = ws_len(a, w0 + stride, items);
      if (w0 + stride < items) wide_load_q<D, G>(a, w0 + stride, qr);
    }
    uint32_t k = 0, t = 0;
    // No warp leaves the item loop on its own: the named-barrier reductions
    // need all four (ok is made uniform by each of them); after a failed wait
    // a warp skips its work until the next reduction.
    for (int64_t w = w0; w < items; w += stride, ++k) {
      const WsItem it = it_nxt;
      const bool has_next = w + stride < items;
      if (it.bad_len && tid == 0) raise_status(a.status, NVFP4_ERR_DEVICE_CHECK);
      auto part_of = [&](int g) {
        return (static_cast<int64_t>(it.b) * a.Hq + it.j * G + g) * a.splits + it.split;
      };
      float xmax[G];
#pragma unroll
      for (int g = 0; g < G; ++g) xmax[g] = -INFINITY;
      // scores of tile tt: from tensor memory, stored, and the maxima kept
      auto score_tile = [&](int64_t tt) {
        const uint32_t sb = t % kScoreSBuf;
        ok = __all_sync(0xFFFFFFFFu, ok && ws_wait(s_full0 + 8 * sb, (t / kScoreSBuf) & 1u, ctl,
                                                   a.status));
        ++t;
        if (!ok) return;
        tc_fence_after();
        uint32_t sr[16];
        tmem_ld16(tmem + lane_base + 192 + 16 * sb, sr);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty0 + 8 * sb);
        const int64_t tok = tt + tid;
        if (tok < it.t1) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float x = __uint_as_float(sr[g]) * qm_cur[g];
            xmax[g] = fmaxf(xmax[g], x);
            a.ws_s[(static_cast<int64_t>(it.b) * a.Hq + it.j * G + g) * a.L_max + tok] = x;
          }
        }
      };
      int64_t tt = it.t0;
      if (tt < it.t1) {
        score_tile(tt);
        tt += kTile;
      }
      if (has_next) {                                    // q of the next item, other buffer
        const uint32_t nb = (k + 1) & 1u;
        if (k >= 1)
          ok = __all_sync(0xFFFFFFFFu, ok && ws_wait(q_empty0 + 8 * nb, ((k - 1) >> 1) & 1u, ctl,
                                                     a.status));
        wide_write_q<D, G>(a, qr, smem + C::kSQh + nb * C::kQhBuf, redq, qm_nxt, ok);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full0 + 8 * nb);
        it_nxt = ws_item(a, w + stride, n_nn);
        n_nn = ws_len(a, w + 2 * stride, items);
        if (w + 2 * stride < items) wide_load_q<D, G>(a, w + 2 * stride, qr);
      }
      if (it.t1 > it.t0) {
        for (; tt < it.t1; tt += kTile) score_tile(tt);
        float* rm = redm + (k & 1u) * 64;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float m = xmax[g];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
          if (lane == 0) rm[warp * 16 + g] = m;
        }
        ok = softmax_bar_and(ok);
        if (!ok) break;
        if (tid < G)
          a.ws_ml[2 * part_of(tid)] =
              fmaxf(fmaxf(rm[tid], rm[16 + tid]), fmaxf(rm[32 + tid], rm[48 + tid]));
      } else {                                           // no cached token in this split
        if (!ok) break;
        for (int e = tid; e < G * D; e += 128) {
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
    tmem_dealloc(tmem, 256);
  }
}


// ---------------------------------------------------------------------------
// Values kernel: warps 0-3 turn the stored scores into P^T and write the split
// partials, 4-11 expand V slices into shared memory (MN-major operand), 12
// copies the raw slices, 13 issues the value MMAs.  Tensor memory: O^T of
// slice s for item parity c at 16 (NS c + s), columns g (high part of P) and
// 8 + g (low part).  Splits without tokens were written by the scores kernel
// and are skipped by every role here.
// ---------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(kWideThreads, kValueCtas)
decode_values_wide_kernel(const __grid_constant__ CUtensorMap tmv,
                          const __grid_constant__ CUtensorMap tsv, const AttnArgs a) {
  using C = WideCfg<D>;
  constexpr int NS = C::NS;
  constexpr uint32_t kCols = NS * 32 <= 32 ? 32u : static_cast<uint32_t>(NS * 32);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  float* redl = reinterpret_cast<float*>(smem + C::kVRed);      // [2][4][16]
  CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + C::kVRed + 768);
  const uint32_t bars = sbase + C::kVRed + 768 + 16;
  auto raw_full = [&](uint32_t st) { return bars + 8u * st; };
  auto raw_empty = [&](uint32_t st) { return bars + 8u * (kValueStages + st); };
  const uint32_t v_full0 = bars + 8u * (2 * kValueStages), v_free0 = v_full0 + 8 * kValueNBuf,
                 p_full0 = v_free0 + 8 * kValueNBuf, p_empty0 = p_full0 + 16,
                 o_full0 = p_empty0 + 16, o_empty0 = o_full0 + 16, fin = o_empty0 + 16;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + C::kVRed + 768 + 16 + 40 * 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    ctl->abort = 0u;
    ctl->timeout_ns = a.timeout_ns;
    for (int st = 0; st < kValueStages; ++st) {
      mbar_init(raw_full(st), 1);
      mbar_init(raw_empty(st), kWideExpWarps);
    }
    for (int h = 0; h < kValueNBuf; ++h) {
      mbar_init(v_full0 + 8 * h, kWideExpWarps);
      mbar_init(v_free0 + 8 * h, 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(p_full0 + 8 * h, kWideFrontWarps);
      mbar_init(p_empty0 + 8 * h, 1);
      mbar_init(o_full0 + 8 * h, 1);
      mbar_init(o_empty0 + 8 * h, kWideFrontWarps);
    }
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), kCols);
    tmem_relinquish();
  }
  for (int i = tid; i < 2 * C::kPhBuf / 16; i += kWideThreads)   // P^T rows past the group stay zero
    reinterpret_cast<uint4*>(smem + C::kVPh)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const int64_t items = static_cast<int64_t>(a.splits) * a.Hkv * a.B;

  if (warp == kWideProdWarp) {
    // ---------------------------------------------------------------- producer
    const uint64_t policy = l2_policy_evict_first();
    uint32_t i = 0;
    bool ok = true, skipped_first = false;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile) {
        for (int s = 0; s < NS && ok; ++s, ++i) {
          const uint32_t st = i % kValueStages;
          if (i >= kValueStages)
            ok = __all_sync(0xFFFFFFFFu, ws_wait(raw_empty(st), ((i / kValueStages) - 1) & 1u,
                                                 ctl, a.status));
          if (!ok) break;
          if (i == 0 && (a.debug_flags & kDebugSkipFirstStage)) {
            skipped_first = true;                        // test hook: this stage never fills
            continue;
          }
          const uint32_t dst = sbase + st * C::kStage;
          const int32_t r = static_cast<int32_t>(it.row0 + tt);
          mbar_arrive_expect_tx_elect(raw_full(st), C::kStage);
          tma_load_2d_elect(dst, &tmv, raw_full(st), 64 * s, r, policy);
          tma_load_2d_elect(dst + C::kRawCodes, &tsv, raw_full(st), 16 * (s >> 1), r, policy);
        }
      }
    }
    const uint32_t issued = i;
    for (uint32_t k = issued > kValueStages ? issued - kValueStages : 0; k < issued; ++k)
      if (k > 0 || !skipped_first) ws_drain(raw_full(k % kValueStages), (k / kValueStages) & 1u,
                                            a.timeout_ns);
  } else if (warp >= kWideFrontWarps && warp < kWideProdWarp) {
    // ------------------------------------------------------- V expansion
    // Lanes 8m .. 8m + 7 (one pass of a 16-byte store) take four blocks of two
    // adjacent rows, so the operand's 128-byte swizzle spreads each pass over
    // all eight bank groups; a thread handles four rows, 32 apart.
    const int e = warp - kWideFrontWarps;
    const int blk = ((lane >> 3) & 1) * 4 + (lane & 3);
    const int rin = (lane >> 4) * 2 + ((lane >> 2) & 1);
    const int trow0 = e * 4 + rin;
    const uint32_t sw = static_cast<uint32_t>(trow0 & 7);
    const uint32_t c = static_cast<uint32_t>(2 * blk) & 7u;
    const uint32_t off0 = (blk >> 2) * 16384 + (trow0 >> 3) * 1024 + sw * 128;
    const uint32_t offlo = off0 + ((c ^ sw) << 4), offhi = off0 + (((c + 1) ^ sw) << 4);
    constexpr int kUnits = 4;
    constexpr uint32_t kUnitStride = 4 * 1024;           // 32 rows
    uint32_t i = 0;
    bool ok = true;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile) {
        const int rows = static_cast<int>(min(static_cast<int64_t>(kTile), it.t1 - tt));
        for (int s = 0; s < NS; ++s, ++i) {
          const uint32_t st = i % kValueStages, vb = i % kValueNBuf;
          ok = __all_sync(0xFFFFFFFFu, ws_wait(raw_full(st), (i / kValueStages) & 1u, ctl,
                                               a.status));
          if (!ok) break;
          const uint8_t* raw = smem + st * C::kStage;
          uint2 vcode[kUnits];
          uint32_t vscale[kUnits];
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            const int t = trow0 + 32 * u;
            vcode[u] = make_uint2(0u, 0u);
            vscale[u] = 0u;
            if (t < rows) {                              // rows past the split stay zero
              const int ch = (blk >> 1) ^ swz64(t);
              vcode[u] = *reinterpret_cast<const uint2*>(raw + t * 64 + ch * 16 + (blk & 1) * 8);
              vscale[u] = raw[C::kRawCodes + t * 16 + (s & 1) * 8 + blk];
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(raw_empty(st));
          if (i >= kValueNBuf)                   // the MMAs of the buffer's last slice are done
            ok = __all_sync(0xFFFFFFFFu, ws_wait(v_free0 + 8 * vb, ((i / kValueNBuf) - 1) & 1u,
                                                 ctl, a.status));
          if (!ok) break;
          uint8_t* vh = smem + C::kVVh + vb * C::kVhBuf;
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            uint4 lo, hi;
            expand16(vcode[u].x, vcode[u].y, vscale[u], lo, hi);
            *reinterpret_cast<uint4*>(vh + offlo + u * kUnitStride) = lo;
            *reinterpret_cast<uint4*>(vh + offhi + u * kUnitStride) = hi;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(v_full0 + 8 * vb);
        }
      }
    }
  } else if (warp == kWideMmaWarp) {
    // ------------------------------------------------------------- value MMAs
    const uint32_t idesc_o = idesc_f16(16, 1);
    uint32_t i = 0, t = 0, kq = 0;
    bool ok = true;
    int n_nxt = ws_len(a, blockIdx.x, items);
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      if (it.t1 <= it.t0) continue;
      const uint32_t oc = kq & 1u;
      if (kq >= 2)                                       // O of item kq - 2 has been read
        ok = __all_sync(0xFFFFFFFFu, ws_wait(o_empty0 + 8 * oc, ((kq >> 1) - 1) & 1u, ctl,
                                             a.status));
      ++kq;
      for (int64_t tt = it.t0; tt < it.t1 && ok; tt += kTile, ++t) {
        const uint32_t pb = t & 1u;
        ok = __all_sync(0xFFFFFFFFu, ws_wait(p_full0 + 8 * pb, (t >> 1) & 1u, ctl, a.status));
        for (int s = 0; s < NS && ok; ++s, ++i) {
          const uint32_t vb = i % kValueNBuf;
          ok = __all_sync(0xFFFFFFFFu, ws_wait(v_full0 + 8 * vb, (i / kValueNBuf) & 1u, ctl,
                                               a.status));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t va =
                sdesc_sw128_mn(sbase + C::kVVh + vb * C::kVhBuf + kk * 2048, 16384, 1024);
            const uint32_t pa = sbase + C::kVPh + pb * C::kPhBuf + (kk >> 2) * 2048 + (kk & 3) * 32;
            tc_mma_f16_elect(tmem + 16 * (NS * oc + s), va, sdesc_sw128(pa), idesc_o,
                             (tt > it.t0 || kk > 0) ? 1u : 0u);
          }
          tc_commit_elect(v_free0 + 8 * vb);
        }
        if (ok) tc_commit_elect(p_empty0 + 8 * pb);
      }
      if (ok) tc_commit_elect(o_full0 + 8 * oc);
    }
    tc_commit_elect(fin);
    ws_drain(fin, 0u, a.timeout_ns);
  } else {
    // ------------------------------------------------------ P^T and the partials
    // Thread tid: token tt + tid of each tile; dimension 128 s + tid of O.
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t pc = (tid >> 6) * 2048 + (tid & 7) * 2;
    bool ok = true;
    uint32_t t = 0, kq = 0;
    int n_nxt = ws_len(a, blockIdx.x, items);
    // No warp leaves the item loop on its own (the sum's reduction needs all four).
    for (int64_t w = blockIdx.x; w < items; w += gridDim.x) {
      const WsItem it = ws_item(a, w, n_nxt);
      n_nxt = ws_len(a, w + gridDim.x, items);
      if (it.t1 <= it.t0) continue;
      const uint32_t oc = kq & 1u;
      auto part_of = [&](int g) {
        return (static_cast<int64_t>(it.b) * a.Hq + it.j * G + g) * a.splits + it.split;
      };
      const float* srow = a.ws_s + (static_cast<int64_t>(it.b) * a.Hq + it.j * G) * a.L_max;
      float m[G], l[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = a.ws_ml[2 * part_of(g)];
        l[g] = 0.0f;
      }
      for (int64_t tt = it.t0; tt < it.t1; tt += kTile, ++t) {
        const uint32_t pb = t & 1u;
        const int64_t tok = tt + tid;
        const bool valid = tok < it.t1;
        float x[G];
#pragma unroll
        for (int g = 0; g < G; ++g)
          x[g] = valid ? srow[static_cast<int64_t>(g) * a.L_max + tok] : -INFINITY;
        if (t >= 2)                                      // the MMAs of tile t - 2 read this buffer
          ok = __all_sync(0xFFFFFFFFu, ok && ws_wait(p_empty0 + 8 * pb, ((t >> 1) - 1) & 1u, ctl,
                                                     a.status));
        if (!ok) break;
        uint8_t* pt = smem + C::kVPh + pb * C::kPhBuf;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = valid ? exp2f(x[g] - m[g]) : 0.0f;
          const __half ph = __float2half_rn(p);
          const __half pl = __float2half_rn(p - __half2float(ph));
          l[g] += p;
          *reinterpret_cast<__half*>(pt + pc + kmajor_chunk(g, (tid & 63) >> 3)) = ph;
          *reinterpret_cast<__half*>(pt + pc + kmajor_chunk(8 + g, (tid & 63) >> 3)) = pl;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full0 + 8 * pb);
      }
      // O of the item, slice by slice
      ok = __all_sync(0xFFFFFFFFu, ok && ws_wait(o_full0 + 8 * oc, (kq >> 1) & 1u, ctl,
                                                 a.status));
      ++kq;
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int s = 0; s < NS; ++s) {
          uint32_t orr[16];
          tmem_ld16(tmem + lane_base + 16 * (NS * oc + s), orr);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < G; ++g)
            a.ws_o[part_of(g) * D + 128 * s + tid] =
                __uint_as_float(orr[g]) + __uint_as_float(orr[8 + g]);
        }
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty0 + 8 * oc);
      float* rl = redl + oc * 64;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float v = l[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (lane == 0) rl[warp * 16 + g] = v;
      }
      ok = softmax_bar_and(ok);
      if (!ok) break;
      if (tid < G)
        a.ws_ml[2 * part_of(tid) + 1] = (rl[tid] + rl[16 + tid]) + (rl[32 + tid] + rl[48 + tid]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

template <typename K>
cudaError_t set_wide_attr(K kern, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
  return e;
}

template <int D, int G>
cudaError_t set_wide_attrs_dg() {
  cudaError_t e = set_wide_attr(decode_scores_wide_kernel<D, G>, wide_scores_bytes<D>());
  if (e == cudaSuccess) e = set_wide_attr(decode_values_wide_kernel<D, G>, wide_values_bytes<D>());
  return e;
}

// groups of 2, 4 and 8 query heads; 512-wide heads take at most 4
template <int D>
cudaError_t set_wide_attrs_d() {
  cudaError_t e = set_wide_attrs_dg<D, 2>();
  if (e == cudaSuccess) e = set_wide_attrs_dg<D, 4>();
  if constexpr (D == 256)
    if (e == cudaSuccess) e = set_wide_attrs_dg<D, 8>();
  return e;
}

// Both kernels persistent (two scores CTAs per SM, kValueCtas values CTAs, or
// one per work item when there are fewer), on the same stream: the values
// kernel reads what the scores kernel wrote.
template <int D, int G>
cudaError_t launch_wide_d_g(const AttnArgs& a, const AttnMaps& m, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t items = static_cast<int64_t>(a.splits) * a.Hkv * a.B;
  auto grid_of = [&](int64_t ctas) { return static_cast<unsigned>(items < ctas ? items : ctas); };
  decode_scores_wide_kernel<D, G><<<grid_of(2LL * sms), kWideThreads, wide_scores_bytes<D>(), s>>>(
      m.k_codes, m.k_scales, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_values_wide_kernel<D, G><<<grid_of(static_cast<int64_t>(kValueCtas) * sms), kWideThreads,
                                    wide_values_bytes<D>(), s>>>(m.v_codes, m.v_scales, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_wide_d(const AttnArgs& a, int G, const AttnMaps& m, cudaStream_t s) {
  if (G == 2) return launch_wide_d_g<D, 2>(a, m, s);
  if (G == 4) return launch_wide_d_g<D, 4>(a, m, s);
  if constexpr (D == 256) return launch_wide_d_g<D, 8>(a, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t init_attention_tc_wide_attributes() {
  cudaError_t e = set_wide_attrs_d<256>();
  if (e == cudaSuccess) e = set_wide_attrs_d<512>();
  return e;
}

cudaError_t launch_decode_attention_tc_wide(const AttnArgs& a, int D, const AttnMaps& m,
                                            cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  if ((D != 256 && D != 512) || (G != 2 && G != 4 && G != 8)) return cudaErrorInvalidValue;
  return D == 256 ? launch_wide_d<256>(a, G, m, s) : launch_wide_d<512>(a, G, m, s);
}

}  // namespace nvfp4
