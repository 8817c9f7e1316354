// NVFP4 block-scaled GEMM and MoE grouped GEMM on 5th-generation tensor cores.
//
// One persistent, warp-specialised kernel serves the single GEMM and the
// grouped GEMM ("The FP4 Frontier", Finding 5: a persistent grouped GEMM over
// all experts to avoid launch overhead; "The SM120 FP4 GEMM Kernel
// Investigation", The Comprehensive Synthesis: A/B FP4 tiles plus their
// scale-factor tiles staged through shared memory over several stages).
//
// Roles of the 192 threads of a CTA (one CTA per SM):
//   warp 0      TMA producer: operand tiles (128-byte swizzle) and scale
//               atoms into a ring of shared-memory stages;
//   warp 1      tensor-memory allocation; lane 0 issues tcgen05.cp (scales
//               -> tensor memory) and tcgen05.mma kind::mxf4nvf4 into a
//               double-buffered FP32 accumulator in tensor memory;
//   warps 2-5   epilogue: tcgen05.ld, global-scale multiply, BF16 store or
//               weighted FP32 scatter-add (MoE combine).
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

namespace nvfp4 {

namespace {

constexpr int kThreads = 192;
constexpr int kRowBytes = 128;                 // 256 FP4 values = one swizzle row
constexpr int kBK = 256;                       // K elements per stage
constexpr int kXTileBytes = 128 * kRowBytes;   // 16 KB
constexpr int kSFStageBytes = 4 * 512;         // four scale atoms (K = 256)
constexpr int kTmemCols = 512;

template <int BN>
struct Cfg {
  static_assert(BN == 128, "tile width");
  static constexpr int kYTileBytes = BN * kRowBytes;
  static constexpr int kStageBytes = kXTileBytes + kYTileBytes + 2 * kSFStageBytes;
  static constexpr int kStages = 6;
  static constexpr int kAccCols = BN;
  static constexpr int kSfColBase = 2 * BN;    // scale columns follow the accumulators
  static_assert(kSfColBase + kStages * 32 <= kTmemCols, "tensor memory budget");
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr int kBarBytes = 8 * (2 * kStages + 5);
  static constexpr int kTableInts = 3 * (kGroupedMaxExperts + 1);
  static constexpr int kCtlOffset = kStages * kStageBytes + kBarBytes;
  static constexpr int kTablesOffset = kCtlOffset + 32;
  static constexpr int kSmemBytes = kTablesOffset + 4 * kTableInts + 1024;  // + align slack
};

struct Unit {
  int32_t x_row0;     // tensor-map row of the X tile
  int32_t y_row0;     // tensor-map row of the Y tile
  int32_t y_rows;     // valid Y rows (1..BN)
  int32_t x_local0;   // first output feature (grouped) / first X row (dense)
  int32_t e;          // expert (grouped)
  int64_t sfx_off;    // byte offset of the X scale atoms at k-block 0
  int64_t sfy_off;
};

struct Tables {
  int32_t* up;        // [E+1] unit prefix
  int32_t* off;       // [E+1] expert offsets
  int32_t* tb;        // [E+1] scale-tile prefix
};

template <int BN>
__device__ __forceinline__ Unit get_unit(int u, int mode, const GemmArgs& a, const Tables& t,
                                         int tiles_x, int64_t atoms_per_rowtile) {
  Unit un;
  if (mode == kGrouped || mode == kGroupedCombine) {
    int lo = 0, hi = a.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (t.up[mid] <= u) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int mtiles = a.n_out >> 7;
    const int local = u - t.up[e];
    const int mt = local % mtiles;
    const int nt = local / mtiles;
    const int cnt = t.off[e + 1] - t.off[e];
    un.e = e;
    un.x_row0 = e * a.n_out + mt * 128;
    un.x_local0 = mt * 128;
    un.y_row0 = t.off[e] + nt * BN;
    un.y_rows = min(BN, cnt - nt * BN);
    un.sfx_off = static_cast<int64_t>(e * mtiles + mt) * atoms_per_rowtile * 512;
    un.sfy_off = static_cast<int64_t>(t.tb[e] + nt * (BN / 128)) * atoms_per_rowtile * 512;
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
  }
  return un;
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

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                  const GemmArgs a, int mode) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kStages * C::kStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * C::kStages + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * C::kStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::kStages + 4);
  CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + C::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kCtlOffset + 16);
  int32_t* tab = reinterpret_cast<int32_t*>(smem + C::kTablesOffset);
  Tables t{tab, tab + (kGroupedMaxExperts + 1), tab + 2 * (kGroupedMaxExperts + 1)};
  __shared__ int32_t s_units;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool grouped = (mode == kGrouped || mode == kGroupedCombine);
  const int64_t atoms_per_rowtile = a.K >> 6;
  const int nkb = static_cast<int>((a.K + kBK - 1) / kBK);
  const int tiles_x = (a.rows_x + 127) >> 7;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(accf_bar(b), 1); mbar_init(acce_bar(b), 128); }
    mbar_init(drain_bar, 1);
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
      const int mtiles = a.n_out >> 7;
      int32_t su = 0, st = 0;
      bool ok = true;
      for (int e = e0; e < e1; ++e) {
        const int32_t o0 = a.expert_offsets[e], o1 = a.expert_offsets[e + 1];
        const int32_t c = o1 - o0;
        ok = ok && (c >= 0);
        t.off[e] = o0;
        su += mtiles * ((c + BN - 1) / BN);
        st += (c + 127) >> 7;
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
        const int32_t c = a.expert_offsets[e + 1] - a.expert_offsets[e];
        t.up[e] = pu; t.tb[e] = pt;
        pu += mtiles * ((c + BN - 1) / BN);
        pt += (c + 127) >> 7;
      }
      const bool all_ok = __all_sync(0xFFFFFFFFu, ok);
      if (lane == 31) {
        const int32_t oE = a.expert_offsets[E];
        t.off[E] = oE;
        t.up[E] = iu;
        t.tb[E] = it;
        const bool good = all_ok && a.expert_offsets[0] == 0 && oE <= a.rows_y;
        if (!good) raise_status(a.status, NVFP4_ERR_DEVICE_CHECK);
        s_units = good ? iu : 0;
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
    if (lane == 0) {
      const uint64_t pol_x = grouped ? l2_policy_evict_first() : l2_policy_evict_last();
      const uint64_t pol_y = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
        const Unit un = get_unit<BN>(u, mode, a, t, tiles_x, atoms_per_rowtile);
        const int ybox = (un.y_rows + 15) >> 4;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, ctl, a.status)) { alive = false; break; }
          const int ksteps = min(4, static_cast<int>((a.K >> 6) - 4 * kb));
          const uint32_t sx = sbase + stage * C::kStageBytes;
          const uint32_t sy = sx + kXTileBytes;
          const uint32_t ssfx = sy + C::kYTileBytes;
          const uint32_t ssfy = ssfx + kSFStageBytes;
          const uint32_t bytes = kXTileBytes + ybox * 16 * kRowBytes + 2 * ksteps * 512;
          mbar_arrive_expect_tx(full_bar(stage), bytes);
          tma_load_2d(sx, &tmx, full_bar(stage), kb * kRowBytes, un.x_row0, pol_x);
          for (int j = 0; j < ybox; ++j)
            tma_load_2d(sy + j * 16 * kRowBytes, &tmy, full_bar(stage), kb * kRowBytes,
                        un.y_row0 + 16 * j, pol_y);
          bulk_load(ssfx, a.sfx + un.sfx_off + kb * kSFStageBytes, ksteps * 512, full_bar(stage),
                    pol_x);
          bulk_load(ssfy, a.sfy + un.sfy_off + kb * kSFStageBytes, ksteps * 512, full_bar(stage),
                    pol_y);
          ++issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // Drain: every copy this thread issued must land before the CTA exits.
      const int64_t first = issued > C::kStages ? issued - C::kStages : 0;
      for (int64_t n = first; n < issued; ++n)
        mbar_wait_drain(full_bar(static_cast<int>(n % C::kStages)),
                        static_cast<uint32_t>((n / C::kStages) & 1), ctl->timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
        const Unit un = get_unit<BN>(u, mode, a, t, tiles_x, atoms_per_rowtile);
        const uint32_t idesc = idesc_nvf4(static_cast<uint32_t>((un.y_rows + 15) & ~15));
        if (!mbar_wait(acce_bar(abuf), aphase ^ 1u, ctl, a.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + abuf * C::kAccCols;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, ctl, a.status)) { alive = false; break; }
          tc_fence_after();
          const int ksteps = min(4, static_cast<int>((a.K >> 6) - 4 * kb));
          const uint32_t sx = sbase + stage * C::kStageBytes;
          const uint32_t sy = sx + kXTileBytes;
          const uint32_t ssfx = sy + C::kYTileBytes;
          const uint32_t ssfy = ssfx + kSFStageBytes;
          const uint32_t tsfx = tmem + C::kSfColBase + stage * 32;
          const uint32_t tsfy = tsfx + 16;
          const uint64_t dx = sdesc_sw128(sx);
          const uint64_t dy = sdesc_sw128(sy);
          for (int ks = 0; ks < ksteps; ++ks) {
            tc_cp_sf_atom(tsfx + 4 * ks, sdesc_sf_atom(ssfx + 512 * ks));
            tc_cp_sf_atom(tsfy + 4 * ks, sdesc_sf_atom(ssfy + 512 * ks));
            tc_mma_nvf4(d_tmem, dx + 2 * ks, dy + 2 * ks, idesc, tsfx + 4 * ks, tsfy + 4 * ks,
                        (kb | ks) != 0 ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!alive) break;
        tc_commit(accf_bar(abuf));
        abuf ^= 1;
        if (abuf == 0) aphase ^= 1u;
      }
      // Drain: wait for every MMA and copy issued above before teardown.
      tc_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, ctl->timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // tensor-memory lane quarter
    const int row = q * 32 + lane;                // row of the X tile
    int abuf = 0;
    uint32_t aphase = 0;
    const float gy = *a.gy;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit un = get_unit<BN>(u, mode, a, t, tiles_x, atoms_per_rowtile);
      // all lanes wait, then agree, so the warp-collective loads below stay converged
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(accf_bar(abuf), aphase, ctl, a.status))) break;
      tc_fence_after();
      const float alpha = __fmul_rn(grouped ? a.gx[un.e] : a.gx[0], gy);
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + abuf * C::kAccCols;
      const int n_valid = un.y_rows;
      const int xr = un.x_local0 + row;            // output feature / X row
      for (int c0 = 0; c0 < n_valid; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        tmem_ld_wait();
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
        } else if (mode == kDenseRowsY || mode == kGrouped) {
          if (mode == kGrouped || xr < a.rows_x) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + xr;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (j < nc) {
                const int64_t y = un.y_row0 + c0 + j;
                dst[y * a.ldc] = f32_to_bf16_rn(__fmul_rn(__uint_as_float(r[j]), alpha));
              }
            }
          }
        } else {  // kGroupedCombine
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < nc) {
              const int p = un.y_row0 + c0 + j;
              const int tok = a.route_token[p];
              const float w = a.topk_w[static_cast<int64_t>(tok) * a.topk + a.route_slot[p]];
              const float v = __fmul_rn(w, __fmul_rn(__uint_as_float(r[j]), alpha));
              atomicAdd(a.ws + static_cast<int64_t>(tok) * a.n_out + xr, v);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acce_bar(abuf));
      abuf ^= 1;
      if (abuf == 0) aphase ^= 1u;
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

cudaError_t init_gemm_attributes() {
  return cudaFuncSetAttribute(nvfp4_gemm_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<128>::kSmemBytes);
}

cudaError_t launch_gemm(const CUtensorMap& tmx, const CUtensorMap& tmy, const GemmArgs& a,
                        int mode, int sms, cudaStream_t s) {
  int grid = sms;
  if (mode == kDenseRowsX || mode == kDenseRowsY) {
    const int64_t units = ((a.rows_x + 127) / 128) * ((a.rows_y + 127) / 128);
    if (units < grid) grid = static_cast<int>(units);
  }
  if (grid < 1) return cudaSuccess;
  nvfp4_gemm_kernel<128><<<grid, kThreads, Cfg<128>::kSmemBytes, s>>>(tmx, tmy, a, mode);
  return cudaGetLastError();
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
