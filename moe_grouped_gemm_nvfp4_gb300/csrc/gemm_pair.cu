// NVFP4 single GEMM on CTA pairs: each block-scaled MMA spans two SMs
// (tcgen05 cta_group::2), M = 256 rows of A split 128 + 128 over the pair and
// the 256 rows of B split the same way, so each SM stages 128 rows of A and
// 128 rows of B per K block for a 128 x 256 share of the output -- two thirds
// of the bytes a one-SM 128 x 256 tile moves ("The Tile That Didn't Fit",
// The Core Finding: tile size and shared memory bound the arithmetic
// intensity of the large FP4 GEMM; on this part the pair of SMs is what
// enlarges the tile).
//
// Roles (352 threads per CTA, one CTA per SM, clusters of two):
//   warp 0      both CTAs: TMA producer.  A's and B's scale atoms, then A
//               rows and B rows, into this CTA's stage; every copy completes
//               on a barrier of the leader CTA (the leader expects both CTAs'
//               bytes): the atoms on the stage's scale barrier, the codes on
//               its full barrier, so the atoms' copies into tensor memory can
//               start while the codes are still arriving;
//   warp 6      leader: scale warp, tcgen05.cp of the stage's scale atoms
//               into both CTAs' tensor memory (each from its own shared
//               memory: A's scales of its own rows, all 256 rows of B's);
//   warp 1      both: tensor-memory allocation for the pair; leader: the
//               MMAs (M 256, N 256, K 64) and the commits that release each
//               stage and the accumulator in both CTAs;
//   warps 2-5, 7-10  both: epilogue of this CTA's 128 rows, columns 0-127
//               and 128-255; the accumulator goes back to the leader's MMA
//               warp by remote arrivals once both CTAs have read it.
// Every wait is bounded; the pair meets at two cluster barriers before
// tensor memory is freed.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kPRowBytes = 128;                  // 256 FP4 values of one row per stage
constexpr int kPCodeBytes = 128 * kPRowBytes;    // 128 rows: 16 KB
constexpr int kPSfBytes = 4 * 512;               // four scale atoms: 128 rows x 256 K

struct PairCfg {
  static constexpr int kStages = 5;
  // stage: [A codes, own 128 rows][A scales][B codes, own 128 rows][B scales, all 256 rows]
  static constexpr int kXsf = kPCodeBytes;
  static constexpr int kY = kXsf + kPSfBytes;
  static constexpr int kYsf = kY + kPCodeBytes;
  static constexpr int kStageBytes = kYsf + 2 * kPSfBytes;
  static_assert(kY % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle alignment");
  static constexpr int kBarOffset = kStages * kStageBytes;
  // full[S], empty[S], scales_ready[S], acc_full, acc_empty, drain, scales_full[S]
  static constexpr int kBarBytes = 8 * (4 * kStages + 3);
  static constexpr int kCtlOffset = kBarOffset + kBarBytes;
  static constexpr int kSmemBytes = kCtlOffset + 64 + 1024;     // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr int kThreads = 11 * 32;
  static constexpr int kEpiWarps = 8;
  static constexpr int kAccCols = 256;
  // scale columns after the accumulator: per stage 4 K steps x (4 for A's
  // atom + 8 for B's two atoms)
  static constexpr int kSfColBase = kAccCols;
  static constexpr int kSfColsPerStage = 16 + 32;
  static_assert(kSfColBase + kStages * kSfColsPerStage <= 512, "tensor memory budget");
};

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t n_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Waits for a phase regardless of the abort flag, bounded by the timeout
// (draining copies and MMAs already in flight).
__device__ __forceinline__ bool pair_wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1; i < 0x7FFFFFFFu; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0 && globaltimer() - t0 > timeout) return false;
  }
  return false;
}

__global__ void __launch_bounds__(PairCfg::kThreads, 1)
nvfp4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmx,
                       const __grid_constant__ CUtensorMap tmy,
                       const __grid_constant__ CUtensorMap tsx,
                       const __grid_constant__ CUtensorMap tsy, const GemmArgs a) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kBarOffset;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  auto sfr_bar = [&](int s) { return bar0 + 8u * (2 * C::kStages + s); };
  const uint32_t accf_bar = bar0 + 8u * (3 * C::kStages);
  const uint32_t acce_bar = accf_bar + 8u;
  const uint32_t drain_bar = accf_bar + 16u;
  // scale atoms landed (both CTAs'), apart from the codes so that their
  // copies into tensor memory run while the codes are still arriving
  auto sff_bar = [&](int s) { return bar0 + 8u * (3 * C::kStages + 3 + s); };
  CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + C::kCtlOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kCtlOffset + 16);
  // stages issued by the other CTA's producer (written there into the leader)
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(smem + C::kCtlOffset + 20);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(n_clusters_x());
  const int64_t apr = a.K >> 6;                         // scale atoms per 128-row tile
  const int nkb = static_cast<int>((a.K + 255) >> 8);
  const int tiles_m = (a.rows_x + 255) >> 8;
  const int tiles_n = (a.rows_y + 255) >> 8;
  const int units = tiles_m * tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sfr_bar(s), 1);
      mbar_init(sff_bar(s), 1);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, 2 * C::kEpiWarps);   // every epilogue warp of both CTAs
    mbar_init(drain_bar, 2);                 // the leader's MMA and scale warps
    ctl->abort = 0;
    ctl->timeout_ns = a.timeout_ns;
    *peer_issued = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // both CTAs' barriers exist before any copy, commit or remote arrival
  // of the other CTA can reach them
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_policy_evict_last();    // every operand row is read by many tiles
    const uint32_t full_leader = mapa_shared(full_bar(0), 0);
    const uint32_t sff_leader = mapa_shared(sff_bar(0), 0);
    int stage = 0;
    uint32_t phase = 0;
    bool alive = true;
    for (int u = pair; u < units && alive; u += npairs) {
      const int tm = u % tiles_m, tn = u / tiles_m;
      const int xrow = tm * 256 + 128 * static_cast<int>(rank);   // this CTA's A rows
      const int yrow = tn * 256 + 128 * static_cast<int>(rank);   // this CTA's half of B
      const int64_t xs = (2 * tm + rank) * apr;                   // its A scale atoms
      const int64_t ys = (2 * tn) * apr;                          // all of B's (two row tiles)
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_bar(stage), phase ^ 1u, ctl, a.status))) {
          alive = false;
          break;
        }
        const uint32_t sx = sbase + stage * C::kStageBytes;
        const uint32_t fb = full_leader + 8u * stage;
        const uint32_t sfb = sff_leader + 8u * stage;
        if (leader) {
          mbar_arrive_expect_tx_elect(sff_bar(stage), 2 * 3 * kPSfBytes);
          mbar_arrive_expect_tx_elect(full_bar(stage), 2 * 2 * kPCodeBytes);
        }
        tma_load_2d_pair_elect(sx + C::kXsf, &tsx, sfb, 0, static_cast<int32_t>(xs + 4 * kb), pol);
        tma_load_2d_pair_elect(sx + C::kYsf, &tsy, sfb, 0, static_cast<int32_t>(ys + 4 * kb), pol);
        tma_load_2d_pair_elect(sx + C::kYsf + kPSfBytes, &tsy, sfb, 0,
                               static_cast<int32_t>(ys + apr + 4 * kb), pol);
        tma_load_2d_pair_elect(sx, &tmx, fb, kb * kPRowBytes, xrow, pol);
        tma_load_2d_pair_elect(sx + C::kY, &tmy, fb, kb * kPRowBytes, yrow, pol);
        ++issued;
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!leader && lane == 0)
      st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(peer_issued)), 0), issued);
    __syncwarp();
  } else if (warp == 6) {
    // ---------------------------------------------------------- scale warp
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      bool alive = true;
      for (int u = pair; u < units && alive; u += npairs) {
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(sff_bar(stage), phase, ctl, a.status))) {
            alive = false;
            break;
          }
          const int ksteps = min(4, static_cast<int>(apr - 4 * kb));
          const uint32_t sx = sbase + stage * C::kStageBytes;
          const uint32_t tsfx = tmem + C::kSfColBase + stage * C::kSfColsPerStage;
          const uint32_t tsfy = tsfx + 16;
          for (int ks = 0; ks < ksteps; ++ks) {
            tc_cp_sf_atom_pair_elect(tsfx + 4 * ks, sdesc_sf_atom(sx + C::kXsf + 512 * ks));
            tc_cp_sf_atom_pair_elect(tsfy + 8 * ks, sdesc_sf_atom(sx + C::kYsf + 512 * ks));
            tc_cp_sf_atom_pair_elect(tsfy + 8 * ks + 4,
                                     sdesc_sf_atom(sx + C::kYsf + kPSfBytes + 512 * ks));
          }
          // the MMA warp issues after this arrive and its after-sync fence;
          // copies followed by MMAs that read their columns run in order
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sfr_bar(stage));
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      tc_commit_pair_elect(drain_bar);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (leader) {
      const uint32_t idesc = idesc_nvf4_m(256, 256);
      int stage = 0;
      uint32_t phase = 0, aphase = 0;
      bool alive = true;
      for (int u = pair; u < units && alive; u += npairs) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(acce_bar, aphase ^ 1u, ctl, a.status))) break;
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(sfr_bar(stage), phase, ctl, a.status) &&
                                           mbar_wait(full_bar(stage), phase, ctl, a.status))) {
            alive = false;
            break;
          }
          tc_fence_after();
          const int ksteps = min(4, static_cast<int>(apr - 4 * kb));
          const uint32_t sx = sbase + stage * C::kStageBytes;
          const uint32_t tsfx = tmem + C::kSfColBase + stage * C::kSfColsPerStage;
          const uint32_t tsfy = tsfx + 16;
          const uint64_t dx = sdesc_sw128(sx);
          const uint64_t dy = sdesc_sw128(sx + C::kY);
          for (int ks = 0; ks < ksteps; ++ks)
            tc_mma_nvf4_pair_elect(tmem, dx + 2 * ks, dy + 2 * ks, idesc, tsfx + 4 * ks,
                                   tsfy + 8 * ks, (kb > 0 || ks > 0) ? 1u : 0u);
          tc_commit_pair_elect(empty_bar(stage));      // the stage is free in both CTAs
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!alive) break;
        tc_commit_pair_elect(accf_bar);                // the accumulator is full in both
        aphase ^= 1u;
      }
      tc_commit_pair_elect(drain_bar);
    }
    // both CTAs: the leader's MMAs and scale copies (which write this CTA's
    // tensor memory and read its shared memory) have completed
    if (lane == 0) pair_wait_drain(drain_bar, 0, ctl->timeout_ns);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // tensor-memory lane quarter
    const int gc0 = warp >= 7 ? 128 : 0;          // this group's accumulator columns
    const int row = q * 32 + lane;
    const uint32_t acce_leader = mapa_shared(acce_bar, 0);
    const float alpha = __fmul_rn(a.gx[0], *a.gy);
    uint32_t aphase = 0;
    for (int u = pair; u < units; u += npairs) {
      const int tm = u % tiles_m, tn = u / tiles_m;
      const int n_valid = min(256, a.rows_y - tn * 256);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_sleepy(accf_bar, aphase, ctl, a.status))) break;
      tc_fence_after();
      // read this warp's 32 rows x 128 columns as BF16, hand the accumulator
      // back, then store (the stores overlap the next tile's MMAs)
      uint32_t pk[4][16];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + gc0;
#pragma unroll
      for (int cp2 = 0; cp2 < 2; ++cp2) {
        if (gc0 + cp2 * 64 < n_valid) {
          uint32_t r[2][32];
          tmem_ld32(taddr + cp2 * 64, r[0]);
          tmem_ld32(taddr + cp2 * 64 + 32, r[1]);
          tmem_ld_wait();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int h = 0; h < 16; ++h)
              pk[2 * cp2 + hh][h] =
                  static_cast<uint32_t>(
                      f32_to_bf16_rn(__fmul_rn(__uint_as_float(r[hh][2 * h]), alpha))) |
                  (static_cast<uint32_t>(
                       f32_to_bf16_rn(__fmul_rn(__uint_as_float(r[hh][2 * h + 1]), alpha)))
                   << 16);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_leader);
      aphase ^= 1u;
      const int xr = tm * 256 + 128 * static_cast<int>(rank) + row;
      if (xr < a.rows_x) {
#pragma unroll
        for (int ci = 0; ci < 4; ++ci) {
          const int c0 = gc0 + ci * 32;
          if (c0 >= n_valid) continue;
          uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + static_cast<int64_t>(xr) * a.ldc +
                          tn * 256 + c0;
          const int lim = min(32, n_valid - c0);
          if (lim == 32 && a.vec_store) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              reinterpret_cast<uint4*>(dst)[v] = make_uint4(pk[ci][4 * v], pk[ci][4 * v + 1],
                                                            pk[ci][4 * v + 2], pk[ci][4 * v + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < lim) dst[i] = static_cast<uint16_t>(pk[ci][i >> 1] >> (16 * (i & 1)));
          }
        }
      }
    }
  }

  // Teardown.  Every copy either producer issued completes on the leader's
  // scale and full barriers: after the first cluster barrier the leader knows both
  // producers' counts and waits for the last stages (already complete when
  // nothing aborted); then the pair frees its tensor memory together.
  tc_fence_before();
  cluster_sync_all();
  if (leader && warp == 0 && lane == 0) {
    const uint32_t n = issued > *peer_issued ? issued : *peer_issued;
    const uint32_t first = n > static_cast<uint32_t>(C::kStages) ? n - C::kStages : 0u;
    for (uint32_t i = first; i < n; ++i) {
      pair_wait_drain(sff_bar(static_cast<int>(i % C::kStages)),
                      (i / C::kStages) & 1u, ctl->timeout_ns);
      pair_wait_drain(full_bar(static_cast<int>(i % C::kStages)),
                      (i / C::kStages) & 1u, ctl->timeout_ns);
    }
  }
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

cudaError_t init_gemm_pair_attributes() {
  return cudaFuncSetAttribute(nvfp4_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PairCfg::kSmemBytes);
}

// Pairs the GPU holds at once with this kernel's shared memory (cached).
static int max_pairs() {
  static int cached = 0;
  if (cached == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(PairCfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, nvfp4_gemm_pair_kernel, &cfg) != cudaSuccess || n < 1)
      n = 1;
    cached = n;
  }
  return cached;
}

cudaError_t launch_gemm_pair(const CUtensorMap& tmx, const CUtensorMap& tmy,
                             const CUtensorMap& tsx, const CUtensorMap& tsy, const GemmArgs& a,
                             cudaStream_t s) {
  const int64_t units = static_cast<int64_t>((a.rows_x + 255) / 256) * ((a.rows_y + 255) / 256);
  int pairs = max_pairs();
  if (units < pairs) pairs = static_cast<int>(units);
  if (pairs < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(PairCfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, nvfp4_gemm_pair_kernel, tmx, tmy, tsx, tsy, a);
}

}  // namespace nvfp4
