// MoE grouped GEMM on CTA pairs for 256-route token tiles (prefill shapes):
// each block-scaled MMA spans two SMs (tcgen05 cta_group::2), M = 256 rows of
// an expert's weights (one 128-row weight tile per SM) against N = 256 routes
// of one token tile, of which each SM stages 128 rows.  Per SM and K block
// that is one weight tile plus half a token tile, where the one-SM kernel
// streams the whole 256-row token tile beside every weight tile: the hot
// experts' weight and token tiles are re-read from L2 by many units, and the
// SMs' ingest from L2 sets the pace ("The Tile That Didn't Fit", The Core
// Finding: tile size and shared memory bound the arithmetic intensity; "The
// FP4 Frontier", Finding 5: one persistent grouped GEMM over all experts).
// (For 128-route tiles of the down projection with its FP32 combine, the
// same pairing measured slower than the one-SM kernel, 0.26 vs 0.22 ms at
// 1024 tokens; those stay there.)
//
// Operands are the grouped operand tiles (128 rows x 256 K: 16 KB of codes
// in the 128-byte swizzle, then 2 KB of scale atoms), copied byte for byte as
// TMA boxes over the tile buffers viewed as rows of 128 bytes; rows past a
// buffer's end read zeros.  Token rows past the expert's routes give output
// columns that are never stored.
//
// Roles (352 threads per CTA, clusters of two):
//   warp 0      both CTAs: producer (the scale atoms of this CTA's weight
//               tile and of the token tile, then the weight tile's codes and
//               this CTA's half of the token tile's codes); the atoms
//               complete on the leader's scale barrier, the codes on its full
//               barrier, so the atoms' copies into tensor memory can start
//               while the codes are still arriving;
//   warp 6      leader: scale warp, tcgen05.cp of the stage's atoms into
//               both CTAs' tensor memory;
//   warp 1      both: tensor-memory allocation; leader: MMAs and commits;
//   warps 2-5, 7-10  both: epilogue of this CTA's 128 features, 128 of the
//               tile's columns each group; the share read and handed back,
//               then transposed BF16 stores in route order.
// Every wait is bounded; the pair meets at two cluster barriers before
// tensor memory is freed.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kGpTileRows = 144;                 // an operand tile as 128-byte rows

struct GPairCfg {
  static constexpr int BN = 256;                              // routes per token tile
  static constexpr int kYRows = BN / 2;                       // token rows per CTA
  static constexpr int kYAtoms = BN / 128;                    // 128-row scale atom sets
  // stage: [X codes 16 KB][X scales 2 KB][Y codes, own half][Y scales, all rows]
  static constexpr int kXsf = 16384;
  static constexpr int kY = kXsf + 2048;
  static constexpr int kYsf = kY + kYRows * 128;
  static constexpr int kStageBytes = kYsf + kYAtoms * 2048;
  static_assert(kY % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle alignment");
  static constexpr int kStages = 5;
  static constexpr int kSfColBase = BN;                       // after the accumulator
  // per stage: 4 K steps x (4 columns of X's atom + 4 per Y atom set)
  static constexpr int kSfColsPerStage = 16 + 16 * kYAtoms;
  static_assert(kSfColBase + kStages * kSfColsPerStage <= 512, "tensor memory budget");
  static constexpr int kBarOffset = kStages * kStageBytes;
  // full[S], empty[S], scales_ready[S], acc_full, acc_empty, drain, scales_full[S]
  static constexpr int kBarBytes = 8 * (4 * kStages + 3);
  static constexpr int kCtlOffset = kBarOffset + kBarBytes;
  static constexpr int kTablesOffset = kCtlOffset + 64;
  static constexpr int kTableInts = 3 * (kGroupedMaxExperts + 1);
  static constexpr int kSmemBytes = kTablesOffset + 4 * kTableInts + 1024;   // + alignment
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr int kThreads = 11 * 32;
  static constexpr int kEpiWarps = 8;
  static constexpr int kGrpCols = BN / 2;                     // columns per epilogue group
};

struct GPairUnit {
  int e;              // expert
  int32_t y_row0;     // first route of the token tile
  int32_t y_rows;     // valid routes (1..BN)
  int32_t x_tile;     // this CTA's weight tile (operand-tile index)
  int32_t x_local0;   // its first output feature
  int32_t y_tile;     // first operand tile of the token tile
};

__device__ __forceinline__ uint32_t gp_cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t gp_n_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// A wait that ignores the abort flag, bounded by the timeout (drains copies
// and MMAs already in flight).
__device__ __forceinline__ void gp_wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1; i < 0x7FFFFFFFu; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 31u) == 0 && globaltimer() - t0 > timeout) return;
  }
}

// 32 x 32 transpose within a warp: lane l's r[i] becomes lane i's r[l].
__device__ __forceinline__ void gp_transpose32(uint32_t (&r)[32], int lane) {
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

// Unit u of the work list: expert e (binary search of the unit prefix), pair
// of weight tiles mp (this CTA takes tile 2 mp + rank), token tile nt.
__device__ __forceinline__ GPairUnit gp_unit(int u, const GemmArgs& a, const int32_t* up,
                                             const int32_t* off, const int32_t* tb,
                                             uint32_t rank) {
  constexpr int BN = GPairCfg::BN;
  int lo = 0, hi = a.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (up[mid] <= u) lo = mid; else hi = mid;
  }
  GPairUnit un;
  un.e = lo;
  const int mpairs = a.n_out >> 8;
  const int local = u - up[lo];
  const int mp = local % mpairs, nt = local / mpairs;
  const int cnt = off[lo + 1] - off[lo];
  un.y_row0 = off[lo] + nt * BN;
  un.y_rows = min(BN, cnt - nt * BN);
  un.x_local0 = (2 * mp + static_cast<int>(rank)) * 128;
  un.x_tile = lo * (a.n_out >> 7) + 2 * mp + static_cast<int>(rank);
  un.y_tile = tb[lo] + nt * (BN / 128);
  return un;
}

__global__ void __launch_bounds__(GPairCfg::kThreads, 1)
nvfp4_grouped_pair_kernel(const __grid_constant__ CUtensorMap tmx,   // weight tiles, 128-row boxes
                          const __grid_constant__ CUtensorMap tmxs,  // weight tiles, 16-row boxes
                          const __grid_constant__ CUtensorMap tmy,   // token tiles, 128-row boxes
                          const __grid_constant__ CUtensorMap tms,   // token tiles, 16-row boxes
                          const GemmArgs a) {
  using C = GPairCfg;
  constexpr int BN = C::BN;
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
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(smem + C::kCtlOffset + 20);
  int32_t* s_units = reinterpret_cast<int32_t*>(smem + C::kCtlOffset + 24);
  int32_t* up = reinterpret_cast<int32_t*>(smem + C::kTablesOffset);
  int32_t* off = up + (kGroupedMaxExperts + 1);
  int32_t* tb = off + (kGroupedMaxExperts + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(gp_cluster_id_x());
  const int npairs = static_cast<int>(gp_n_clusters_x());
  const int k64 = static_cast<int>(a.K >> 6);
  const int nkb = (k64 + 3) >> 2;

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
  // Work list (both CTAs alike): per expert, (n_out / 256) weight-tile pairs
  // times its token tiles of 256 routes; operand tiles of 128 routes.
  if (warp == 2) {
    const int E = a.E;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    const int mpairs = a.n_out >> 8;
    for (int i = lane; i <= E; i += 32) off[i] = a.expert_offsets[i];
    __syncwarp();
    int32_t su = 0, st = 0;
    bool ok = true;
    for (int e = e0; e < e1; ++e) {
      const int32_t c = off[e + 1] - off[e];
      ok = ok && (c >= 0);
      su += mpairs * ((c + BN - 1) / BN);
      st += (c + 127) / 128;
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
      const int32_t c = off[e + 1] - off[e];
      up[e] = pu;
      tb[e] = pt;
      pu += mpairs * ((c + BN - 1) / BN);
      pt += (c + 127) / 128;
    }
    const bool all_ok = __all_sync(0xFFFFFFFFu, ok);
    if (lane == 31) {
      up[E] = iu;
      tb[E] = it;
      const bool good = all_ok && off[0] == 0 && off[E] <= a.rows_y;
      if (!good && leader) raise_status(a.status, NVFP4_ERR_DEVICE_CHECK);
      *s_units = good ? iu : 0;
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // both CTAs' barriers and tables exist before any copy, commit or remote
  // arrival of the other CTA can reach them
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int units = *s_units;
  uint32_t issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Weight tiles of an expert with one token tile are read once and stream
    // through L2 (evict first); with more token tiles the others read them
    // again (normal).  Token tiles are read by all of the expert's
    // weight-tile pairs (evict last).
    const uint64_t pol_once = l2_policy_evict_first();
    const uint64_t pol_again = l2_policy_evict_normal();
    const uint64_t pol_y = l2_policy_evict_last();
    const uint32_t full_leader = mapa_shared(full_bar(0), 0);
    const uint32_t sff_leader = mapa_shared(sff_bar(0), 0);
    int stage = 0;
    uint32_t phase = 0;
    bool alive = true;
    for (int u = pair; u < units && alive; u += npairs) {
      const GPairUnit un = gp_unit(u, a, up, off, tb, rank);
      const uint64_t pol_x = (off[un.e + 1] - off[un.e] > BN) ? pol_again : pol_once;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_bar(stage), phase ^ 1u, ctl, a.status))) {
          alive = false;
          break;
        }
        if ((a.debug_flags & kDebugSkipFirstStage) && issued == 0) {
          // test hook: stage 0 never fills; its waits end by their time limit
          ++issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
          continue;
        }
        const uint32_t sx = sbase + stage * C::kStageBytes;
        const uint32_t fb = full_leader + 8u * stage;
        const uint32_t sfb = sff_leader + 8u * stage;
        if (leader) {
          mbar_arrive_expect_tx_elect(sff_bar(stage), 2 * 2048 * (1 + C::kYAtoms));
          mbar_arrive_expect_tx_elect(full_bar(stage), 2 * (16384 + C::kYRows * 128));
        }
        // the scale rows (rows 128-143 of each operand tile) first, then the codes
        const int32_t xt_row = (un.x_tile * nkb + kb) * kGpTileRows;
        tma_load_2d_pair_elect(sx + C::kXsf, &tmxs, sfb, 0, xt_row + 128, pol_x);
#pragma unroll
        for (int j = 0; j < C::kYAtoms; ++j)
          tma_load_2d_pair_elect(sx + C::kYsf + 2048 * j, &tms, sfb, 0,
                                 ((un.y_tile + j) * nkb + kb) * kGpTileRows + 128, pol_y);
        tma_load_2d_pair_elect(sx, &tmx, fb, 0, xt_row, pol_x);
        // this CTA's half of the token tile: operand tile y_tile + rank
        tma_load_2d_pair_elect(sx + C::kY, &tmy, fb, 0,
                               ((un.y_tile + static_cast<int>(rank)) * nkb + kb) * kGpTileRows,
                               pol_y);
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
          const int ksteps = min(4, k64 - 4 * kb);
          const uint32_t sx = sbase + stage * C::kStageBytes;
          const uint32_t tsfx = tmem + C::kSfColBase + stage * C::kSfColsPerStage;
          const uint32_t tsfy = tsfx + 16;
          for (int ks = 0; ks < ksteps; ++ks) {
            tc_cp_sf_atom_pair_elect(tsfx + 4 * ks, sdesc_sf_atom(sx + C::kXsf + 512 * ks));
#pragma unroll
            for (int j = 0; j < C::kYAtoms; ++j)
              tc_cp_sf_atom_pair_elect(tsfy + 4 * C::kYAtoms * ks + 4 * j,
                                       sdesc_sf_atom(sx + C::kYsf + 2048 * j + 512 * ks));
          }
          // the MMA warp issues after this arrive and its after-sync fence
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
      const uint32_t idesc = idesc_nvf4_m(256, BN);
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
          const int ksteps = min(4, k64 - 4 * kb);
          const uint32_t sx = sbase + stage * C::kStageBytes;
          const uint32_t tsfx = tmem + C::kSfColBase + stage * C::kSfColsPerStage;
          const uint32_t tsfy = tsfx + 16;
          const uint64_t dx = sdesc_sw128(sx);
          const uint64_t dy = sdesc_sw128(sx + C::kY);
          for (int ks = 0; ks < ksteps; ++ks)
            tc_mma_nvf4_pair_elect(tmem, dx + 2 * ks, dy + 2 * ks, idesc, tsfx + 4 * ks,
                                   tsfy + 4 * C::kYAtoms * ks, (kb > 0 || ks > 0) ? 1u : 0u);
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
    if (lane == 0) gp_wait_drain(drain_bar, 0, ctl->timeout_ns);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // BF16 in route order: the share read and converted, the accumulator
    // handed back (a cluster-scope release, before any store of this unit),
    // then the stores, which overlap the next unit's MMAs.
    constexpr int kChunks = C::kGrpCols / 32;
    const int q = warp & 3;                           // tensor-memory lane quarter
    const int gc0 = warp >= 7 ? C::kGrpCols : 0;      // this group's token columns
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acce_leader = mapa_shared(acce_bar, 0);
    const float gy = *a.gy;
    uint32_t aphase = 0;
    for (int u = pair; u < units; u += npairs) {
      const GPairUnit un = gp_unit(u, a, up, off, tb, rank);
      const int n_valid = un.y_rows;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_sleepy(accf_bar, aphase, ctl, a.status))) break;
      tc_fence_after();
      const float alpha = __fmul_rn(a.gx[un.e], gy);
      const int f0 = un.x_local0 + q * 32;            // first feature of this warp
      const uint32_t taddr = tmem + lane_base + gc0;
      uint32_t pk[kChunks][16];
#pragma unroll
      for (int ci = 0; ci < kChunks; ++ci) {
        if (gc0 + ci * 32 < n_valid) {
          uint32_t r[32];
          tmem_ld32(taddr + ci * 32, r);
          tmem_ld_wait();
          gp_transpose32(r, lane);
#pragma unroll
          for (int h = 0; h < 16; ++h)
            pk[ci][h] = static_cast<uint32_t>(
                            f32_to_bf16_rn(__fmul_rn(__uint_as_float(r[2 * h]), alpha))) |
                        (static_cast<uint32_t>(
                             f32_to_bf16_rn(__fmul_rn(__uint_as_float(r[2 * h + 1]), alpha)))
                         << 16);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_leader);
      aphase ^= 1u;
#pragma unroll
      for (int ci = 0; ci < kChunks; ++ci) {
        const int col = gc0 + ci * 32 + lane;
        if (col < n_valid) {
          uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) +
                          static_cast<int64_t>(un.y_row0 + col) * a.ldc + f0;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            reinterpret_cast<uint4*>(dst)[v] = make_uint4(pk[ci][4 * v], pk[ci][4 * v + 1],
                                                          pk[ci][4 * v + 2], pk[ci][4 * v + 3]);
        }
      }
    }
  }

  // Teardown.  Every copy either producer issued completes on the leader's
  // full barriers: after the first cluster barrier the leader knows both
  // producers' counts and waits for the last stages; then the pair frees its
  // tensor memory together.
  tc_fence_before();
  cluster_sync_all();
  if (leader && warp == 0 && lane == 0) {
    const uint32_t n = issued > *peer_issued ? issued : *peer_issued;
    const uint32_t first = n > static_cast<uint32_t>(C::kStages) ? n - C::kStages : 0u;
    for (uint32_t i = first; i < n; ++i) {
      gp_wait_drain(sff_bar(static_cast<int>(i % C::kStages)), (i / C::kStages) & 1u,
                    ctl->timeout_ns);
      gp_wait_drain(full_bar(static_cast<int>(i % C::kStages)), (i / C::kStages) & 1u,
                    ctl->timeout_ns);
    }
  }
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Pairs the GPU holds at once with this kernel's shared memory (cached).
int gp_max_pairs() {
  static int cached = 0;
  if (cached == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(GPairCfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = GPairCfg::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, nvfp4_grouped_pair_kernel, &cfg) != cudaSuccess ||
        n < 1)
      n = 1;
    cached = n;
  }
  return cached;
}

}  // namespace

cudaError_t init_grouped_pair_attributes() {
  return cudaFuncSetAttribute(nvfp4_grouped_pair_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, GPairCfg::kSmemBytes);
}

int grouped_pair_width(const GemmArgs& a, int mode) {
  if (a.x_map || a.sparse_w || (a.n_out & 255) != 0 || mode != kGrouped) return 0;
  return grouped_tile_width(a.rows_y, a.E) == GPairCfg::BN ? GPairCfg::BN : 0;
}

cudaError_t launch_grouped_pair(const GroupedPairMaps& m, const GemmArgs& a, int mode,
                                cudaStream_t s) {
  if (grouped_pair_width(a, mode) != GPairCfg::BN) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * gp_max_pairs(), 1, 1);
  cfg.blockDim = dim3(GPairCfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = GPairCfg::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, nvfp4_grouped_pair_kernel, m.x_codes, m.x_scales, m.y_codes,
                            m.y_scales,
                            a);
}

}  // namespace nvfp4
