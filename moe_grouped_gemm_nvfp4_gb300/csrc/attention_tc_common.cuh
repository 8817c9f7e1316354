// Device helpers shared by the tensor-core decode-attention kernels
// (attention_tc.cu: heads of 64 and 128; attention_tc_wide.cu: heads of 256
// and 512): the exact E2M1 x E4M3 -> FP16 expansion of NVFP4 cache rows, the
// 128-byte swizzle of K-major operand rows, bounded mbarrier waits, work-item
// decoding and the softmax warps' named-barrier reductions.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "attention.h"

namespace nvfp4 {
namespace {

constexpr int kTile = 128;               // cached tokens per tile
constexpr float kLog2eTc = 1.4426950408889634f;

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two E2M1 codes (low nibble first) -> FP16x2, exactly.
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h) : "r"(byte & 0xFFu));
  return h;
}

// One E4M3 scale byte -> FP16x2 (the scale in both halves), exactly.
__device__ __forceinline__ uint32_t e4m3_f16x2_dup(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h) : "r"((byte & 0xFFu) * 0x101u));
  return h;
}

// 16 NVFP4 values (8 code bytes) times their block scale -> two 16-byte
// chunks of 8 FP16 values each.
__device__ __forceinline__ void expand16(uint32_t c0, uint32_t c1, uint32_t sbyte, uint4& lo,
                                         uint4& hi) {
  const uint32_t s2 = e4m3_f16x2_dup(sbyte);
  lo.x = hmul2_bits(e2m1x2_f16x2(c0), s2);
  lo.y = hmul2_bits(e2m1x2_f16x2(c0 >> 8), s2);
  lo.z = hmul2_bits(e2m1x2_f16x2(c0 >> 16), s2);
  lo.w = hmul2_bits(e2m1x2_f16x2(c0 >> 24), s2);
  hi.x = hmul2_bits(e2m1x2_f16x2(c1), s2);
  hi.y = hmul2_bits(e2m1x2_f16x2(c1 >> 8), s2);
  hi.z = hmul2_bits(e2m1x2_f16x2(c1 >> 16), s2);
  hi.w = hmul2_bits(e2m1x2_f16x2(c1 >> 24), s2);
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a K-major 128-byte
// swizzled block (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint32_t kmajor_chunk(int r, int c) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
}

// Wait for an mbarrier phase, bounded; false after the time limit.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1; i < 0x7FFFFFFFu; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
  return false;
}

// bar.red over the softmax warps (named barrier 1): every one of them
// arrives whether or not its own waits succeeded, so none is left behind.
__device__ __forceinline__ bool softmax_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)) : "memory");
  return r != 0;
}

__device__ __forceinline__ bool softmax_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)) : "memory");
  return r != 0;
}

struct WsItem {
  int split, j, b;
  int64_t t0, t1, row0;
  bool bad_len;
};

// Prefetch loads: volatile, so that the compiler issues them where they are
// written (one work item ahead) instead of next to their first use.
__device__ __forceinline__ int ld_prefetch_s32(const int32_t* p) {
  int v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_prefetch_u16(const uint16_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Work item w as (split, KV head, sequence), in 32-bit arithmetic: the
// items number fewer than 2^31 / 128 (fewer than 2^31 cache rows, at least
// 128 tokens per split), and a 64-bit division costs every role hundreds of
// cycles at each item boundary.
struct WsIdx {
  uint32_t split, j, b;
};
__device__ __forceinline__ WsIdx ws_idx(const AttnArgs& a, int64_t w) {
  const uint32_t wu = static_cast<uint32_t>(w), ns = static_cast<uint32_t>(a.splits);
  const uint32_t q = wu / ns;
  return WsIdx{wu - q * ns, q % static_cast<uint32_t>(a.Hkv), q / static_cast<uint32_t>(a.Hkv)};
}

// The sequence length work item w reads (prefetched one item ahead by every
// role, so that its latency stays off the item boundary).
__device__ __forceinline__ int ws_len(const AttnArgs& a, int64_t w, int64_t items) {
  if (w >= items) return 0;
  return ld_prefetch_s32(a.seq_lens + ws_idx(a, w).b);
}

__device__ __forceinline__ WsItem ws_item(const AttnArgs& a, int64_t w, int n) {
  WsItem it;
  const WsIdx x = ws_idx(a, w);
  it.split = static_cast<int>(x.split);
  it.j = static_cast<int>(x.j);
  it.b = static_cast<int>(x.b);
  it.bad_len = n < 0 || n > a.L_max;
  if (it.bad_len) n = 0;
  it.t0 = static_cast<int64_t>(it.split) * a.chunk;
  it.t1 = min(static_cast<int64_t>(n), it.t0 + a.chunk);
  it.row0 = (static_cast<int64_t>(it.b) * a.Hkv + it.j) * a.L_max;
  return it;
}

// mbarrier wait that suspends the thread until the phase completes or about
// `hint_ns` pass, instead of spinning on the issue slots the expansion needs.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

// Bounded wait of the pipelined kernel: false when another role has aborted
// or after the control block's time limit (then NVFP4_ERR_TIMEOUT).
__device__ __forceinline__ bool ws_wait(uint32_t bar, uint32_t parity, CtaCtl* ctl, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t k = 0; k < 0x7FFFFFFFu; ++k) {
    if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
    if (*reinterpret_cast<volatile uint32_t*>(&ctl->abort)) return false;
    if (globaltimer() - t0 > ctl->timeout_ns) break;
  }
  *reinterpret_cast<volatile uint32_t*>(&ctl->abort) = 1u;
  raise_status(status, NVFP4_ERR_TIMEOUT);
  return false;
}

// Bounded wait that ignores the abort flag: used to drain copies and MMAs in
// flight before the CTA frees its shared and tensor memory.
__device__ __forceinline__ void ws_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  (void)tc_wait(bar, parity, limit_ns);
}

__device__ __forceinline__ void mbar_arrive_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}"
      :: "r"(bar) : "memory");
}

}  // namespace
}  // namespace nvfp4
