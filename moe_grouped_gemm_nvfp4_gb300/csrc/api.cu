// C ABI of the NVFP4 library: argument validation, tensor-map encoding and
// launches on the caller's stream.  See include/nvfp4.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/nvfp4.h"
#include "kernels.h"
#include "attention.h"

namespace {

// Per-device status word of the kernels (first error wins).
__device__ int g_status_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool sm103 = false;
  int sms = 0;
  int* status = nullptr;   // device address of g_status_word
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<uint32_t> g_debug_flags{0u};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

nvfp4_status cuda_fail() {
  cudaGetLastError();   // clear the sticky-free error so later calls can run
  return NVFP4_ERR_CUDA;
}

// Looks up (once per device, with that device current) the SM count, the
// architecture and the device address of the status word, and sets the
// kernels' shared-memory attributes.
nvfp4_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
  if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cuda_fail();
    d.sm103 = (major == 10 && minor == 3);
    d.sms = sms;
    if (d.sm103) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return cuda_fail();
      d.status = static_cast<int*>(p);
      if (nvfp4::init_gemm_attributes() != cudaSuccess) return cuda_fail();
      if (nvfp4::init_gemm_pair_attributes() != cudaSuccess) return cuda_fail();
      if (nvfp4::init_grouped_pair_attributes() != cudaSuccess) return cuda_fail();
      if (nvfp4::init_attention_tc_attributes() != cudaSuccess) return cuda_fail();
      if (nvfp4::init_route_attributes() != cudaSuccess) return cuda_fail();
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return cuda_fail();
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (const char* env = std::getenv("NVFP4_TIMEOUT_NS")) {
      const unsigned long long v = std::strtoull(env, nullptr, 10);
      if (v > 0) g_timeout_ns.store(v);
    }
    d.ready = true;
  }
  if (!d.sm103) return NVFP4_ERR_UNSUPPORTED;
  *out = &d;
  return NVFP4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The grouped activation tiles proper, and the scratch after them that holds
// the tensor amax's per-block maxima between the amax and dispatch kernels.
// Upper bound on the token tiles (layout chunks) of R routes over E experts.
int64_t grouped_token_tiles(int64_t R, int32_t E) {
  const int64_t chunk = nvfp4::grouped_chunk_rows(R, E);
  const int64_t nonempty = R < E ? R : E;
  return (R + (chunk - 1) * nonempty) / chunk;
}

size_t grouped_tiles_body_bytes(int64_t R, int32_t E, int64_t K) {
  return static_cast<size_t>(grouped_token_tiles(R, E)) * static_cast<size_t>((K + 255) / 256) *
         static_cast<size_t>(nvfp4::kOperandTileBytes);
}
constexpr size_t kAmaxScratchBytes = 16384;

// 2-D map over a packed operand [rows, row_bytes] (uint8), box of 128 bytes
// x box_rows rows, 128-byte swizzle.  Out-of-range boxes read zeros.
nvfp4_status make_operand_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes,
                              uint32_t box_rows) {
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED;
}

// 2-D map over a buffer of grouped operand tiles viewed as rows of 128 bytes
// (a tile is 144 such rows: 128 of codes in the 128-byte swizzle, then 16 of
// scale atoms), boxes of box_rows rows, no swizzle, so the tiles land in
// shared memory byte for byte.  Rows past the buffer read zeros.
nvfp4_status make_tile_rows_map(CUtensorMap* m, const void* base, uint64_t rows,
                                uint32_t box_rows) {
  const cuuint64_t dims[2] = {128u, rows};
  const cuuint64_t strides[1] = {128u};
  const cuuint32_t box[2] = {128u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED;
}

// 2-D map over a KV-cache code array [rows, D/2] (uint8) for the tensor-core
// attention: boxes of 128 rows, each the whole row with the swizzle of the row
// width (64 bytes for D = 128, 32 for D = 64) or, for D = 256 and 512, 64
// bytes of it (128 head dimensions) with the 64-byte swizzle.  Rows past the
// array read zeros.
nvfp4_status make_kv_code_map(CUtensorMap* m, const void* base, uint64_t rows, int D) {
  const uint64_t row_bytes = static_cast<uint64_t>(D / 2);
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes < 64 ? row_bytes : 64), 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              D >= 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED;
}

// 2-D map over a KV-cache scale array [rows, D/16] (uint8) for the
// tensor-core attention.  D = 64 and 128: viewed as 16-byte rows, boxes of 128
// cache rows (rows * D/16 a multiple of 16).  D = 256 and 512: the rows as they
// are, boxes of 16 bytes (two slices of 128 dimensions) x 128 rows.  Rows past
// the array read zeros.
nvfp4_status make_kv_scale_map(CUtensorMap* m, const void* base, uint64_t rows, int D) {
  const uint64_t sb = static_cast<uint64_t>(D / 16);
  const bool wide = sb >= 16;                      // rows of 16 or 32 bytes, 16-byte boxes
  const cuuint64_t dims[2] = {wide ? sb : 16u, wide ? rows : rows * sb / 16};
  const cuuint64_t strides[1] = {wide ? sb : 16u};
  const cuuint32_t box[2] = {16u, static_cast<cuuint32_t>(wide ? 128 : 128 * sb / 16)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED;
}

// 2-D map over atom-layout scales of a [rows, K] operand viewed as rows of
// one 512-byte atom (128 32-bit words), box of four atoms (one 256-K block
// of a 128-row tile).  Rows past the last atom read zeros.
nvfp4_status make_scale_map(CUtensorMap* m, const void* base, uint64_t rows, int64_t K) {
  const cuuint64_t dims[2] = {128u, ((rows + 127) / 128) * static_cast<uint64_t>(K / 64)};
  const cuuint64_t strides[1] = {512u};
  const cuuint32_t box[2] = {128u, 4u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
    case NVFP4_ERR_UNSUPPORTED: return "NVFP4_ERR_UNSUPPORTED";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
    case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
    case NVFP4_ERR_DEVICE_CHECK: return "NVFP4_ERR_DEVICE_CHECK";
    default: return "NVFP4_ERR_UNKNOWN";
  }
}

int nvfp4_version(void) { return 100; }

nvfp4_status nvfp4_set_timeout_ns(uint64_t ns) {
  if (ns == 0) return NVFP4_ERR_INVALID_ARG;
  g_timeout_ns.store(ns);
  return NVFP4_OK;
}

nvfp4_status nvfp4_debug_set_flags(uint32_t flags) {
  if (flags & ~nvfp4::kDebugSkipFirstStage) return NVFP4_ERR_INVALID_ARG;
  g_debug_flags.store(flags);
  return NVFP4_OK;
}

nvfp4_status nvfp4_device_status(void* stream, int reset, int* status_out) {
  if (!status_out) return NVFP4_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return cuda_fail();
  if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_fail();
  if (reset) {
    if (cudaMemsetAsync(d->status, 0, sizeof(int), s) != cudaSuccess) return cuda_fail();
    if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_fail();
  }
  *status_out = v;
  return NVFP4_OK;
}

nvfp4_status nvfp4_last_device_status(void* stream) {
  int v = 0;
  const nvfp4_status st = nvfp4_device_status(stream, 0, &v);
  return st != NVFP4_OK ? st : static_cast<nvfp4_status>(v);
}

size_t nvfp4_prepacked_scales_bytes(int64_t rows, int64_t kblk) {
  if (rows < 0 || kblk < 0) return 0;
  return nvfp4_atom_scales_bytes(rows, 16 * ((kblk + 3) / 4 * 4));
}

size_t nvfp4_grouped_gemm_workspace_bytes(int64_t T, int32_t topk, int32_t E, int64_t N,
                                          int64_t K, int32_t combine) {
  if (T < 0 || topk <= 0 || E <= 0 || N < 0 || K < 0) return 0;
  return grouped_tiles_body_bytes(T * topk, E, K) +
         (combine ? nvfp4_combine_workspace_bytes(T, N) : 0);
}

size_t nvfp4_atom_scales_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>(cols / 16);
}

size_t nvfp4_operand_tiles_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((K + 255) / 256) *
         static_cast<size_t>(nvfp4::kOperandTileBytes);
}

int nvfp4_grouped_chunk_rows(int64_t R, int32_t E) {
  return nvfp4::grouped_chunk_rows(R < 0 ? 0 : R, E);
}

size_t nvfp4_grouped_tiles_bytes(int64_t R, int32_t E, int64_t K) {
  if (R < 0 || E < 0 || K < 0) return 0;
  return grouped_tiles_body_bytes(R, E, K) + kAmaxScratchBytes;
}

size_t nvfp4_combine_workspace_bytes(int64_t T, int64_t N) {
  if (T < 0 || N < 0) return 0;
  return static_cast<size_t>(T) * static_cast<size_t>(N) * sizeof(float);
}

nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                            uint8_t* packed, uint8_t* scales, float* global_scale,
                            uint32_t flags, void* stream) {
  if (rows < 0 || cols < 0 || ld < cols) return NVFP4_ERR_INVALID_ARG;
  if (flags & ~(NVFP4_SF_ATOMS | NVFP4_GLOBAL_GIVEN)) return NVFP4_ERR_INVALID_ARG;
  if (!global_scale || (rows > 0 && cols > 0 && (!x || !packed || !scales)))
    return NVFP4_ERR_INVALID_ARG;
  if (cols % 16 != 0 || ld % 8 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((flags & NVFP4_SF_ATOMS) &&
      (cols % 64 != 0 || (scales && (reinterpret_cast<uintptr_t>(scales) & 3u))))
    return NVFP4_ERR_UNSUPPORTED;
  if ((x && !aligned16(x)) || (packed && (reinterpret_cast<uintptr_t>(packed) & 7u)) ||
      (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  if (!(flags & NVFP4_GLOBAL_GIVEN)) {
    if (nvfp4::launch_amax(xb, rows, cols, ld, global_scale, d->sms, s) != cudaSuccess)
      return cuda_fail();
  }
  if (nvfp4::launch_quantize(xb, rows, cols, ld, packed, scales,
                             (flags & NVFP4_SF_ATOMS) ? 1 : 0, global_scale, d->sms, s) !=
      cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_prepack_weights(const uint8_t* scales_rowmajor, int64_t rows, int64_t kblk,
                                   uint8_t* scales_atoms, void* stream) {
  if (rows < 0 || kblk < 0) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && kblk > 0 && (!scales_rowmajor || !scales_atoms)) return NVFP4_ERR_INVALID_ARG;
  if (kblk % 4 != 0) return NVFP4_ERR_UNSUPPORTED;
  if (scales_atoms && (reinterpret_cast<uintptr_t>(scales_atoms) & 3u)) return NVFP4_ERR_UNSUPPORTED;
  if (scales_rowmajor && (reinterpret_cast<uintptr_t>(scales_rowmajor) & 3u))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  if (kblk == 0) return NVFP4_OK;
  if (nvfp4::launch_prepack(scales_rowmajor, rows, kblk, scales_atoms, d->sms,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_gemm(const uint8_t* A, const uint8_t* sfA, const float* gA,
                        const uint8_t* B, const uint8_t* sfB, const float* gB,
                        void* C, int64_t M, int64_t N, int64_t K, int64_t ldc, void* stream) {
  if (!A || !sfA || !gA || !B || !sfB || !gB || !C) return NVFP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || ldc < N) return NVFP4_ERR_INVALID_ARG;
  if (K % 64 != 0) return NVFP4_ERR_UNSUPPORTED;
  if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 31)) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(sfA) || !aligned16(sfB) ||
      (reinterpret_cast<uintptr_t>(C) & 1u))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  // Large M and N: CTA pairs, 256 x 256 tiles with one MMA across two SMs.
  if (M >= 256 && N >= 256) {
    CUtensorMap tmx, tmy, tsx, tsy;
    if (make_operand_map(&tmx, A, M, K / 2, 128) != NVFP4_OK ||
        make_operand_map(&tmy, B, N, K / 2, 128) != NVFP4_OK ||
        make_scale_map(&tsx, sfA, M, K) != NVFP4_OK || make_scale_map(&tsy, sfB, N, K) != NVFP4_OK)
      return NVFP4_ERR_UNSUPPORTED;
    nvfp4::GemmArgs a{};
    a.gx = gA;
    a.gy = gB;
    a.K = K;
    a.rows_x = static_cast<int32_t>(M);
    a.rows_y = static_cast<int32_t>(N);
    a.out = C;
    a.ldc = ldc;
    a.vec_store = (ldc % 8 == 0 && aligned16(C)) ? 1 : 0;
    a.status = d->status;
    a.timeout_ns = g_timeout_ns.load();
    if (nvfp4::launch_gemm_pair(tmx, tmy, tsx, tsy, a, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return cuda_fail();
    return NVFP4_OK;
  }
  // Small M (decode-like): weights on the MMA's M side, tokens on its N side.
  const bool swap = M <= 64;
  const uint8_t* X = swap ? B : A;
  const uint8_t* Y = swap ? A : B;
  const int64_t rows_x = swap ? N : M;
  const int64_t rows_y = swap ? M : N;
  // Y in one box per stage: 256 rows for the 256-wide tiles the launch picks
  // when Y has at least 256 rows (kDenseRowsX), 128 rows when its tiles are
  // full, else 16-row boxes
  const uint32_t ybox_rows = (!swap && rows_y >= 256) ? 256u : (rows_y >= 128 ? 128u : 16u);
  CUtensorMap tmx, tmy;
  if (make_operand_map(&tmx, X, rows_x, K / 2, 128) != NVFP4_OK ||
      make_operand_map(&tmy, Y, rows_y, K / 2, ybox_rows) != NVFP4_OK)
    return NVFP4_ERR_UNSUPPORTED;
  nvfp4::GemmArgs a{};
  a.sfx = swap ? sfB : sfA;
  a.sfy = swap ? sfA : sfB;
  a.gx = swap ? gB : gA;
  a.gy = swap ? gA : gB;
  a.K = K;
  a.rows_x = static_cast<int32_t>(rows_x);
  a.rows_y = static_cast<int32_t>(rows_y);
  a.out = C;
  a.ldc = ldc;
  a.vec_store = (ldc % 8 == 0 && aligned16(C)) ? 1 : 0;
  a.ybox_rows = static_cast<int32_t>(ybox_rows);
  a.status = d->status;
  a.timeout_ns = g_timeout_ns.load();
  a.debug_flags = g_debug_flags.load();
  if (nvfp4::launch_gemm(tmx, tmy, a, swap ? nvfp4::kDenseRowsY : nvfp4::kDenseRowsX, d->sms,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_moe_route(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                             int32_t* expert_offsets, int32_t* route_token, int32_t* route_slot,
                             int32_t* route_pos, void* stream) {
  if (T < 0 || topk <= 0 || E <= 0 || !expert_offsets) return NVFP4_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !route_token || !route_slot)) return NVFP4_ERR_INVALID_ARG;
  if (E > 1024 || T * topk > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  if (nvfp4::launch_route(topk_ids, T, topk, E, expert_offsets, route_token, route_slot,
                          route_pos, d->status, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_prepack_weight_tiles(const uint8_t* packed, const uint8_t* scales_rowmajor,
                                        int64_t rows, int64_t K, uint8_t* tiles, void* stream) {
  if (rows < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && K > 0 && (!packed || !scales_rowmajor || !tiles)) return NVFP4_ERR_INVALID_ARG;
  if (K % 64 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((packed && !aligned16(packed)) || (tiles && !aligned16(tiles)) ||
      (scales_rowmajor && (reinterpret_cast<uintptr_t>(scales_rowmajor) & 3u)))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  if (nvfp4::launch_prepack_tiles(packed, scales_rowmajor, rows, K, tiles, d->sms,
                                  static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_quantize_dispatch(const void* x, int64_t rows, int64_t K, int64_t ld,
                                     const int32_t* route_pos, int32_t fanout,
                                     const int32_t* expert_offsets, int32_t E, int64_t R,
                                     uint8_t* tiles, float* global_scale, uint32_t flags,
                                     void* stream) {
  if (rows < 0 || K <= 0 || ld < K || E <= 0 || R < 0 || fanout <= 0) return NVFP4_ERR_INVALID_ARG;
  if (flags & ~static_cast<uint32_t>(NVFP4_GLOBAL_GIVEN | NVFP4_AMAX_DONE))
    return NVFP4_ERR_INVALID_ARG;
  if ((flags & NVFP4_GLOBAL_GIVEN) && (flags & NVFP4_AMAX_DONE)) return NVFP4_ERR_INVALID_ARG;
  if (!expert_offsets || !global_scale || (rows > 0 && (!x || !tiles)))
    return NVFP4_ERR_INVALID_ARG;
  if (!route_pos && (fanout != 1 || rows != R)) return NVFP4_ERR_INVALID_ARG;
  if (K % 64 != 0 || ld % 8 != 0 || E > 1024) return NVFP4_ERR_UNSUPPORTED;
  if ((x && !aligned16(x)) || (tiles && !aligned16(tiles))) return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  uint32_t* partials = nullptr;
  int n_partials = 0;
  if (!(flags & NVFP4_GLOBAL_GIVEN)) {
    if (rows == 0) {                     // nothing to quantise: g = 0
      if (cudaMemsetAsync(global_scale, 0, sizeof(float), s) != cudaSuccess) return cuda_fail();
      return NVFP4_OK;
    }
    // per-block maxima go to the scratch after the tiles; the dispatch
    // kernel reduces them and stores g
    n_partials = nvfp4::amax_partials_count(rows, K, d->sms);
    if (static_cast<size_t>(n_partials) * sizeof(uint32_t) > kAmaxScratchBytes)
      return NVFP4_ERR_UNSUPPORTED;
    partials = reinterpret_cast<uint32_t*>(tiles + grouped_tiles_body_bytes(R, E, K));
    // NVFP4_AMAX_DONE: nvfp4_amax_partials already left them there
    if (!(flags & NVFP4_AMAX_DONE) &&
        nvfp4::launch_amax_partials(xb, rows, K, ld, partials, d->sms, s) != cudaSuccess)
      return cuda_fail();
  }
  if (nvfp4::launch_quantize_dispatch(xb, rows, K, ld, route_pos, fanout, expert_offsets, E, R,
                                      nvfp4::grouped_chunk_rows(R, E), tiles, global_scale,
                                      partials, n_partials, d->status, d->sms, s) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_amax_partials(const void* x, int64_t rows, int64_t K, int64_t ld, int64_t R,
                                 int32_t E, uint8_t* tiles, void* stream) {
  if (rows < 0 || K <= 0 || ld < K || E <= 0 || R < 0) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && (!x || !tiles)) return NVFP4_ERR_INVALID_ARG;
  if (K % 64 != 0 || ld % 8 != 0 || E > 1024) return NVFP4_ERR_UNSUPPORTED;
  if ((x && !aligned16(x)) || (tiles && !aligned16(tiles))) return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  if (rows == 0) return NVFP4_OK;
  const int n_partials = nvfp4::amax_partials_count(rows, K, d->sms);
  if (static_cast<size_t>(n_partials) * sizeof(uint32_t) > kAmaxScratchBytes)
    return NVFP4_ERR_UNSUPPORTED;
  uint32_t* partials = reinterpret_cast<uint32_t*>(tiles + grouped_tiles_body_bytes(R, E, K));
  if (nvfp4::launch_amax_partials(static_cast<const uint16_t*>(x), rows, K, ld, partials, d->sms,
                                  static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

static nvfp4_status grouped_gemm_impl(const uint8_t* A_tiles, const float* gA,
                                      const uint8_t* W_tiles, const float* gW,
                                      const int32_t* expert_offsets, int32_t E,
                                      int64_t T, int32_t topk, int64_t N, int64_t K,
                                      const int32_t* route_token, const int32_t* route_slot,
                                      const float* topk_weights,
                                      void* out, float* workspace, size_t workspace_bytes,
                                      bool sparse_w, const CUtensorMap* w_map, void* stream) {
  if (!A_tiles || !gA || !W_tiles || !gW || !expert_offsets || !out) return NVFP4_ERR_INVALID_ARG;
  if (E <= 0 || T < 0 || topk <= 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
  const bool combine = topk_weights != nullptr;
  if (combine && (!route_token || !route_slot || !workspace)) return NVFP4_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 64 != 0 || E > nvfp4::kGroupedMaxExperts) return NVFP4_ERR_UNSUPPORTED;
  const int64_t R = T * topk;
  if (R > (1LL << 30) || static_cast<int64_t>(E) * N > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED;
  if (combine && workspace_bytes < nvfp4_combine_workspace_bytes(T, N)) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned16(A_tiles) || !aligned16(W_tiles) || !aligned16(out) ||
      (combine && !aligned16(workspace)))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (R == 0) {
    if (combine && T > 0 && cudaMemsetAsync(out, 0, T * N * 2, s) != cudaSuccess) return cuda_fail();
    return NVFP4_OK;
  }
  // operand tiles need no tensor map; row-major weights come through w_map
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  nvfp4::GemmArgs a{};
  a.sfx = W_tiles;
  a.x_map = w_map ? 1 : 0;
  a.sfy = A_tiles;
  a.gx = gW;
  a.gy = gA;
  a.K = K;
  a.rows_x = static_cast<int32_t>(E * N);
  a.rows_y = static_cast<int32_t>(R);
  a.expert_offsets = expert_offsets;
  a.E = E;
  a.n_out = static_cast<int32_t>(N);
  a.out = out;
  a.ldc = N;
  a.vec_store = 1;
  a.ybox_rows = 16;
  a.route_token = route_token;
  a.route_slot = route_slot;
  a.topk_w = topk_weights;
  a.topk = topk;
  a.n_tokens = static_cast<int32_t>(T);
  a.ws = workspace;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns.load();
  a.debug_flags = g_debug_flags.load();
  a.sparse_w = sparse_w ? 1 : 0;
  if (combine && cudaMemsetAsync(workspace, 0, nvfp4_combine_workspace_bytes(T, N), s) != cudaSuccess)
    return cuda_fail();
  const int mode = combine ? nvfp4::kGroupedCombine : nvfp4::kGrouped;
  const int pair_width = nvfp4::grouped_pair_width(a, mode);
  if (pair_width > 0) {
    // 128- and 256-route token tiles of dense operand tiles: the CTA-pair kernel
    nvfp4::GroupedPairMaps pm;
    const uint64_t nkb = static_cast<uint64_t>((K + 255) / 256);
    const uint64_t x_rows = static_cast<uint64_t>(E) * static_cast<uint64_t>(N / 128) * nkb * 144;
    const uint64_t y_rows = static_cast<uint64_t>(grouped_token_tiles(R, E)) * nkb * 144;
    if (make_tile_rows_map(&pm.x_codes, W_tiles, x_rows, 128) != NVFP4_OK ||
        make_tile_rows_map(&pm.x_scales, W_tiles, x_rows, 16) != NVFP4_OK ||
        make_tile_rows_map(&pm.y_codes, A_tiles, y_rows, static_cast<uint32_t>(pair_width / 2)) !=
            NVFP4_OK ||
        make_tile_rows_map(&pm.y_scales, A_tiles, y_rows, 16) != NVFP4_OK)
      return NVFP4_ERR_UNSUPPORTED;
    if (nvfp4::launch_grouped_pair(pm, a, mode, s) != cudaSuccess) return cuda_fail();
  } else if (nvfp4::launch_gemm(w_map ? *w_map : unused, unused, a, mode, d->sms, s) !=
             cudaSuccess) {
    return cuda_fail();
  }
  if (combine && nvfp4::launch_combine_finalize(workspace, T, N, out, d->sms, s) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_grouped_gemm_tiles(const uint8_t* A_tiles, const float* gA,
                                      const uint8_t* W_tiles, const float* gW,
                                      const int32_t* expert_offsets, int32_t E,
                                      int64_t T, int32_t topk, int64_t N, int64_t K,
                                      const int32_t* route_token, const int32_t* route_slot,
                                      const float* topk_weights,
                                      void* out, float* workspace, size_t workspace_bytes,
                                      void* stream) {
  return grouped_gemm_impl(A_tiles, gA, W_tiles, gW, expert_offsets, E, T, topk, N, K,
                           route_token, route_slot, topk_weights, out, workspace,
                           workspace_bytes, false, nullptr, stream);
}

nvfp4_status nvfp4_grouped_gemm_sparse(const uint8_t* A_tiles, const float* gA,
                                       const uint8_t* W_sparse_tiles, const float* gW,
                                       const int32_t* expert_offsets, int32_t E,
                                       int64_t T, int32_t topk, int64_t N, int64_t K,
                                       const int32_t* route_token, const int32_t* route_slot,
                                       const float* topk_weights,
                                       void* out, float* workspace, size_t workspace_bytes,
                                       void* stream) {
  return grouped_gemm_impl(A_tiles, gA, W_sparse_tiles, gW, expert_offsets, E, T, topk, N, K,
                           route_token, route_slot, topk_weights, out, workspace,
                           workspace_bytes, true, nullptr, stream);
}

nvfp4_status nvfp4_grouped_gemm(const uint8_t* A, const uint8_t* sfA, const float* gA,
                                const uint8_t* W, const uint8_t* sfW_tc, const float* gW,
                                const int32_t* expert_offsets, int32_t E,
                                const int32_t* route_token, const float* topk_weights,
                                const int32_t* route_slot, int64_t T, int32_t topk, int64_t N,
                                int64_t K, void* out, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (!A || !sfA || !gA || !W || !sfW_tc || !gW || !expert_offsets || !out || !workspace)
    return NVFP4_ERR_INVALID_ARG;
  if (E <= 0 || T < 0 || topk <= 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
  const bool combine = topk_weights != nullptr;
  if (combine && (!route_token || !route_slot)) return NVFP4_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 64 != 0 || E > nvfp4::kGroupedMaxExperts) return NVFP4_ERR_UNSUPPORTED;
  const int64_t R = T * topk;
  if (R > (1LL << 30) || static_cast<int64_t>(E) * N > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED;
  if (workspace_bytes < nvfp4_grouped_gemm_workspace_bytes(T, topk, E, N, K, combine ? 1 : 0))
    return NVFP4_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(W) || !aligned16(sfW_tc) || !aligned16(out) ||
      !aligned16(workspace))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (R == 0) {
    if (combine && T > 0 && cudaMemsetAsync(out, 0, T * N * 2, s) != cudaSuccess) return cuda_fail();
    return NVFP4_OK;
  }
  // the activation rows into route order, as grouped operand tiles at the
  // start of the workspace; the FP32 combine sums follow them
  uint8_t* a_tiles = static_cast<uint8_t*>(workspace);
  const size_t tiles_bytes = grouped_tiles_body_bytes(R, E, K);
  // gather by route_token only when the output stays in route order; the
  // combine's input (the experts' intermediate) is already route-ordered
  const bool gather = route_token != nullptr && !combine;
  if (nvfp4::launch_gather_dispatch(A, sfA, gather ? T : R, K, gather ? route_token : nullptr,
                                    expert_offsets, E, R, nvfp4::grouped_chunk_rows(R, E), a_tiles,
                                    d->status, d->sms, s) != cudaSuccess)
    return cuda_fail();
  CUtensorMap w_map;
  if (make_operand_map(&w_map, W, static_cast<uint64_t>(E) * N, K / 2, 128) != NVFP4_OK)
    return NVFP4_ERR_UNSUPPORTED;
  float* ws = combine ? reinterpret_cast<float*>(a_tiles + tiles_bytes) : nullptr;
  return grouped_gemm_impl(a_tiles, gA, sfW_tc, gW, expert_offsets, E, T, topk, N, K,
                           route_token, route_slot, topk_weights, out, ws,
                           combine ? nvfp4_combine_workspace_bytes(T, N) : 0, false, &w_map,
                           stream);
}

size_t nvfp4_sparse_tiles_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((K + 255) / 256) *
         static_cast<size_t>(nvfp4::kSparseTileBytes);
}

nvfp4_status nvfp4_prune_2of4(const void* w, int64_t rows, int64_t cols, int64_t ld, void* out,
                              int64_t ld_out, void* stream) {
  if (rows < 0 || cols < 0 || ld < cols || ld_out < cols) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && (!w || !out)) return NVFP4_ERR_INVALID_ARG;
  if (cols % 8 != 0 || ld % 8 != 0 || ld_out % 8 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((w && !aligned16(w)) || (out && !aligned16(out))) return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  if (nvfp4::launch_prune_2of4(static_cast<const uint16_t*>(w), rows, cols, ld,
                               static_cast<uint16_t*>(out), ld_out, d->sms,
                               static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_prepack_sparse_weight_tiles(const uint8_t* packed,
                                               const uint8_t* scales_rowmajor, int64_t rows,
                                               int64_t K, uint8_t* tiles, void* stream) {
  if (rows < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && K > 0 && (!packed || !scales_rowmajor || !tiles)) return NVFP4_ERR_INVALID_ARG;
  if (K % 64 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((packed && !aligned16(packed)) || (tiles && !aligned16(tiles)) ||
      (scales_rowmajor && (reinterpret_cast<uintptr_t>(scales_rowmajor) & 3u)))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  if (nvfp4::launch_prepack_sparse_tiles(packed, scales_rowmajor, rows, K, tiles, d->status,
                                         d->sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

size_t nvfp4_decode_attention_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int64_t L_max,
                                              int32_t D) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L_max < 0 || D <= 0) return 0;
  const int ch = nvfp4::attention_chunk(L_max, B, Hkv);
  const int64_t splits = (L_max + ch - 1) / ch;
  // heads of 256 and 512 also keep every cached token's base-2 score per query
  // head (the tensor-core path writes them in one pass and reads them in the
  // next)
  const size_t scores = D >= 256 ? static_cast<size_t>(B) * static_cast<size_t>(Hq) *
                                       static_cast<size_t>(L_max) * sizeof(float)
                                 : 0;
  return static_cast<size_t>(B) * static_cast<size_t>(Hq) * static_cast<size_t>(splits) *
             static_cast<size_t>(D + 2) * sizeof(float) +
         scores;
}

nvfp4_status nvfp4_decode_attention(const void* q, const uint8_t* k_packed,
                                    const uint8_t* k_scales, const float* gk,
                                    const uint8_t* v_packed, const uint8_t* v_scales,
                                    const float* gv, const int32_t* seq_lens, int32_t B,
                                    int32_t Hq, int32_t Hkv, int64_t L_max, int32_t D, float scale,
                                    void* out, float* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || L_max < 0 || D <= 0) return NVFP4_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return NVFP4_ERR_INVALID_ARG;
  if (B == 0) return NVFP4_OK;
  if (!q || !gk || !gv || !seq_lens || !out || !workspace) return NVFP4_ERR_INVALID_ARG;
  if (L_max > 0 && (!k_packed || !k_scales || !v_packed || !v_scales)) return NVFP4_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (D != 64 && D != 128 && D != 256 && D != 512) return NVFP4_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return NVFP4_ERR_UNSUPPORTED;
  if (D == 512 && G == 8) return NVFP4_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535 || static_cast<int64_t>(B) * Hq > (1LL << 31) - 1)
    return NVFP4_ERR_UNSUPPORTED;
  if (L_max > (1LL << 31) - 1) return NVFP4_ERR_UNSUPPORTED;
  if (workspace_bytes < nvfp4_decode_attention_workspace_bytes(B, Hq, Hkv, L_max, D))
    return NVFP4_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) ||
      (k_packed && !aligned16(k_packed)) || (v_packed && !aligned16(v_packed)) ||
      (k_scales && (reinterpret_cast<uintptr_t>(k_scales) & 3u)) ||
      (v_scales && (reinterpret_cast<uintptr_t>(v_scales) & 3u)) ||
      (reinterpret_cast<uintptr_t>(gk) & 3u) || (reinterpret_cast<uintptr_t>(gv) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  nvfp4::AttnArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k_packed = k_packed;
  a.k_scales = k_scales;
  a.v_packed = v_packed;
  a.v_scales = v_scales;
  a.gk = gk;
  a.gv = gv;
  a.debug_flags = g_debug_flags.load();
  a.seq_lens = seq_lens;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.L_max = L_max;
  a.chunk = nvfp4::attention_chunk(L_max, B, Hkv);
  a.splits = static_cast<int32_t>((L_max + a.chunk - 1) / a.chunk);
  a.scale = scale;
  a.out = static_cast<uint16_t*>(out);
  a.ws_o = workspace;
  a.ws_ml = workspace + static_cast<int64_t>(B) * Hq * a.splits * D;
  a.ws_s = a.ws_ml + static_cast<int64_t>(B) * Hq * a.splits * 2;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns.load();
  nvfp4::AttnMaps maps;
  const bool tc = nvfp4::decode_attention_tc_applies(a, D);
  if (tc) {
    const uint64_t rows = static_cast<uint64_t>(B) * Hkv * L_max;
    if (make_kv_code_map(&maps.k_codes, k_packed, rows, D) != NVFP4_OK ||
        make_kv_code_map(&maps.v_codes, v_packed, rows, D) != NVFP4_OK ||
        make_kv_scale_map(&maps.k_scales, k_scales, rows, D) != NVFP4_OK ||
        make_kv_scale_map(&maps.v_scales, v_scales, rows, D) != NVFP4_OK)
      return NVFP4_ERR_UNSUPPORTED;
  }
  if (nvfp4::launch_decode_attention(a, D, tc ? &maps : nullptr,
                                     static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_moe_gate_up_silu(const uint8_t* A_tiles, const float* gA,
                                    const uint8_t* W_tiles, const float* gW,
                                    const int32_t* expert_offsets, int32_t E, int64_t T,
                                    int32_t topk, int64_t N, int64_t K, const float* g_h,
                                    uint8_t* h_tiles, void* stream) {
  if (!A_tiles || !gA || !W_tiles || !gW || !expert_offsets || !g_h || !h_tiles)
    return NVFP4_ERR_INVALID_ARG;
  if (E <= 0 || T < 0 || topk <= 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
  if (N % 256 != 0 || K % 64 != 0 || E > nvfp4::kGroupedMaxExperts) return NVFP4_ERR_UNSUPPORTED;
  const int64_t R = T * topk;
  if (R > (1LL << 30) || static_cast<int64_t>(E) * N > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned16(A_tiles) || !aligned16(W_tiles) || !aligned16(h_tiles) ||
      (reinterpret_cast<uintptr_t>(g_h) & 3u))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  if (R == 0) return NVFP4_OK;
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  nvfp4::GemmArgs a{};
  a.sfx = W_tiles;
  a.sfy = A_tiles;
  a.gx = gW;
  a.gy = gA;
  a.K = K;
  a.rows_x = static_cast<int32_t>(E * N);
  a.rows_y = static_cast<int32_t>(R);
  a.expert_offsets = expert_offsets;
  a.E = E;
  a.n_out = static_cast<int32_t>(N);
  a.ldc = N;
  a.vec_store = 1;
  a.ybox_rows = 16;
  a.topk = topk;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns.load();
  a.debug_flags = g_debug_flags.load();
  a.h_tiles = h_tiles;
  a.g_h = g_h;
  a.h_nkb = static_cast<int32_t>((N / 2 + 255) / 256);
  if (nvfp4::launch_gemm(unused, unused, a, nvfp4::kGroupedSiluMul, d->sms,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

nvfp4_status nvfp4_moe_gate_up_silu_bf16(const uint8_t* A_tiles, const float* gA,
                                         const uint8_t* W_tiles, const float* gW,
                                         const int32_t* expert_offsets, int32_t E, int64_t T,
                                         int32_t topk, int64_t N, int64_t K, void* h_out,
                                         void* stream) {
  if (!A_tiles || !gA || !W_tiles || !gW || !expert_offsets || !h_out)
    return NVFP4_ERR_INVALID_ARG;
  if (E <= 0 || T < 0 || topk <= 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
  if (N % 256 != 0 || K % 64 != 0 || E > nvfp4::kGroupedMaxExperts) return NVFP4_ERR_UNSUPPORTED;
  const int64_t R = T * topk;
  if (R > (1LL << 30) || static_cast<int64_t>(E) * N > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned16(A_tiles) || !aligned16(W_tiles) || !aligned16(h_out))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  if (R == 0) return NVFP4_OK;
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  nvfp4::GemmArgs a{};
  a.sfx = W_tiles;
  a.sfy = A_tiles;
  a.gx = gW;
  a.gy = gA;
  a.K = K;
  a.rows_x = static_cast<int32_t>(E * N);
  a.rows_y = static_cast<int32_t>(R);
  a.expert_offsets = expert_offsets;
  a.E = E;
  a.n_out = static_cast<int32_t>(N);
  a.out = h_out;
  a.ldc = N / 2;
  a.vec_store = 1;
  a.ybox_rows = 16;
  a.topk = topk;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns.load();
  a.debug_flags = g_debug_flags.load();
  if (nvfp4::launch_gemm(unused, unused, a, nvfp4::kGroupedSiluBf16, d->sms,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return NVFP4_OK;
}

size_t nvfp4_moe_mlp_workspace_bytes(int64_t T, int32_t topk, int32_t E, int64_t N2) {
  if (T < 0 || topk <= 0 || E <= 0 || N2 < 0) return 0;
  const size_t sums = nvfp4_combine_workspace_bytes(T, N2);
  return sums + static_cast<size_t>(grouped_token_tiles(T * topk, E)) * sizeof(uint32_t);
}

nvfp4_status nvfp4_moe_mlp(const uint8_t* A_tiles, const float* gA, const uint8_t* W1_tiles,
                           const float* gW1, const uint8_t* W2_tiles, const float* gW2,
                           const int32_t* expert_offsets, int32_t E, int64_t T, int32_t topk,
                           int64_t N1, int64_t K1, int64_t N2, const float* g_h, uint8_t* h_tiles,
                           const int32_t* route_token, const int32_t* route_slot,
                           const float* topk_weights, void* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (!A_tiles || !gA || !W1_tiles || !gW1 || !W2_tiles || !gW2 || !expert_offsets || !g_h ||
      !h_tiles || !route_token || !route_slot || !topk_weights || !out || !workspace)
    return NVFP4_ERR_INVALID_ARG;
  if (E <= 0 || T < 0 || topk <= 0 || N1 <= 0 || K1 <= 0 || N2 <= 0) return NVFP4_ERR_INVALID_ARG;
  if (N1 % 256 != 0 || N2 % 256 != 0 || K1 % 64 != 0 || E > nvfp4::kGroupedMaxExperts)
    return NVFP4_ERR_UNSUPPORTED;
  const int64_t R = T * topk;
  if (R > (1LL << 30) || static_cast<int64_t>(E) * N1 > (1LL << 30) ||
      static_cast<int64_t>(E) * N2 > (1LL << 30))
    return NVFP4_ERR_UNSUPPORTED;
  if (workspace_bytes < nvfp4_moe_mlp_workspace_bytes(T, topk, E, N2)) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned16(A_tiles) || !aligned16(W1_tiles) || !aligned16(W2_tiles) || !aligned16(h_tiles) ||
      !aligned16(out) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(g_h) & 3u))
    return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (R == 0) {
    if (T > 0 && cudaMemsetAsync(out, 0, T * N2 * 2, s) != cudaSuccess) return cuda_fail();
    return NVFP4_OK;
  }
  // FP32 sums of the combine, then one ready count per token tile; both start at zero
  float* ws = static_cast<float*>(workspace);
  uint32_t* ready = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) +
                                                nvfp4_combine_workspace_bytes(T, N2));
  if (cudaMemsetAsync(workspace, 0, nvfp4_moe_mlp_workspace_bytes(T, topk, E, N2), s) !=
      cudaSuccess)
    return cuda_fail();
  nvfp4::GemmArgs a{};
  a.sfx = W1_tiles;
  a.sfy = A_tiles;
  a.gx = gW1;
  a.gy = gA;
  a.K = K1;
  a.rows_x = static_cast<int32_t>(E * N1);
  a.rows_y = static_cast<int32_t>(R);
  a.expert_offsets = expert_offsets;
  a.E = E;
  a.n_out = static_cast<int32_t>(N1);
  a.ldc = N2;
  a.vec_store = 1;
  a.ybox_rows = 16;
  a.route_token = route_token;
  a.route_slot = route_slot;
  a.topk_w = topk_weights;
  a.topk = topk;
  a.n_tokens = static_cast<int32_t>(T);
  a.ws = ws;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns.load();
  a.debug_flags = g_debug_flags.load();
  a.h_tiles = h_tiles;
  a.g_h = g_h;
  a.h_nkb = static_cast<int32_t>((N1 / 2 + 255) / 256);
  a.sfx2 = W2_tiles;
  a.gx2 = gW2;
  a.K2 = N1 / 2;
  a.n_out2 = static_cast<int32_t>(N2);
  a.ready = ready;
  if (nvfp4::launch_mlp_fused(a, d->sms, s) != cudaSuccess) return cuda_fail();
  if (nvfp4::launch_combine_finalize(ws, T, N2, out, d->sms, s) != cudaSuccess) return cuda_fail();
  return NVFP4_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of the weighted-combine grouped GEMM.
// ---------------------------------------------------------------------------
namespace {

// FP32 combine workspace shared by every call of
// nvfp4_grouped_gemm_combine_noalloc on a device.  Every GPU that loads this
// library holds it until the process exits.
constexpr size_t kNoallocWorkspaceFloats = 4u * 1024u * 1024u;   // 16 MiB
static __device__ __align__(256) float g_noalloc_workspace[kNoallocWorkspaceFloats];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the workspace for the current device.  In host code the
// array's name only stands in for the symbol, so the address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
nvfp4_status noalloc_workspace(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
  if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return cuda_fail();
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return NVFP4_OK;
}

}  // namespace

extern "C" {

size_t nvfp4_noalloc_workspace_floats(void) { return kNoallocWorkspaceFloats; }

nvfp4_status nvfp4_grouped_gemm_combine_noalloc(const uint8_t* A_tiles, const float* gA,
                                                const uint8_t* W_tiles, const float* gW,
                                                const int32_t* expert_offsets, int32_t E,
                                                int64_t T, int32_t topk, int64_t N, int64_t K,
                                                const int32_t* route_token,
                                                const int32_t* route_slot,
                                                const float* topk_weights, void* out,
                                                void* stream) {
  if (!A_tiles || !gA || !W_tiles || !gW || !expert_offsets || !out || !route_token ||
      !route_slot || !topk_weights)
    return NVFP4_ERR_INVALID_ARG;
  if (E <= 0 || T < 0 || topk <= 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 64 != 0 || E > nvfp4::kGroupedMaxExperts) return NVFP4_ERR_UNSUPPORTED;
  // the combine workspace holds T x N floats: refuse what does not fit
  if (T > 0 && static_cast<uint64_t>(T) * static_cast<uint64_t>(N) > kNoallocWorkspaceFloats)
    return NVFP4_ERR_UNSUPPORTED;
  const int64_t R = T * topk;
  if (R > (1LL << 30) || static_cast<int64_t>(E) * N > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED;
  if (!aligned16(A_tiles) || !aligned16(W_tiles) || !aligned16(out)) return NVFP4_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  nvfp4_status st = device_state(&d);
  if (st != NVFP4_OK) return st;
  float* ws = nullptr;
  st = noalloc_workspace(&ws);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (R == 0) {
    if (T > 0 && cudaMemsetAsync(out, 0, T * N * 2, s) != cudaSuccess) return cuda_fail();
    return NVFP4_OK;
  }
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  nvfp4::GemmArgs a{};
  a.sfx = W_tiles;
  a.sfy = A_tiles;
  a.gx = gW;
  a.gy = gA;
  a.K = K;
  a.rows_x = static_cast<int32_t>(E * N);
  a.rows_y = static_cast<int32_t>(R);
  a.expert_offsets = expert_offsets;
  a.E = E;
  a.n_out = static_cast<int32_t>(N);
  a.out = out;
  a.ldc = N;
  a.vec_store = 1;
  a.ybox_rows = 16;
  a.route_token = route_token;
  a.route_slot = route_slot;
  a.topk_w = topk_weights;
  a.topk = topk;
  a.n_tokens = static_cast<int32_t>(T);
  a.ws = ws;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns.load();
  a.debug_flags = g_debug_flags.load();
  // the workspace keeps the previous call's sums: clear the part this call uses
  if (cudaMemsetAsync(ws, 0, static_cast<size_t>(T) * N * sizeof(float), s) != cudaSuccess)
    return cuda_fail();
  if (nvfp4::launch_gemm(unused, unused, a, nvfp4::kGroupedCombine, d->sms, s) != cudaSuccess)
    return cuda_fail();
  if (nvfp4::launch_combine_finalize(ws, T, N, out, d->sms, s) != cudaSuccess) return cuda_fail();
  return NVFP4_OK;
}

}  // extern "C"
