"""Thin Python binding of the C ABI in include/nvfp4.h.

Argument marshalling only: every step runs in the CUDA library.  Functions
carry the C names; tensors are torch CUDA tensors (torch supplies device
memory and the current stream).  A missing library or a non-OK status
raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_UNSUPPORTED = 2
NVFP4_ERR_CUDA = 3
NVFP4_ERR_TIMEOUT = 4
NVFP4_ERR_DEVICE_CHECK = 5

NVFP4_SF_ROWMAJOR = 0
NVFP4_SF_ATOMS = 1
NVFP4_GLOBAL_GIVEN = 2
NVFP4_AMAX_DONE = 4

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_U32 = ctypes.c_uint32
_SZ = ctypes.c_size_t

_SIGS = {
    "nvfp4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "nvfp4_version": (ctypes.c_int, []),
    "nvfp4_device_status": (ctypes.c_int, [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
    "nvfp4_set_timeout_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "nvfp4_debug_set_flags": (ctypes.c_int, [ctypes.c_uint32]),
    "nvfp4_atom_scales_bytes": (_SZ, [_I64, _I64]),
    "nvfp4_last_device_status": (ctypes.c_int, [_P]),
    "nvfp4_prepacked_scales_bytes": (_SZ, [_I64, _I64]),
    "nvfp4_grouped_gemm_workspace_bytes": (_SZ, [_I64, _I32, _I32, _I64, _I64, _I32]),
    "nvfp4_quantize": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _U32, _P]),
    "nvfp4_prepack_weights": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "nvfp4_gemm": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "nvfp4_moe_route": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P]),
    "nvfp4_operand_tiles_bytes": (_SZ, [_I64, _I64]),
    "nvfp4_prepack_weight_tiles": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
    "nvfp4_grouped_chunk_rows": (ctypes.c_int, [_I64, _I32]),
    "nvfp4_grouped_tiles_bytes": (_SZ, [_I64, _I32, _I64]),
    "nvfp4_quantize_dispatch": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I32, _P, _I32, _I64,
                                               _P, _P, _U32, _P]),
    "nvfp4_amax_partials": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _I32, _P, _P]),
    "nvfp4_combine_workspace_bytes": (_SZ, [_I64, _I64]),
    "nvfp4_grouped_gemm": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _I64,
                                          _I32, _I64, _I64, _P, _P, _SZ, _P]),
    "nvfp4_grouped_gemm_tiles": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _I32, _I64,
                                                _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_moe_gate_up_silu": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _I32, _I64, _I64,
                                              _P, _P, _P]),
    "nvfp4_moe_gate_up_silu_bf16": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _I32, _I64,
                                                   _I64, _P, _P]),
    "nvfp4_moe_mlp_workspace_bytes": (_SZ, [_I64, _I32, _I32, _I64]),
    "nvfp4_moe_mlp": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I32, _I64, _I64,
                                     _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_noalloc_workspace_floats": (_SZ, []),
    "nvfp4_decode_attention_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I64, _I32]),
    "nvfp4_decode_attention": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32,
                                              _I64, _I32, ctypes.c_float, _P, _P, _SZ, _P]),
    "nvfp4_prune_2of4": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _P]),
    "nvfp4_sparse_tiles_bytes": (_SZ, [_I64, _I64]),
    "nvfp4_prepack_sparse_weight_tiles": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
    "nvfp4_grouped_gemm_sparse": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _I32, _I64,
                                                 _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_grouped_gemm_combine_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _I32,
                                                          _I64, _I64, _P, _P, _P, _P, _P]),
}


class NVFP4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {nvfp4_status_string(status)} ({status})")


def lib_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Loads the in-tree library (building it first if sources are newer)."""
    global _lib
    if _lib is None:
        path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"NVFP4 CUDA library missing: {path}")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _row_stride(x):
    """Row stride in elements; a single row may carry any stride in torch
    (0 for a broadcast view), and its stride is never used, so pass the width."""
    return x.stride(0) if x.shape[0] > 1 else x.shape[1]


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _check(fn, st):
    if st != NVFP4_OK:
        raise NVFP4Error(fn, st)


# ------------------------------------------------------------ C entry points

def nvfp4_status_string(status: int) -> str:
    return load().nvfp4_status_string(int(status)).decode()


def nvfp4_version() -> int:
    return load().nvfp4_version()


def nvfp4_device_status(reset: bool = True, stream=None) -> int:
    out = ctypes.c_int(0)
    _check("nvfp4_device_status",
           load().nvfp4_device_status(_stream(stream), int(reset), ctypes.byref(out)))
    return out.value


def nvfp4_set_timeout_ns(ns: int) -> None:
    _check("nvfp4_set_timeout_ns", load().nvfp4_set_timeout_ns(int(ns)))


def nvfp4_debug_set_flags(flags: int) -> None:
    _check("nvfp4_debug_set_flags", load().nvfp4_debug_set_flags(int(flags)))


def nvfp4_last_device_status(stream=None) -> int:
    """The device status word (not cleared); see nvfp4_device_status."""
    return load().nvfp4_last_device_status(_stream(stream))


def nvfp4_prepacked_scales_bytes(rows: int, kblk: int) -> int:
    return load().nvfp4_prepacked_scales_bytes(rows, kblk)


def nvfp4_grouped_gemm_workspace_bytes(T: int, topk: int, E: int, N: int, K: int,
                                       combine: bool) -> int:
    return load().nvfp4_grouped_gemm_workspace_bytes(T, topk, E, N, K, int(bool(combine)))


def nvfp4_atom_scales_bytes(rows: int, cols: int) -> int:
    return load().nvfp4_atom_scales_bytes(rows, cols)


def nvfp4_operand_tiles_bytes(rows: int, K: int) -> int:
    return load().nvfp4_operand_tiles_bytes(rows, K)


def nvfp4_grouped_chunk_rows(R: int, E: int) -> int:
    return load().nvfp4_grouped_chunk_rows(R, E)


def nvfp4_grouped_tiles_bytes(R: int, E: int, K: int) -> int:
    return load().nvfp4_grouped_tiles_bytes(R, E, K)


def nvfp4_combine_workspace_bytes(T: int, N: int) -> int:
    return load().nvfp4_combine_workspace_bytes(T, N)


def nvfp4_quantize(x, packed, scales, global_scale, flags: int = 0, stream=None) -> None:
    rows, cols = x.shape
    _check("nvfp4_quantize", load().nvfp4_quantize(
        _ptr(x), rows, cols, _row_stride(x), _ptr(packed), _ptr(scales), _ptr(global_scale),
        flags, _stream(stream)))


def nvfp4_prepack_weights(scales_rowmajor, scales_atoms, stream=None) -> None:
    rows, kblk = scales_rowmajor.shape
    _check("nvfp4_prepack_weights", load().nvfp4_prepack_weights(
        _ptr(scales_rowmajor), rows, kblk, _ptr(scales_atoms), _stream(stream)))


def nvfp4_gemm(A, sfA, gA, B, sfB, gB, C, K: int, stream=None) -> None:
    M, N = C.shape
    _check("nvfp4_gemm", load().nvfp4_gemm(
        _ptr(A), _ptr(sfA), _ptr(gA), _ptr(B), _ptr(sfB), _ptr(gB), _ptr(C), M, N, K,
        C.stride(0), _stream(stream)))


def nvfp4_moe_route(topk_ids, E: int, expert_offsets, route_token, route_slot, route_pos=None,
                    stream=None) -> None:
    T, topk = topk_ids.shape
    _check("nvfp4_moe_route", load().nvfp4_moe_route(
        _ptr(topk_ids), T, topk, E, _ptr(expert_offsets), _ptr(route_token), _ptr(route_slot),
        _ptr(route_pos), _stream(stream)))


def nvfp4_prepack_weight_tiles(packed, scales_rowmajor, tiles, stream=None) -> None:
    rows, half = packed.shape
    _check("nvfp4_prepack_weight_tiles", load().nvfp4_prepack_weight_tiles(
        _ptr(packed), _ptr(scales_rowmajor), rows, 2 * half, _ptr(tiles), _stream(stream)))


def nvfp4_quantize_dispatch(x, route_pos, fanout: int, expert_offsets, E: int, R: int, tiles,
                            global_scale, flags: int = 0, stream=None) -> None:
    rows, K = x.shape
    _check("nvfp4_quantize_dispatch", load().nvfp4_quantize_dispatch(
        _ptr(x), rows, K, _row_stride(x), _ptr(route_pos), fanout, _ptr(expert_offsets), E, R,
        _ptr(tiles), _ptr(global_scale), flags, _stream(stream)))


def nvfp4_moe_gate_up_silu(A_tiles, gA, W_tiles, gW, expert_offsets, E: int, T: int, topk: int,
                           N: int, K: int, g_h, h_tiles, stream=None) -> None:
    _check("nvfp4_moe_gate_up_silu", load().nvfp4_moe_gate_up_silu(
        _ptr(A_tiles), _ptr(gA), _ptr(W_tiles), _ptr(gW), _ptr(expert_offsets), E, T, topk, N, K,
        _ptr(g_h), _ptr(h_tiles), _stream(stream)))


def nvfp4_moe_gate_up_silu_bf16(A_tiles, gA, W_tiles, gW, expert_offsets, E: int, T: int,
                                topk: int, N: int, K: int, h_out, stream=None) -> None:
    _check("nvfp4_moe_gate_up_silu_bf16", load().nvfp4_moe_gate_up_silu_bf16(
        _ptr(A_tiles), _ptr(gA), _ptr(W_tiles), _ptr(gW), _ptr(expert_offsets), E, T, topk, N, K,
        _ptr(h_out), _stream(stream)))


def nvfp4_moe_mlp_workspace_bytes(T: int, topk: int, E: int, N2: int) -> int:
    return load().nvfp4_moe_mlp_workspace_bytes(T, topk, E, N2)


def nvfp4_moe_mlp(A_tiles, gA, W1_tiles, gW1, W2_tiles, gW2, expert_offsets, E: int, T: int,
                  topk: int, N1: int, K1: int, N2: int, g_h, h_tiles, route_token, route_slot,
                  topk_weights, out, workspace, stream=None) -> None:
    """The expert MLP (gate_up, SiLU * up, NVFP4 h, down, combine) in one
    persistent launch; see include/nvfp4.h."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("nvfp4_moe_mlp", load().nvfp4_moe_mlp(
        _ptr(A_tiles), _ptr(gA), _ptr(W1_tiles), _ptr(gW1), _ptr(W2_tiles), _ptr(gW2),
        _ptr(expert_offsets), E, T, topk, N1, K1, N2, _ptr(g_h), _ptr(h_tiles), _ptr(route_token),
        _ptr(route_slot), _ptr(topk_weights), _ptr(out), _ptr(workspace), ws_bytes,
        _stream(stream)))


def nvfp4_amax_partials(x, R: int, E: int, tiles, stream=None) -> None:
    rows, K = x.shape
    _check("nvfp4_amax_partials", load().nvfp4_amax_partials(
        _ptr(x), rows, K, _row_stride(x), R, E, _ptr(tiles), _stream(stream)))


def nvfp4_grouped_gemm(A, sfA, gA, W, sfW_tc, gW, expert_offsets, E: int, route_token,
                       topk_weights, route_slot, T: int, topk: int, N: int, K: int, out,
                       workspace, stream=None) -> None:
    """Grouped GEMM on plain NVFP4 operands (packed rows + row-major scales for
    A, packed rows + atom-layout scales for W); see include/nvfp4.h."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("nvfp4_grouped_gemm", load().nvfp4_grouped_gemm(
        _ptr(A), _ptr(sfA), _ptr(gA), _ptr(W), _ptr(sfW_tc), _ptr(gW), _ptr(expert_offsets), E,
        _ptr(route_token), _ptr(topk_weights), _ptr(route_slot), T, topk, N, K, _ptr(out),
        _ptr(workspace), ws_bytes, _stream(stream)))


def nvfp4_grouped_gemm_tiles(A_tiles, gA, W_tiles, gW, expert_offsets, E: int, T: int,
                             topk: int, N: int, K: int, route_token, route_slot, topk_weights,
                             out, workspace, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("nvfp4_grouped_gemm_tiles", load().nvfp4_grouped_gemm_tiles(
        _ptr(A_tiles), _ptr(gA), _ptr(W_tiles), _ptr(gW), _ptr(expert_offsets), E, T, topk, N,
        K, _ptr(route_token), _ptr(route_slot), _ptr(topk_weights), _ptr(out),
        _ptr(workspace), ws_bytes, _stream(stream)))


def nvfp4_prune_2of4(w, out, stream=None) -> None:
    """2:4 magnitude pruning over element pairs of BF16 [rows, cols]; out may be w."""
    rows, cols = w.shape
    _check("nvfp4_prune_2of4", load().nvfp4_prune_2of4(
        _ptr(w), rows, cols, _row_stride(w), _ptr(out), _row_stride(out), _stream(stream)))


def nvfp4_sparse_tiles_bytes(rows: int, K: int) -> int:
    return load().nvfp4_sparse_tiles_bytes(rows, K)


def nvfp4_prepack_sparse_weight_tiles(packed, scales_rowmajor, tiles, stream=None) -> None:
    rows, half = packed.shape
    _check("nvfp4_prepack_sparse_weight_tiles", load().nvfp4_prepack_sparse_weight_tiles(
        _ptr(packed), _ptr(scales_rowmajor), rows, 2 * half, _ptr(tiles), _stream(stream)))


def nvfp4_grouped_gemm_sparse(A_tiles, gA, W_sparse_tiles, gW, expert_offsets, E: int, T: int,
                              topk: int, N: int, K: int, route_token, route_slot, topk_weights,
                              out, workspace, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("nvfp4_grouped_gemm_sparse", load().nvfp4_grouped_gemm_sparse(
        _ptr(A_tiles), _ptr(gA), _ptr(W_sparse_tiles), _ptr(gW), _ptr(expert_offsets), E, T,
        topk, N, K, _ptr(route_token), _ptr(route_slot), _ptr(topk_weights), _ptr(out),
        _ptr(workspace), ws_bytes, _stream(stream)))


def nvfp4_decode_attention_workspace_bytes(B: int, Hq: int, Hkv: int, L_max: int, D: int) -> int:
    return load().nvfp4_decode_attention_workspace_bytes(B, Hq, Hkv, L_max, D)


def nvfp4_decode_attention(q, k_packed, k_scales, gk, v_packed, v_scales, gv, seq_lens,
                           scale: float, out, workspace, stream=None) -> None:
    """q BF16 [B, Hq, D]; caches [B, Hkv, L_max, D/2] codes and [.., D/16] scales."""
    B, Hq, D = q.shape
    _, Hkv, L_max, _ = k_packed.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("nvfp4_decode_attention", load().nvfp4_decode_attention(
        _ptr(q), _ptr(k_packed), _ptr(k_scales), _ptr(gk), _ptr(v_packed), _ptr(v_scales),
        _ptr(gv), _ptr(seq_lens), B, Hq, Hkv, L_max, D, float(scale), _ptr(out), _ptr(workspace),
        ws_bytes, _stream(stream)))


def nvfp4_noalloc_workspace_floats() -> int:
    return load().nvfp4_noalloc_workspace_floats()


def nvfp4_grouped_gemm_combine_noalloc(A_tiles, gA, W_tiles, gW, expert_offsets, E: int, T: int,
                                       topk: int, N: int, K: int, route_token, route_slot,
                                       topk_weights, out, stream=None) -> None:
    """Weighted-combine grouped GEMM using the library's own fixed workspace,
    for callers that cannot allocate device memory at call time (see the C
    header for the size limit and the rule that overlapping calls race)."""
    _check("nvfp4_grouped_gemm_combine_noalloc", load().nvfp4_grouped_gemm_combine_noalloc(
        _ptr(A_tiles), _ptr(gA), _ptr(W_tiles), _ptr(gW), _ptr(expert_offsets), E, T, topk, N,
        K, _ptr(route_token), _ptr(route_slot), _ptr(topk_weights), _ptr(out), _stream(stream)))


# ------------------------------------------- allocating conveniences (torch)

def quantize(x, atoms: bool = False, global_scale=None, stream=None):
    """BF16 [rows, cols] -> (packed, scales, g) with fresh device outputs."""
    rows, cols = x.shape
    dev = x.device
    packed = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    if atoms:
        scales = torch.empty(nvfp4_atom_scales_bytes(rows, cols), dtype=torch.uint8, device=dev)
    else:
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
    flags = NVFP4_SF_ATOMS if atoms else 0
    if global_scale is None:
        g = torch.empty(1, dtype=torch.float32, device=dev)
    else:
        g = global_scale
        flags |= NVFP4_GLOBAL_GIVEN
    nvfp4_quantize(x, packed, scales, g, flags, stream)
    return packed, scales, g


def moe_route(topk_ids, E: int, stream=None):
    """int32 [T, topk] -> (expert_offsets [E+1], route_token, route_slot, route_pos)."""
    T, k = topk_ids.shape
    dev = topk_ids.device
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    tok = torch.empty(T * k, dtype=torch.int32, device=dev)
    slot = torch.empty(T * k, dtype=torch.int32, device=dev)
    pos = torch.empty(T * k, dtype=torch.int32, device=dev)
    nvfp4_moe_route(topk_ids, E, off, tok, slot, pos, stream)
    return off, tok, slot, pos
