"""The C-ABI library builds, loads without a GPU and exports every entry point
declared in include/nvfp4.h; host-side validation rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

from moe_grouped_gemm_nvfp4_gb300 import build, nvfp4 as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("nvfp4_quantize", "nvfp4_prepack_weights", "nvfp4_gemm", "nvfp4_grouped_gemm",
                 "nvfp4_grouped_gemm_tiles", "nvfp4_moe_route", "nvfp4_quantize_dispatch",
                 "nvfp4_prepacked_scales_bytes", "nvfp4_grouped_gemm_workspace_bytes",
                 "nvfp4_last_device_status"):
        assert want in names


def test_library_exports_every_declared_symbol():
    path = build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    # and the Python binding wraps every one of them under the same name
    for n in _declared():
        assert hasattr(F, n), n


def test_pure_host_helpers():
    assert F.nvfp4_version() == 100
    assert F.nvfp4_status_string(4) == "NVFP4_ERR_TIMEOUT"
    assert F.nvfp4_status_string(99) == "NVFP4_ERR_UNKNOWN"
    assert F.nvfp4_atom_scales_bytes(300, 512) == 384 * 32
    assert F.nvfp4_atom_scales_bytes(0, 512) == 0
    assert F.nvfp4_combine_workspace_bytes(256, 6144) == 256 * 6144 * 4
    # grouped GEMM on plain operands: activation tiles (+ FP32 sums with the combine)
    tiles_2048 = (2048 + 31 * 128) // 32 * 24 * 18432
    assert F.nvfp4_grouped_gemm_workspace_bytes(256, 8, 128, 4096, 6144, False) == tiles_2048
    assert F.nvfp4_grouped_gemm_workspace_bytes(256, 8, 128, 6144, 2048, True) == \
        (2048 + 31 * 128) // 32 * 8 * 18432 + 256 * 6144 * 4
    assert F.nvfp4_prepacked_scales_bytes(300, 32) == F.nvfp4_atom_scales_bytes(300, 512)
    assert F.nvfp4_prepacked_scales_bytes(1, 3) == 128 * 4      # kblk padded to 4
    # operand tiles: 18432 bytes per 128 rows x 256 K
    assert F.nvfp4_operand_tiles_bytes(300, 512) == 3 * 2 * 18432
    assert F.nvfp4_operand_tiles_bytes(128, 64) == 18432
    # grouped tiles: chunk width from the mean routes per expert; every non-empty
    # expert wastes at most chunk - 1 rows
    assert F.nvfp4_grouped_chunk_rows(2048, 128) == 32        # 16 per expert
    assert F.nvfp4_grouped_chunk_rows(4096, 128) == 64        # 32 per expert
    assert F.nvfp4_grouped_chunk_rows(6144, 128) == 64        # 48 per expert
    assert F.nvfp4_grouped_chunk_rows(8192, 128) == 128       # 64 per expert
    assert F.nvfp4_grouped_chunk_rows(12288, 128) == 128      # 96 per expert
    assert F.nvfp4_grouped_chunk_rows(65536, 128) == 128
    # tiles proper + 16 KB of scratch for the tensor amax's per-block maxima
    assert F.nvfp4_grouped_tiles_bytes(2048, 128, 6144) == \
        (2048 + 31 * 128) // 32 * 24 * 18432 + 16384
    assert F.nvfp4_grouped_tiles_bytes(1, 128, 64) == 18432 + 16384
    # 2:4-sparse tiles: 12288 bytes per 128 rows x 256 K, two thirds of a dense tile
    assert F.nvfp4_sparse_tiles_bytes(300, 512) == 3 * 2 * 12288
    assert F.nvfp4_sparse_tiles_bytes(128 * 4096, 6144) * 3 == \
        F.nvfp4_operand_tiles_bytes(128 * 4096, 6144) * 2
    assert F.nvfp4_sparse_tiles_bytes(-1, 64) == 0
    # decode attention: per (sequence, query head, split) D partial values + max + sum
    assert F.nvfp4_decode_attention_workspace_bytes(2, 8, 2, 1000, 128) == 2 * 8 * 8 * 130 * 4
    # 2048-token splits: ~1024 (sequence, KV head, split) work items
    assert F.nvfp4_decode_attention_workspace_bytes(16, 32, 8, 16384, 128) == \
        16 * 32 * (16384 // 2048) * 130 * 4
    # 512-wide heads also hold every token's score per query head
    assert F.nvfp4_decode_attention_workspace_bytes(8, 8, 2, 32768, 512) == \
        8 * 8 * (32768 // 512) * 514 * 4 + 8 * 8 * 32768 * 4
    assert F.nvfp4_decode_attention_workspace_bytes(16, 8, 8, 65536, 512) == \
        16 * 8 * (65536 // 4096) * 514 * 4 + 16 * 8 * 65536 * 4   # 4096-token splits
    assert F.nvfp4_decode_attention_workspace_bytes(0, 8, 2, 1000, 128) == 0


def test_host_validation_without_device():
    lib = F.load()
    # null operands / bad sizes return INVALID_ARG before any CUDA call
    assert lib.nvfp4_gemm(None, None, None, None, None, None, None, 16, 16, 64, 16, None) == 1
    assert lib.nvfp4_quantize(None, -1, 16, 16, None, None, None, 0, None) == 1
    assert lib.nvfp4_quantize(None, 4, 16, 16, None, None, None, 0, None) == 1
    assert lib.nvfp4_moe_route(None, 4, 0, 8, None, None, None, None, None) == 1
    assert lib.nvfp4_grouped_gemm_tiles(*([None] * 5), 8, 4, 2, 128, 128, None, None, None,
                                        None, None, 0, None) == 1
    assert lib.nvfp4_grouped_gemm(*([None] * 7), 8, None, None, None, 4, 2, 128, 128, None,
                                  None, 0, None) == 1
    assert lib.nvfp4_prepack_weight_tiles(None, None, 4, 64, None, None) == 1
    assert lib.nvfp4_set_timeout_ns(0) == 1
    assert lib.nvfp4_device_status(None, 0, None) == 1
    assert lib.nvfp4_amax_partials(None, 4, 64, 64, 8, 2, None, None) == 1
    assert lib.nvfp4_moe_gate_up_silu(*([None] * 5), 4, 8, 2, 256, 128, None, None, None) == 1
    assert lib.nvfp4_grouped_gemm_combine_noalloc(*([None] * 5), 4, 8, 2, 128, 128,
                                                  None, None, None, None, None) == 1
    assert lib.nvfp4_grouped_gemm_sparse(*([None] * 5), 8, 4, 2, 128, 128, None, None, None,
                                         None, None, 0, None) == 1
    assert lib.nvfp4_prune_2of4(None, 4, 16, 16, None, 16, None) == 1
    assert lib.nvfp4_prune_2of4(None, 4, 16, 8, None, 16, None) == 1           # ld < cols
    assert lib.nvfp4_prepack_sparse_weight_tiles(None, None, 4, 64, None, None) == 1
    assert lib.nvfp4_decode_attention(*([None] * 8), 1, 4, 1, 16, 64, 0.1, None, None, 0,
                                      None) == 1
    assert lib.nvfp4_decode_attention(*([None] * 8), 1, 6, 4, 16, 64, 0.1, None, None, 0,
                                      None) == 1                                # Hq % Hkv
    # unsupported shapes are refused before any CUDA call too
    p = ctypes.c_void_p(256)
    assert lib.nvfp4_gemm(p, p, p, p, p, p, p, 16, 16, 48, 16, None) == 2
    assert lib.nvfp4_quantize(p, 4, 24, 24, p, p, p, 0, None) == 2
    assert lib.nvfp4_amax_partials(p, 4, 48, 48, 8, 2, p, None) == 2            # K % 64
    assert lib.nvfp4_prune_2of4(p, 4, 12, 12, p, 12, None) == 2                 # cols % 8
    assert lib.nvfp4_prepack_sparse_weight_tiles(p, p, 4, 96, p, None) == 2     # K % 64
    assert lib.nvfp4_grouped_gemm_sparse(p, p, p, p, p, 4, 8, 2, 200, 128, p, p, None, p,
                                         None, 0, None) == 2                     # N % 128
    # the plain-operand grouped GEMM: N % 128, then a workspace that is too small
    assert lib.nvfp4_grouped_gemm(*([p] * 7), 8, p, None, p, 4, 2, 200, 128, p, p, 1 << 30,
                                  None) == 2
    assert lib.nvfp4_grouped_gemm(*([p] * 7), 8, p, None, p, 4, 2, 256, 128, p, p, 1024,
                                  None) == 2
    q = ctypes.c_void_p(4096)
    assert lib.nvfp4_decode_attention(*([q] * 8), 1, 4, 1, 16, 96, 0.1, q, q, 1 << 20,
                                      None) == 2                                # head width
    assert lib.nvfp4_decode_attention(*([q] * 8), 1, 16, 1, 16, 128, 0.1, q, q, 1 << 20,
                                      None) == 2                                # group of 16
    assert lib.nvfp4_decode_attention(*([q] * 8), 1, 4, 1, 16, 128, 0.1, q, q, 16,
                                      None) == 2                                # workspace
    # fused MLP: N must split into gate and up halves of whole 128-row tiles
    assert lib.nvfp4_moe_gate_up_silu(p, p, p, p, p, 4, 8, 2, 384, 128, p, p, None) == 2
    # conflicting quantiser flags: a given global and amax maxima already present
    assert lib.nvfp4_quantize_dispatch(p, 4, 64, 64, p, 2, p, 4, 8, p, p,
                                       F.NVFP4_GLOBAL_GIVEN | F.NVFP4_AMAX_DONE, None) == 1


def test_binding_raises_without_cuda_tensors():
    import torch
    x = torch.zeros((4, 16), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        F.quantize(x)
