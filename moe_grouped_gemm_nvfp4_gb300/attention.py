"""Decode attention over an NVFP4 KV cache: cache quantisation and the call.

Argument marshalling around the C ABI ("The Blackwell architectural split",
The A4Q Kernel: the cache stays in NVFP4 and is dequantised inside the
attention loop).  The arithmetic runs in the CUDA kernels.
"""
from __future__ import annotations

import torch

from . import nvfp4 as F


def quantize_kv(x: torch.Tensor, g: torch.Tensor = None, stream=None):
    """BF16 cache [B, Hkv, L, D] -> (codes [B, Hkv, L, D/2], scales [B, Hkv, L,
    D/16], g).  g: the cache's global (device float [1]); computed from this
    tensor's amax when not given."""
    B, Hkv, L, D = x.shape
    dev = x.device
    packed = torch.empty((B, Hkv, L, D // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((B, Hkv, L, D // 16), dtype=torch.uint8, device=dev)
    flags = 0
    if g is None:
        g = torch.empty(1, dtype=torch.float32, device=dev)
    else:
        flags = F.NVFP4_GLOBAL_GIVEN
    F.nvfp4_quantize(x.reshape(B * Hkv * L, D), packed.view(B * Hkv * L, D // 2),
                     scales.view(B * Hkv * L, D // 16), g, flags, stream)
    return packed, scales, g


class DecodeAttention:
    """Workspace and output for one decode-attention shape."""

    def __init__(self, B: int, Hq: int, Hkv: int, L_max: int, D: int, device="cuda"):
        self.shape = (B, Hq, Hkv, L_max, D)
        nbytes = F.nvfp4_decode_attention_workspace_bytes(B, Hq, Hkv, L_max, D)
        self.workspace = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=device)
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)

    def run(self, q, k, v, seq_lens, scale: float, stream=None):
        """k = (codes, scales, g) and v likewise, as from quantize_kv."""
        F.nvfp4_decode_attention(q, k[0], k[1], k[2], v[0], v[1], v[2], seq_lens, scale,
                                 self.out, self.workspace, stream)
        return self.out
