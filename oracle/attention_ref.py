"""Plain CPU restatement of decode attention over an NVFP4 KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

"The Blackwell architectural split", The Breakthrough -- The A4Q Kernel and
Preserving precision: attention whose keys and values are held in NVFP4
(E2M1 values, an E4M3 scale per 16 numbers, a global tensor scale for K and
one for V) and dequantised inside the attention loop.  The pages fix the
format, not the attention arithmetic; the readings written here:

* Decode: one query token per sequence.  q is BF16 [B, Hq, D]; the cache
  holds, for sequence b and KV head j, seq_len[b] tokens of K and V, each
  token a D-vector quantised in 16-element blocks along D with the cache's
  global scale (one for K, one for V).
* Grouped query heads: G = Hq / Hkv, query head h reads KV head h // G.
* out[b, h] = sum_t p_t v_hat_t with p = softmax(scale * q . k_hat_t) over
  t < seq_len[b]; an empty sequence gives a zero output.  Everything in
  float64 here; the dequantised K and V are exact (see `dequantize`).
"""
from __future__ import annotations

import numpy as np

from .nvfp4_ref import dequantize, quantize

__all__ = ["quantize_kv", "dequantize_kv", "decode_attention"]


def quantize_kv(x, g):
    """BF16-valued cache [..., D] -> (packed [..., D/2], scales [..., D/16]),
    quantised along D with the given global g (the ordinary NVFP4 recipe)."""
    x = np.asarray(x, dtype=np.float32)
    shape = x.shape
    p, s, _ = quantize(x.reshape(-1, shape[-1]), g=np.float32(g))
    return p.reshape(*shape[:-1], shape[-1] // 2), s.reshape(*shape[:-1], shape[-1] // 16)


def dequantize_kv(packed, scales, g):
    """Inverse direction of quantize_kv, exact in float64."""
    packed = np.asarray(packed)
    D = packed.shape[-1] * 2
    out = dequantize(packed.reshape(-1, D // 2), np.asarray(scales).reshape(-1, D // 16), g)
    return out.reshape(*packed.shape[:-1], D)


def decode_attention(q, k_hat, v_hat, seq_lens, scale):
    """q [B, Hq, D]; k_hat, v_hat [B, Hkv, L, D] (dequantised, float64);
    seq_lens [B]; returns float64 [B, Hq, D]."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_hat.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(seq_lens[b])
        if n == 0:
            continue
        for h in range(Hq):
            j = h // G
            s = scale * (k_hat[b, j, :n] @ q[b, h])
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ v_hat[b, j, :n]
    return out
