"""Pins of the decode-attention oracle ("The Blackwell architectural split",
The A4Q Kernel): against the library's scaled-dot-product attention, closed
forms (one token, identical keys, empty sequence), the convex-hull property
and the grouped-query head mapping."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_nvfp4_gb300 import inputs


def _random(g, B, Hq, Hkv, L, D):
    q = g.standard_normal((B, Hq, D))
    k = g.standard_normal((B, Hkv, L, D))
    v = g.standard_normal((B, Hkv, L, D))
    return q, k, v


@pytest.mark.parametrize("B,Hq,Hkv,L,D", [(2, 4, 4, 37, 64), (3, 8, 2, 50, 128), (1, 6, 1, 9, 32)])
def test_matches_library_attention(B, Hq, Hkv, L, D):
    g = inputs.rng(B * 100 + Hq + L)
    q, k, v = _random(g, B, Hq, Hkv, L, D)
    lens = g.integers(1, L + 1, size=B)
    lens[0] = L
    scale = 1.0 / np.sqrt(D)
    got = oracle.decode_attention(q, k, v, lens, scale)
    G = Hq // Hkv
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1)          # [B, Hq, L, D]
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1)
    qt = torch.from_numpy(q)[:, :, None, :]                       # one query per sequence
    mask = torch.arange(L)[None, None, None, :] < torch.from_numpy(lens)[:, None, None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(got, ref[:, :, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_closed_forms():
    g = inputs.rng(7)
    q, k, v = _random(g, 1, 2, 1, 16, 64)
    # one token: the output is that token's value
    out = oracle.decode_attention(q, k, v, [1], 0.125)
    assert np.array_equal(out[0, 0], v[0, 0, 0]) and np.array_equal(out[0, 1], v[0, 0, 0])
    # identical keys: uniform weights, the mean of the values
    k_same = np.repeat(k[:, :, :1], 16, axis=2)
    out = oracle.decode_attention(q, k_same, v, [16], 0.125)
    np.testing.assert_allclose(out[0, 0], v[0, 0].mean(axis=0), rtol=1e-13, atol=1e-14)
    # empty sequence: zeros
    out = oracle.decode_attention(q, k, v, [0], 0.125)
    assert not out.any()
    # a convex combination of the values, coordinate by coordinate
    out = oracle.decode_attention(q, k, v, [16], 0.5)
    assert (out[0] >= v[0, 0].min(axis=0) - 1e-12).all()
    assert (out[0] <= v[0, 0].max(axis=0) + 1e-12).all()


def test_grouped_heads_read_their_own_kv_head():
    """Constant values per KV head: query head h must return the constant of
    KV head h // G (consecutive grouping)."""
    g = inputs.rng(8)
    B, Hq, Hkv, L, D = 1, 8, 2, 12, 32
    q, k, _ = _random(g, B, Hq, Hkv, L, D)
    v = np.zeros((B, Hkv, L, D))
    v[0, 0] = 1.0
    v[0, 1] = -2.0
    out = oracle.decode_attention(q, k, v, [L], 0.2)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], 1.0 if h // 4 == 0 else -2.0, rtol=1e-13)


def test_kv_quantisation_is_the_row_quantiser():
    g = inputs.rng(9)
    x = inputs.to_bf16(g.standard_normal((2, 3, 5, 64), dtype=np.float32)).float().numpy()
    gk = oracle.global_scale(x)
    p, s = oracle.quantize_kv(x, gk)
    assert p.shape == (2, 3, 5, 32) and s.shape == (2, 3, 5, 4)
    p2, s2, _ = oracle.quantize(x.reshape(-1, 64), g=gk)
    assert np.array_equal(p.reshape(-1, 32), p2) and np.array_equal(s.reshape(-1, 4), s2)
    xh = oracle.dequantize_kv(p, s, gk)
    # NVFP4 keeps each element within half a step of its block's grid
    assert np.abs(xh - x).max() <= np.abs(x).max() / 6 * 1.01
