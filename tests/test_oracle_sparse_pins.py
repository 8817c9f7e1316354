"""Pins of the 2:4-sparse part of the oracle ("The FP4 Frontier", Finding 6).

Pruning is checked against a brute-force search over all six ways of
keeping two pairs of a group; the compressed form against its inverse and
against a product that reads the compressed bytes directly; the sparse tile
layout against its inverse, a covering of the tile's bytes and the dense
tile layout the tensor cores read.
"""
import itertools

import numpy as np
import pytest

import oracle
from moe_grouped_gemm_nvfp4_gb300 import inputs


def _bf16_values(g, shape, pool=None):
    if pool is not None:                       # few distinct magnitudes: many ties
        v = g.choice(np.asarray(pool, np.float32), size=shape)
        return v * np.where(g.random(shape) < 0.5, -1.0, 1.0).astype(np.float32)
    return inputs.to_bf16(g.standard_normal(shape, dtype=np.float32)).float().numpy()


def _brute_force_prune(w):
    """Per group: the two-pair subset with the largest exact score sum; among
    equal sums the lexicographically smallest positions."""
    out = np.zeros_like(w)
    rows, cols = w.shape
    for r in range(rows):
        for g in range(cols // 8):
            grp = w[r, 8 * g:8 * g + 8].astype(np.float64)
            score = [float(np.float32(abs(np.float32(grp[2 * i])))
                           + np.float32(abs(np.float32(grp[2 * i + 1]))))
                     for i in range(4)]
            best = None
            for sub in itertools.combinations(range(4), 2):
                tot = score[sub[0]] + score[sub[1]]
                if best is None or tot > best[0]:
                    best = (tot, sub)
            for i in best[1]:
                out[r, 8 * g + 2 * i:8 * g + 2 * i + 2] = w[r, 8 * g + 2 * i:8 * g + 2 * i + 2]
    return out


@pytest.mark.parametrize("pool", [None, [0.0, 0.5, 1.0, 2.0], [1.0], [0.0, 3.0]])
def test_prune_matches_brute_force(pool):
    g = inputs.rng(11)
    w = _bf16_values(g, (24, 64), pool)
    assert np.array_equal(oracle.prune_pairs_2of4(w), _brute_force_prune(w))


def test_prune_invariants():
    g = inputs.rng(12)
    w = _bf16_values(g, (40, 128))
    p = oracle.prune_pairs_2of4(w)
    pairs = p.reshape(40, 16, 4, 2)
    nz = (pairs != 0).any(axis=-1).sum(axis=-1)
    assert (nz <= 2).all()
    kept = p != 0
    assert np.array_equal(p[kept], w[kept])               # kept values unchanged
    assert np.array_equal(oracle.prune_pairs_2of4(p), p)  # idempotent
    # a group that already has two zero pairs is left alone
    w2 = w.copy()
    w2[:, 2:6] = 0.0
    assert np.array_equal(oracle.prune_pairs_2of4(w2)[:, :8], w2[:, :8])
    # pruned pairs are +0 (the quantiser then writes the byte 0x00)
    assert not np.signbit(p[p == 0]).any()


def test_combination_order_is_lexicographic():
    assert oracle.PAIR_COMBOS == ((0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3))


def _random_sparse_packed(g, rows, half):
    out = np.zeros((rows, half), np.uint8)
    special = np.array([0x00, 0x08, 0x80, 0x88, 0x01, 0xF7], np.uint8)   # signed zeros too
    for r in range(rows):
        for grp in range(half // 4):
            pos = g.choice(4, size=2, replace=False)
            for p in pos:
                out[r, 4 * grp + p] = (special[g.integers(len(special))] if g.random() < 0.3
                                       else g.integers(256))
    return out


def test_compress_round_trip_and_sizes():
    g = inputs.rng(13)
    packed = _random_sparse_packed(g, 33, 64)
    kept, combo = oracle.sparse_compress(packed)
    assert kept.shape == (33, 32) and combo.shape == (33, 16)
    assert combo.max() <= 5
    assert np.array_equal(oracle.sparse_decompress(kept, combo), packed)


def test_compress_every_mask():
    """Each group of <= 2 non-zero bytes: the stored positions cover the
    non-zero ones and are made up with the lowest zero positions."""
    for mask in range(16):
        grp = np.array([[(0x35 + 16 * i) if (mask >> i) & 1 else 0 for i in range(4)]], np.uint8)
        nz = [i for i in range(4) if (mask >> i) & 1]
        if len(nz) > 2:
            with pytest.raises(ValueError):
                oracle.sparse_compress(grp)
            continue
        kept, combo = oracle.sparse_compress(grp)
        pos = oracle.PAIR_COMBOS[int(combo[0, 0])]
        assert set(nz) <= set(pos)
        extra = sorted(set(pos) - set(nz))
        zeros = [i for i in range(4) if i not in nz]
        assert extra == zeros[:len(extra)]
        assert list(kept[0]) == [grp[0, pos[0]], grp[0, pos[1]]]


def test_pruned_then_quantised_is_2of4_over_bytes():
    g = inputs.rng(14)
    w = _bf16_values(g, (16, 256))
    p = oracle.prune_pairs_2of4(w)
    packed, sf, gs = oracle.quantize(p)
    kept, combo = oracle.sparse_compress(packed)          # raises if not 2:4
    assert np.array_equal(oracle.sparse_decompress(kept, combo), packed)
    # the global scale sees only the kept values
    assert gs == oracle.global_scale(p)


def test_sparse_product_equals_dense_gemm_of_pruned_weights():
    """The compressed form read directly (values placed by their combination
    index) gives the same product as the dense GEMM of the pruned weights."""
    g = inputs.rng(15)
    w = oracle.prune_pairs_2of4(_bf16_values(g, (24, 128)))
    x = _bf16_values(g, (5, 128))
    wp, ws, wg = oracle.quantize(w)
    xp, xs, xg = oracle.quantize(x)
    kept, combo = oracle.sparse_compress(wp)
    got = oracle.sparse_rowwise_product(kept, combo, ws, wg, oracle.dequantize(xp, xs, xg))
    ref = oracle.gemm(xp, xs, xg, wp, ws, wg)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # a wrong combination table changes the product
    combo_bad = combo.copy()
    combo_bad[combo_bad == 1] = 2
    bad = oracle.sparse_rowwise_product(kept, combo_bad, ws, wg, oracle.dequantize(xp, xs, xg))
    assert not np.allclose(bad, ref)


def test_sparse_tile_offsets_cover_the_tile_once():
    r = np.arange(128)[:, None]
    kept = oracle.sparse_kept_offset(0, r, 0, np.arange(64)[None, :], 1).ravel()
    cb, sh = oracle.sparse_combo_offset(0, r, 0, np.arange(32)[None, :], 1)
    combo_bytes = np.unique(cb.ravel())
    assert combo_bytes.size == 128 * 16
    # every combination byte holds exactly two groups, one per nibble
    pairs = {(int(b), int(s)) for b, s in zip(cb.ravel(), np.broadcast_to(sh, cb.shape).ravel())}
    assert len(pairs) == 128 * 32
    scales = oracle.sparse_scale_offset(0, r, 0, np.arange(16)[None, :], 1).ravel()
    allb = np.concatenate([kept, combo_bytes, scales])
    assert np.array_equal(np.sort(allb), np.arange(oracle.SPARSE_TILE_BYTES))


@pytest.mark.parametrize("rows,K", [(128, 256), (200, 320), (64, 1024)])
def test_sparse_tiles_round_trip(rows, K):
    g = inputs.rng(16)
    packed = _random_sparse_packed(g, rows, K // 2)
    sf = g.integers(0, 127, size=(rows, K // 16), dtype=np.uint8)
    buf = oracle.sparse_operand_tiles(packed, sf)
    n_rt, n_kb = -(-rows // 128), -(-K // 256)
    assert buf.size == n_rt * n_kb * oracle.SPARSE_TILE_BYTES
    p2, s2 = oracle.sparse_operand_rows(buf, rows, K)
    assert np.array_equal(p2, packed) and np.array_equal(s2, sf)


def test_sparse_tiles_expand_to_the_dense_tiles():
    g = inputs.rng(17)
    rows, K = 200, 512
    packed = _random_sparse_packed(g, rows, K // 2)
    sf = g.integers(0, 127, size=(rows, K // 16), dtype=np.uint8)
    buf = oracle.sparse_operand_tiles(packed, sf)
    dense = oracle.sparse_tiles_to_dense_tiles(buf, 2, 2)
    assert np.array_equal(dense, oracle.operand_tiles(packed, sf))
    # the sparse form is two thirds of the dense one
    assert buf.size * 3 == dense.size * 2
