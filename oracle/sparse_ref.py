"""Plain CPU restatement of 2:4-sparse NVFP4 weights.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

"The FP4 Frontier", Finding 6 (sparse FP4 assessment): structured 2:4
sparsity halves the bits an NVFP4 weight occupies, and in an MoE model every
expert can be pruned on its own.  The page fixes neither the granularity,
nor the pruning criterion, nor a storage format.  The readings written here:

* Granularity.  The unit is the packed byte, i.e. the pair of E2M1 values at
  K = 2i, 2i+1.  Along K, every aligned group of four bytes (eight values)
  keeps at most two non-zero bytes: 2:4 over element pairs, 50% density.
* Pruning (BF16 weights, before quantisation).  Pair i scores
  |w[2i]| + |w[2i+1]| in one binary32 addition; in each group the two pairs
  with the highest scores stay, ties going to the lower position; the other
  two pairs become +0.  The pruned tensor is then quantised with the ordinary
  recipe (its global and block scales see only the kept values), so every
  pruned pair is the byte 0x00.
* Storage.  Per group: the two kept bytes in position order, and the
  combination index c of their positions (i0 < i1) in lexicographic order:
  (0,1) (0,2) (0,3) (1,2) (1,3) (2,3) -> c = 0..5.  A group with fewer than
  two non-zero bytes keeps the lowest zero positions to make up two.

The GEMM over sparse weights is the ordinary GEMM of the pruned, quantised
weights (the zeros contribute exact zeros), so its oracle is `gemm` /
`grouped_gemm` on the pruned operand.
"""
from __future__ import annotations

import itertools

import numpy as np

from .nvfp4_ref import TILE_BYTES, tile_byte_offset, tile_scale_offset

__all__ = [
    "PAIR_COMBOS", "prune_pairs_2of4", "sparse_compress", "sparse_decompress",
    "SPARSE_TILE_BYTES", "sparse_kept_offset", "sparse_combo_offset",
    "sparse_scale_offset", "sparse_operand_tiles", "sparse_operand_rows",
    "sparse_tiles_to_dense_tiles", "sparse_rowwise_product",
]

F32 = np.float32

# positions (i0, i1) of the two kept bytes of a group, by combination index
PAIR_COMBOS = tuple(itertools.combinations(range(4), 2))


def prune_pairs_2of4(w) -> np.ndarray:
    """BF16-valued [rows, cols] (cols % 8 == 0) -> the pruned copy, float32.

    Per group of four pairs, the two pairs with the highest binary32 score
    |a| + |b| stay (ties: lower position); the others become +0.
    """
    w = np.asarray(w, dtype=F32)
    rows, cols = w.shape
    assert cols % 8 == 0
    pairs = w.reshape(rows, cols // 8, 4, 2).copy()
    score = np.abs(pairs[..., 0]) + np.abs(pairs[..., 1])          # float32 adds
    # descending score; the stable sort keeps equal scores in position order
    order = np.argsort(-score, axis=-1, kind="stable")
    drop = order[..., 2:]
    np.put_along_axis(pairs[..., 0], drop, F32(0.0), axis=-1)
    np.put_along_axis(pairs[..., 1], drop, F32(0.0), axis=-1)
    return pairs.reshape(rows, cols)


def _kept_positions(mask):
    """Kept positions (i0 < i1) of a group whose non-zero bytes form the 4-bit
    mask: the non-zero positions, made up to two with the lowest zero ones.
    None when more than two bytes are non-zero."""
    nz = [i for i in range(4) if (mask >> i) & 1]
    if len(nz) > 2:
        return None
    pos = list(nz)
    for i in range(4):
        if len(pos) == 2:
            break
        if i not in pos:
            pos.append(i)
    return tuple(sorted(pos))


# non-zero mask -> combination index (-1: not 2:4)
_MASK_COMBO = np.array([PAIR_COMBOS.index(_kept_positions(m)) if _kept_positions(m) else -1
                        for m in range(16)], dtype=np.int64)


def sparse_compress(packed):
    """Packed codes [rows, K/2] with at most two non-zero bytes in every group
    of four -> (kept [rows, K/4] bytes, combo [rows, K/8] indices 0..5)."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    assert half % 4 == 0
    grp = packed.reshape(rows, half // 4, 4)
    mask = ((grp != 0).astype(np.int64) << np.arange(4)).sum(axis=-1)
    combo = _MASK_COMBO[mask]
    if (combo < 0).any():
        r, g = np.argwhere(combo < 0)[0]
        raise ValueError(f"row {r} group {g}: more than two non-zero bytes")
    pos = np.array(PAIR_COMBOS, dtype=np.int64)[combo]                  # [rows, groups, 2]
    kept = np.take_along_axis(grp, pos, axis=-1).reshape(rows, half // 2)
    return kept.astype(np.uint8), combo.astype(np.uint8)


def sparse_decompress(kept, combo) -> np.ndarray:
    """Inverse of sparse_compress: (kept, combo) -> packed codes [rows, K/2]."""
    kept = np.asarray(kept, dtype=np.uint8)
    combo = np.asarray(combo, dtype=np.int64)
    rows, ng = combo.shape
    out = np.zeros((rows, ng, 4), np.uint8)
    pos = np.array(PAIR_COMBOS, dtype=np.int64)[combo]
    np.put_along_axis(out, pos, kept.reshape(rows, ng, 2), axis=-1)
    return out.reshape(rows, 4 * ng)


# ---------------------------------------------------------------------------
# Sparse operand tiles
# ---------------------------------------------------------------------------
# A sparse tile covers the same 128 rows x 256 K-elements as a dense operand
# tile and holds 12288 bytes:
#   [0, 8192)       kept bytes: K slice j (64 elements, 16 kept bytes per
#                   row) of row r at j * 2048 + r * 16;
#   [8192, 10240)   combination indices, one 4-bit field per group: half h
#                   (128 elements, 16 groups) of row r at 8192 + h * 1024 +
#                   r * 8, group g of the half in byte g // 2 (low nibble
#                   for even g);
#   [10240, 12288)  the scales, laid out as in the dense tile (four 512-byte
#                   atoms).
# Tiles are ordered row-tile major, then K block.

SPARSE_TILE_BYTES = 12288


def sparse_kept_offset(rt, r, kb, i, n_kb):
    """Byte of kept byte i (0..63) of row r in row tile rt, K block kb."""
    rt, r, kb, i = (np.asarray(v, dtype=np.int64) for v in (rt, r, kb, i))
    return (rt * n_kb + kb) * SPARSE_TILE_BYTES + (i >> 4) * 2048 + r * 16 + (i & 15)


def sparse_combo_offset(rt, r, kb, g, n_kb):
    """(byte, nibble shift) of the combination index of group g (0..31) of row
    r in row tile rt, K block kb."""
    rt, r, kb, g = (np.asarray(v, dtype=np.int64) for v in (rt, r, kb, g))
    byte = ((rt * n_kb + kb) * SPARSE_TILE_BYTES + 8192 + (g >> 4) * 1024 + r * 8
            + ((g & 15) >> 1))
    return byte, 4 * (g & 1)


def sparse_scale_offset(rt, r, kb, s, n_kb):
    """Byte of scale column s (0..15) of row r in row tile rt, K block kb."""
    rt, r, kb, s = (np.asarray(v, dtype=np.int64) for v in (rt, r, kb, s))
    return ((rt * n_kb + kb) * SPARSE_TILE_BYTES + 10240 + (s >> 2) * 512 + (r & 31) * 16
            + ((r >> 5) & 3) * 4 + (s & 3))


def sparse_operand_tiles(packed, sf):
    """Packed [rows, K/2] (2:4 over bytes) + row-major scales [rows, K/16] ->
    sparse tiles.  Rows are padded to a multiple of 128 and K to a multiple of
    256 with zero bytes (whose groups are stored as combination 0)."""
    packed = np.asarray(packed, dtype=np.uint8)
    sf = np.asarray(sf, dtype=np.uint8)
    rows, half = packed.shape
    n_rt = -(-rows // 128)
    n_kb = -(-(2 * half) // 256)
    pp = np.zeros((n_rt * 128, n_kb * 128), np.uint8)
    pp[:rows, :half] = packed
    kept, combo = sparse_compress(pp)
    out = np.zeros(n_rt * n_kb * SPARSE_TILE_BYTES, np.uint8)
    r = np.arange(n_rt * 128)[:, None]
    i = np.arange(kept.shape[1])[None, :]
    out[sparse_kept_offset(r // 128, r % 128, i // 64, i % 64, n_kb)] = kept
    g = np.arange(combo.shape[1])
    for gg in g:
        byte, sh = sparse_combo_offset(r[:, 0] // 128, r[:, 0] % 128, gg // 32, gg % 32, n_kb)
        out[byte] |= (combo[:, gg] << sh).astype(np.uint8)
    s = np.arange(sf.shape[1])[None, :]
    rr = np.arange(rows)[:, None]
    out[sparse_scale_offset(rr // 128, rr % 128, s // 16, s % 16, n_kb)] = sf
    return out


def sparse_operand_rows(buf, rows, K):
    """Inverse of sparse_operand_tiles: the tile buffer -> (packed [rows, K/2],
    scales [rows, K/16]), read back from the same positions."""
    buf = np.asarray(buf, dtype=np.uint8)
    n_kb = -(-K // 256)
    r = np.arange(rows)[:, None]
    i = np.arange(K // 4)[None, :]
    kept = buf[sparse_kept_offset(r // 128, r % 128, i // 64, i % 64, n_kb)]
    combo = np.zeros((rows, K // 8), np.uint8)
    for g in range(K // 8):
        byte, sh = sparse_combo_offset(r[:, 0] // 128, r[:, 0] % 128, g // 32, g % 32, n_kb)
        combo[:, g] = (buf[byte] >> sh) & 0xF
    s = np.arange(K // 16)[None, :]
    sf = buf[sparse_scale_offset(r // 128, r % 128, s // 16, s % 16, n_kb)]
    return sparse_decompress(kept, combo), sf


def sparse_tiles_to_dense_tiles(buf, n_rt, n_kb):
    """What expanding every sparse tile yields: the dense operand tiles of the
    same codes and scales (the layout the tensor cores read)."""
    buf = np.asarray(buf, dtype=np.uint8)
    rows, K = n_rt * 128, n_kb * 256
    packed, sf = sparse_operand_rows(buf, rows, K)
    out = np.zeros(n_rt * n_kb * TILE_BYTES, np.uint8)
    r = np.arange(rows)[:, None]
    c = np.arange(K // 2)[None, :]
    out[tile_byte_offset(r // 128, r % 128, c // 128, c % 128, n_kb)] = packed
    s = np.arange(K // 16)[None, :]
    out[tile_scale_offset(r // 128, r % 128, s // 16, s % 16, n_kb)] = sf
    return out


def sparse_rowwise_product(kept, combo, w_scale_rows, g_w, x_hat):
    """Y[m, n] = sum over the kept values of row n only: an independent
    formulation of the sparse GEMM that reads the compressed form directly.

    kept / combo: compressed weights [N, K/4] / [N, K/8]; w_scale_rows: E4M3
    scale codes [N, K/16]; g_w: the weights' global; x_hat: dequantised
    activations [M, K] (float64).  Returns float64 [M, N].
    """
    from .nvfp4_ref import E2M1_TABLE, e4m3_decode
    kept = np.asarray(kept, dtype=np.uint8)
    combo = np.asarray(combo, dtype=np.uint8)
    N = kept.shape[0]
    M, K = x_hat.shape
    sfv = e4m3_decode(np.asarray(w_scale_rows, dtype=np.uint8))
    y = np.zeros((M, N))
    for n in range(N):
        acc = np.zeros(M)
        for g in range(K // 8):
            pos = PAIR_COMBOS[int(combo[n, g])]
            for t in range(2):
                byte = int(kept[n, 2 * g + t])
                for nib in range(2):
                    k = 8 * g + 2 * pos[t] + nib
                    v = E2M1_TABLE[(byte >> (4 * nib)) & 0xF] * sfv[n, k // 16] * float(g_w)
                    acc += v * x_hat[:, k]
        y[:, n] = acc
    return y
