"""Plain CPU restatement of NVFP4 quantisation and (grouped) block-scaled GEMM.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Format and recipe
-----------------
* The element format is E2M1: 1 sign, 2 exponent and 1 mantissa bit
  ("The Blackwell architectural split", Preserving precision -- dual-tier
  scale handling).  Two elements share a byte; the element with the lower
  K index sits in the low nibble.
* Scaling is dual-tier: one FP32 global scale per tensor plus one block
  scale per 16 consecutive values along K (same section).  The block scale
  is FP8 E4M3; block scale s = (block_amax / 6) / g with the global
  g = tensor_amax / (6 * 448), so that x ~ e2m1 * e4m3(s) * g.
* Every quantiser step is an IEEE binary32 operation rounded to nearest
  even, in the order written below; E4M3 and E2M1 encodings round to
  nearest even and saturate to the largest finite value.
* GEMM: C = (gA * gB) * sum_k e2m1(A) sfA * e2m1(B) sfB, i.e. the exact
  product of the dequantised operands; written in FP64 here.
* MoE grouped GEMM ("The FP4 Frontier", Finding 5: grouped GEMM over all
  experts): each expert's GEMM runs on the token rows routed to it; the
  down projection combines the routes of a token with its routing weights.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "E2M1_TABLE", "e4m3_decode", "e4m3_encode", "e2m1_encode",
    "global_scale", "quantize", "pack_codes", "unpack_codes", "dequantize",
    "gemm", "route", "grouped_gemm", "combine", "prepack_scales",
    "unprepack_scales", "grouped_sf_layout", "sf_tiles_per_expert",
    "TILE_BYTES", "operand_tiles", "grouped_operand_tiles", "tile_byte_offset",
    "tile_scale_offset", "grouped_operand_rows", "silu", "silu_mul",
]

F32 = np.float32

# ---------------------------------------------------------------------------
# Element and scale formats
# ---------------------------------------------------------------------------

# E2M1 decoded through a 16-entry table indexed by the 4-bit code
# (bit 3 = sign, bits 2..1 = exponent, bit 0 = mantissa).
E2M1_TABLE = np.array(
    [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
     -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=np.float64)


def e4m3_decode(code) -> np.ndarray:
    """FP8 E4M3 (bias 7, no infinities) decoded by bit field, as float64.

    Exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN.
    """
    c = np.asarray(code, dtype=np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


# The 127 non-negative finite E4M3 values, ascending with the code.
_E4M3_POS = e4m3_decode(np.arange(127))


def _nearest_even(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the grid value nearest to each |x|; ties go to the even index.

    `grid` is ascending and indexed by code, so "even index" is "even
    mantissa".  Values beyond the last grid point saturate to it.
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(grid, mag, side="left")
    hi = np.clip(hi, 1, len(grid) - 1)
    lo = hi - 1
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= grid[-1], len(grid) - 1, idx)
    idx = np.where(mag <= grid[0], 0, idx)
    return idx.astype(np.int64)


def e4m3_encode(s) -> np.ndarray:
    """FP32 -> E4M3 code: round to nearest even, saturate to +-448."""
    s = np.asarray(s, dtype=np.float32).astype(np.float64)
    code = _nearest_even(np.abs(s), _E4M3_POS)
    return (code | (np.signbit(s).astype(np.int64) << 7)).astype(np.uint8)


_E2M1_MAG = E2M1_TABLE[:8]


def e2m1_encode(q) -> np.ndarray:
    """FP32 -> E2M1 code: round to nearest even, saturate to +-6, sign kept."""
    q = np.asarray(q, dtype=np.float32).astype(np.float64)
    code = _nearest_even(np.abs(q), _E2M1_MAG)
    return (code | (np.signbit(q).astype(np.int64) << 3)).astype(np.uint8)


# ---------------------------------------------------------------------------
# Quantiser
# ---------------------------------------------------------------------------

def global_scale(x) -> np.float32:
    """g = tensor_amax / (6 * 448), one FP32 division."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x)) if x.size else F32(0.0)
    return F32(F32(amax) / F32(6.0 * 448.0))


def quantize(x, g=None):
    """BF16/FP32 matrix [rows, cols] (cols % 16 == 0) -> NVFP4.

    Returns (packed uint8 [rows, cols/2], scales uint8 [rows, cols/16],
    g float32).  If g is given it is used as the global scale.

    Steps, all binary32 round-to-nearest-even:
      1. g = tensor_amax / 2688                       (unless given)
      2. per 16-block: amax_b; s = (amax_b / 6) / g   (s = 0 when g == 0)
      3. sf = E4M3(s);  d = decode(sf) * g
      4. per element: code = E2M1(x / d), or the signed zero code when d == 0
      5. pack two codes per byte, low nibble = lower K index
    """
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % 16 == 0
    g = global_scale(x) if g is None else F32(g)
    xb = x.reshape(rows, cols // 16, 16)
    amax_b = np.max(np.abs(xb), axis=2) if cols else np.zeros((rows, 0), F32)
    if g > 0:
        s = (amax_b / F32(6.0)) / g
    else:
        s = np.zeros_like(amax_b)
    sf = e4m3_encode(s)
    d = (e4m3_decode(sf).astype(np.float32) * g).astype(np.float32)
    dd = d[:, :, None]
    safe = np.where(dd == 0, F32(1.0), dd)
    with np.errstate(over="ignore", invalid="ignore"):
        q = (xb / safe).astype(np.float32)
    codes = e2m1_encode(q)
    zero_code = (np.signbit(xb).astype(np.uint8) << 3).astype(np.uint8)
    codes = np.where(dd == 0, zero_code, codes).reshape(rows, cols)
    return pack_codes(codes), sf, g


def pack_codes(codes) -> np.ndarray:
    """[rows, cols] 4-bit codes -> [rows, cols/2] bytes, low nibble = even K."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    """[rows, cols/2] bytes -> [rows, cols] 4-bit codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def dequantize(packed, scales, g) -> np.ndarray:
    """x_hat = E2M1[code] * E4M3[sf] * g, exact in float64."""
    codes = unpack_codes(packed)
    rows, cols = codes.shape
    vals = E2M1_TABLE[codes].reshape(rows, cols // 16, 16)
    sfv = e4m3_decode(np.asarray(scales))[:, :, None]
    return (vals * sfv * np.float64(g)).reshape(rows, cols)


# ---------------------------------------------------------------------------
# GEMM, routing, grouped GEMM, combine
# ---------------------------------------------------------------------------

def gemm(a_packed, sfa, ga, b_packed, sfb, gb) -> np.ndarray:
    """C[M, N] = A_hat @ B_hat^T in float64 (A: [M, K/2], B: [N, K/2])."""
    return dequantize(a_packed, sfa, ga) @ dequantize(b_packed, sfb, gb).T


def route(topk_ids, E):
    """Counting sort of the (token, slot) routes by expert, stable by token.

    Returns (expert_offsets int32 [E+1], route_token int32 [R],
    route_slot int32 [R]) where the routes of expert e are positions
    expert_offsets[e] .. expert_offsets[e+1]-1, in ascending token order.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)                       # flat index i = t * k + slot
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets, (order // k).astype(np.int32), (order % k).astype(np.int32)


def grouped_gemm(a_hat_rows, w_hat, expert_offsets) -> np.ndarray:
    """Per expert e: Y[p] = a_hat_rows[p] @ w_hat[e]^T for its routes p.

    a_hat_rows: float64 [R, K], the dequantised activation of every route
    in sorted order; w_hat: float64 [E, N, K].  Returns float64 [R, N].
    """
    R = a_hat_rows.shape[0]
    E, N, _ = w_hat.shape
    y = np.zeros((R, N), dtype=np.float64)
    for e in range(E):
        lo, hi = int(expert_offsets[e]), int(expert_offsets[e + 1])
        if hi > lo:
            y[lo:hi] = a_hat_rows[lo:hi] @ w_hat[e].T
    return y


def silu(z) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)), in float64 (the usual
    definition; the pages name the gated MLP, not its formula)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def silu_mul(y_gate_up) -> np.ndarray:
    """Expert MLP gate: y [R, N] -> h [R, N/2] = SiLU(y[:, :N/2]) * y[:, N/2:]
    (rows [0, N/2) of the gate_up weight are the gate projection, rows
    [N/2, N) the up projection of the same features), float64.  The fused
    step between the two projections of "The FP4 Frontier", Finding 5."""
    y = np.asarray(y_gate_up, dtype=np.float64)
    half = y.shape[1] // 2
    return silu(y[:, :half]) * y[:, half:]


def combine(y, route_token, route_slot, topk_weights, T) -> np.ndarray:
    """out[t] = sum over the routes p of token t of w[t, slot(p)] * y[p] (float64)."""
    w = np.asarray(topk_weights, dtype=np.float64)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for p in range(y.shape[0]):
        t = int(route_token[p])
        out[t] += w[t, int(route_slot[p])] * y[p]
    return out


# ---------------------------------------------------------------------------
# Scale-factor layouts consumed by the tensor cores
# ---------------------------------------------------------------------------
# Scales are stored in 512-byte atoms covering 128 rows x 4 consecutive
# scale columns (64 K-elements): byte (r % 32) * 16 + ((r % 128) // 32) * 4
# + (c % 4).  Atoms are ordered row-tile major, scale-column-group minor.

def _atom_offset(r, c, n_cgroups):
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    atom = (r // 128) * n_cgroups + c // 4
    return atom * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def prepack_scales(sf) -> np.ndarray:
    """Row-major scales [rows, ks] (ks % 4 == 0) -> atom layout, rows padded to 128."""
    sf = np.asarray(sf, dtype=np.uint8)
    rows, ks = sf.shape
    assert ks % 4 == 0
    rows_pad = -(-rows // 128) * 128
    out = np.zeros(rows_pad * ks, dtype=np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(ks), indexing="ij")
    out[_atom_offset(r, c, ks // 4)] = sf
    return out


def unprepack_scales(buf, rows, ks) -> np.ndarray:
    """Inverse of prepack_scales."""
    buf = np.asarray(buf, dtype=np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(ks), indexing="ij")
    return buf[_atom_offset(r, c, ks // 4)]


def sf_tiles_per_expert(expert_offsets) -> np.ndarray:
    """128-row scale tiles per expert: ceil(count_e / 128)."""
    off = np.asarray(expert_offsets, dtype=np.int64)
    return -(-(off[1:] - off[:-1]) // 128)


def grouped_sf_layout(sf_routes, expert_offsets) -> np.ndarray:
    """Route-ordered scales [R, ks] -> per-expert atom layout.

    Expert e's routes start a fresh 128-row tile: route p of expert e sits in
    padded row 128 * tb[e] + (p - offsets[e]), tb[e] = sum over e' < e of
    ceil(count_e' / 128).  Padding bytes are zero.
    """
    sf = np.asarray(sf_routes, dtype=np.uint8)
    R, ks = sf.shape
    off = np.asarray(expert_offsets, dtype=np.int64)
    tiles = sf_tiles_per_expert(off)
    tb = np.concatenate([[0], np.cumsum(tiles)])
    out = np.zeros(int(tb[-1]) * 128 * ks, dtype=np.uint8)
    for e in range(len(tiles)):
        for p in range(int(off[e]), int(off[e + 1])):
            prow = 128 * int(tb[e]) + (p - int(off[e]))
            out[_atom_offset(prow, np.arange(ks), ks // 4)] = sf[p]
    return out


# ---------------------------------------------------------------------------
# Operand tiles: the layout a pipeline stage copies in one piece
# ---------------------------------------------------------------------------
# A tile covers 128 rows x 256 K-elements.  Its first 16384 bytes are the
# packed codes, row r at r * 128, with the 16-byte chunk j of a row stored at
# chunk position j XOR (r % 8) (the 128-byte shared-memory swizzle of the
# tensor cores); the next 2048 bytes are the tile's scales as four 512-byte
# atoms, one per 64-element K step.  Tiles are ordered row-tile major, then
# K block; a tile is 18432 bytes.

TILE_BYTES = 16384 + 2048


def tile_byte_offset(rt, r, kb, c, n_kb):
    """Byte of packed byte c (0..127) of row r in row tile rt, K block kb."""
    rt, r, kb, c = (np.asarray(v, dtype=np.int64) for v in (rt, r, kb, c))
    return ((rt * n_kb + kb) * TILE_BYTES + r * 128 + (((c >> 4) ^ (r & 7)) << 4) + (c & 15))


def tile_scale_offset(rt, r, kb, s, n_kb):
    """Byte of scale column s (0..15) of row r in row tile rt, K block kb."""
    rt, r, kb, s = (np.asarray(v, dtype=np.int64) for v in (rt, r, kb, s))
    return ((rt * n_kb + kb) * TILE_BYTES + 16384 + (s >> 2) * 512 + (r & 31) * 16
            + ((r >> 5) & 3) * 4 + (s & 3))


def _scatter_rows(out, packed, sf, rows_rt, rows_r, n_kb):
    """Writes rows (packed [n, K/2], sf [n, K/16]) to row tiles rows_rt, rows rows_r."""
    n, half = packed.shape
    c = np.arange(half)
    out[tile_byte_offset(rows_rt[:, None], rows_r[:, None], c[None, :] // 128,
                         c[None, :] % 128, n_kb)] = packed
    s = np.arange(sf.shape[1])
    out[tile_scale_offset(rows_rt[:, None], rows_r[:, None], s[None, :] // 16,
                          s[None, :] % 16, n_kb)] = sf


def operand_tiles(packed, sf):
    """Packed [rows, K/2] + row-major scales [rows, K/16] -> tile layout.

    Rows are padded to a multiple of 128 and K to a multiple of 256; padding
    bytes are zero.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    sf = np.asarray(sf, dtype=np.uint8)
    rows, half = packed.shape
    n_rt = -(-rows // 128)
    n_kb = -(-(2 * half) // 256)
    out = np.zeros(n_rt * n_kb * TILE_BYTES, dtype=np.uint8)
    r = np.arange(rows)
    _scatter_rows(out, packed, sf, r // 128, r % 128, n_kb)
    return out


def grouped_operand_tiles(packed_routes, sf_routes, expert_offsets, chunk_rows=128):
    """Route-ordered rows -> tiles where each expert's routes are cut into
    chunks of `chunk_rows` (32, 64 or 128) and every chunk starts a fresh row
    tile: route p of expert e, local index j = p - offsets[e], is row
    j % chunk_rows of tile tb[e] + j // chunk_rows, with tb[e] = sum over
    e' < e of ceil(count_e' / chunk_rows)."""
    packed = np.asarray(packed_routes, dtype=np.uint8)
    sf = np.asarray(sf_routes, dtype=np.uint8)
    R, half = packed.shape
    off = np.asarray(expert_offsets, dtype=np.int64)
    counts = off[1:] - off[:-1]
    chunks = -(-counts // chunk_rows)
    tb = np.concatenate([[0], np.cumsum(chunks)])
    n_kb = -(-(2 * half) // 256)
    out = np.zeros(int(tb[-1]) * n_kb * TILE_BYTES, dtype=np.uint8)
    for e in range(len(counts)):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            j = np.arange(hi - lo)
            _scatter_rows(out, packed[lo:hi], sf[lo:hi], tb[e] + j // chunk_rows,
                          j % chunk_rows, n_kb)
    return out


def grouped_operand_rows(buf, expert_offsets, K, chunk_rows):
    """Inverse of grouped_operand_tiles: the tile buffer -> (packed [R, K/2],
    scales [R, K/16]) of the routes, read back from the same positions."""
    buf = np.asarray(buf, dtype=np.uint8)
    off = np.asarray(expert_offsets, dtype=np.int64)
    counts = off[1:] - off[:-1]
    chunks = -(-counts // chunk_rows)
    tb = np.concatenate([[0], np.cumsum(chunks)])
    n_kb = -(-K // 256)
    R = int(off[-1])
    packed = np.zeros((R, K // 2), np.uint8)
    sf = np.zeros((R, K // 16), np.uint8)
    c = np.arange(K // 2)
    sc = np.arange(K // 16)
    for e in range(len(counts)):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            j = np.arange(hi - lo)
            rt = (tb[e] + j // chunk_rows)[:, None]
            r = (j % chunk_rows)[:, None]
            packed[lo:hi] = buf[tile_byte_offset(rt, r, c[None, :] // 128, c[None, :] % 128, n_kb)]
            sf[lo:hi] = buf[tile_scale_offset(rt, r, sc[None, :] // 16, sc[None, :] % 16, n_kb)]
    return packed, sf
