"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against the format definitions, closed forms,
library routines for special cases, brute force on tiny inputs, or exact
rational arithmetic, so that a dropped term, wrong sign, wrong index or
transposed operand in the oracle fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_nvfp4_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- E2M1 ------

def test_e2m1_table_matches_representable_set():
    for code, val in _read("e2m1_values.txt"):
        got = oracle.E2M1_TABLE[int(code)]
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e2m1_table_matches_bit_fields():
    # 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is subnormal.
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + 0.5 * m)
        assert oracle.E2M1_TABLE[code] == (-mag if s else mag)


def test_e2m1_encode_midpoints_and_saturation():
    for q, val, code in _read("e2m1_rne_midpoints.txt"):
        got = int(oracle.e2m1_encode(np.float32(float(q))))
        assert got == int(code), (q, got, code)
        assert oracle.E2M1_TABLE[got] == float(val)


def test_e2m1_encode_round_trips_every_code():
    assert list(oracle.e2m1_encode(oracle.E2M1_TABLE)) == list(range(16))


def test_e2m1_encode_brute_force():
    # Argmin of |q - v| over the 8 magnitudes, ties to the even code, on a
    # dense grid that includes every midpoint and values past saturation.
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    grid = np.concatenate([np.arange(0, 8.0, 1 / 64), [0.2500001, 6.5, 1e6]])
    grid = np.concatenate([grid, -grid]).astype(np.float32)
    got = oracle.e2m1_encode(grid)
    for q, c in zip(grid.tolist(), got.tolist()):
        d = [abs(abs(q) - v) for v in mags]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        want = [i for i in cands if i % 2 == 0][0] if len(cands) > 1 else cands[0]
        want |= 8 if math.copysign(1.0, q) < 0 else 0
        assert c == want, (q, c, want)


# ---------------------------------------------------------------- E4M3 ------

def test_e4m3_decode_golden_points():
    for code, val in _read("e4m3_points.txt"):
        got = float(oracle.e4m3_decode(int(code, 16)))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(np.arange(256))
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert np.sum(np.isnan(got)) == 2


def test_e4m3_encode_matches_torch_below_overflow():
    # torch's float8_e4m3fn cast rounds to nearest even; below the overflow
    # midpoint (464) it must agree with the oracle code for code.
    g = inputs.rng(123)
    s = np.concatenate([
        g.uniform(0, 464, 20000), g.uniform(0, 1e-2, 20000), np.exp2(g.uniform(-12, 8.8, 20000)),
        oracle.e4m3_decode(np.arange(127)),
        (oracle.e4m3_decode(np.arange(126)) + oracle.e4m3_decode(np.arange(1, 127))) / 2,
    ]).astype(np.float32)
    s = s[s < 464]
    ref = torch.from_numpy(s).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(s)
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates_and_underflows():
    assert int(oracle.e4m3_encode(np.float32(448.0))) == 0x7E
    assert int(oracle.e4m3_encode(np.float32(448.00003))) == 0x7E
    assert int(oracle.e4m3_encode(np.float32(1e9))) == 0x7E
    assert int(oracle.e4m3_encode(np.float32(2.0 ** -10))) == 0x00   # tie -> even (0)
    assert int(oracle.e4m3_encode(np.float32(2.0 ** -10 * 1.0001))) == 0x01
    assert int(oracle.e4m3_encode(np.float32(2.0 ** -9))) == 0x01


def test_e4m3_round_trip_and_monotone():
    codes = np.arange(127)
    vals = oracle.e4m3_decode(codes)
    assert np.all(np.diff(vals) > 0)
    assert np.array_equal(oracle.e4m3_encode(vals.astype(np.float32)), codes.astype(np.uint8))


# ------------------------------------------------------------- quantiser ----

def _exact_block_tensor(g, rows, cols):
    """Blocks x = v * S * g with v in E2M1 and S in E4M3, block max = 6 S."""
    gglob = 0.125                                     # tensor amax 336 = 2688 * 0.125
    codes = g.integers(0, 16, (rows, cols)).astype(np.uint8)
    codes.reshape(rows, -1, 16)[:, :, 0] = 7          # every block holds +6
    S = oracle.e4m3_decode(g.integers(0x08, 0x7E, (rows, cols // 16)))
    S[0, 0] = 448.0
    x = oracle.E2M1_TABLE[codes].reshape(rows, -1, 16) * S[:, :, None] * gglob
    return x.reshape(rows, cols).astype(np.float32), codes, S, gglob


def test_quantize_exact_round_trip_of_representable_blocks():
    g = inputs.rng(7)
    x, codes, S, gg = _exact_block_tensor(g, 6, 64)
    packed, sf, gq = oracle.quantize(x)
    assert gq == np.float32(gg)
    assert np.array_equal(oracle.e4m3_decode(sf), S)
    # negative zero and positive zero both decode to 0; compare the values
    assert np.array_equal(oracle.dequantize(packed, sf, gq), x.astype(np.float64))
    nz = oracle.E2M1_TABLE[codes] != 0
    assert np.array_equal(oracle.unpack_codes(packed)[nz], codes[nz])


def test_quantize_zero_block_and_zero_tensor():
    x = np.zeros((2, 32), np.float32)
    x[0, 16:] = np.linspace(-3, 3, 16)
    x[1, :16] = -0.0
    packed, sf, g = oracle.quantize(x)
    assert sf[0, 0] == 0 and sf[1, 0] == 0 and sf[1, 1] == 0
    codes = oracle.unpack_codes(packed)
    assert np.all(codes[0, :16] == 0)
    assert np.all(codes[1, :16] == 8)              # -0 keeps its sign bit
    p2, s2, g2 = oracle.quantize(np.zeros((3, 16), np.float32))
    assert g2 == 0 and np.all(s2 == 0) and np.all(p2 == 0)


def test_quantize_block_max_is_six_in_normal_scale_range():
    g = inputs.rng(11)
    x = inputs.normal_bf16(g, (64, 256)).float().numpy()
    x[:, 100:116] *= 1e-3                            # small blocks, still normal scale
    packed, sf, gq = oracle.quantize(x)
    codes = oracle.unpack_codes(packed).reshape(64, 16, 16)
    mags = np.abs(oracle.E2M1_TABLE[codes])
    normal = oracle.e4m3_decode(sf) >= 2.0 ** -6
    assert normal.sum() > 0.9 * normal.size
    assert np.all(mags.max(axis=2)[normal] == 6.0)


def test_quantize_sign_symmetry():
    g = inputs.rng(12)
    x = inputs.normal_bf16(g, (16, 128)).float().numpy()
    p1, s1, g1 = oracle.quantize(x)
    p2, s2, g2 = oracle.quantize(-x)
    assert g1 == g2 and np.array_equal(s1, s2)
    assert np.array_equal(oracle.unpack_codes(p2), oracle.unpack_codes(p1) ^ 8)


def test_quantize_power_of_two_scaling():
    g = inputs.rng(13)
    x = inputs.normal_bf16(g, (8, 128)).float().numpy()
    p1, s1, g1 = oracle.quantize(x)
    for j in (-3, 5):
        p2, s2, g2 = oracle.quantize(x * np.float32(2.0 ** j))
        assert g2 == np.float32(g1 * 2.0 ** j)
        assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def test_quantize_codes_minimise_error_brute_force():
    # For every element: the chosen magnitude is the nearest E2M1 value to
    # |x| / d (exact rational), except where the binary32 quotient sits on a
    # midpoint, where the even code wins.
    g = inputs.rng(14)
    x = inputs.normal_bf16(g, (4, 64)).float().numpy()
    packed, sf, gq = oracle.quantize(x)
    codes = oracle.unpack_codes(packed)
    mags = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    for r in range(4):
        for c in range(64):
            d = Fraction(float(np.float32(oracle.e4m3_decode(sf[r, c // 16]) * np.float64(gq))))
            q = abs(Fraction(float(x[r, c]))) / d
            dist = [abs(q - m) for m in mags]
            best = min(dist)
            chosen = int(codes[r, c]) & 7
            assert dist[chosen] <= best + Fraction(1, 2 ** 20) * max(q, 1)


def test_quantize_scale_is_nearest_e4m3_brute_force():
    g = inputs.rng(15)
    x = inputs.normal_bf16(g, (8, 64)).float().numpy() * np.float32(3.7)
    _, sf, gq = oracle.quantize(x)
    grid = [Fraction(float(v)) for v in oracle.e4m3_decode(np.arange(127))]
    amax_b = np.abs(x.reshape(8, 4, 16)).max(axis=2)
    for r in range(8):
        for b in range(4):
            s = Fraction(float(np.float32(np.float32(amax_b[r, b] / np.float32(6)) / gq)))
            dist = [abs(s - v) for v in grid]
            best = min(dist)
            cands = [i for i, di in enumerate(dist) if di == best]
            want = [i for i in cands if i % 2 == 0][0] if len(cands) > 1 else cands[0]
            assert int(sf[r, b]) == want


# ------------------------------------------------------------------ GEMM ----

def _exact_gemm(a_codes, a_sf, ga, b_codes, b_sf, gb):
    """Exact rational C = A_hat B_hat^T from codes (pure Python)."""
    e2 = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    def val(code, sf, g):
        v = e2[code & 7] * (-1 if code & 8 else 1)
        return v * Fraction(float(oracle.e4m3_decode(sf))) * Fraction(float(g))
    M, K = a_codes.shape
    N = b_codes.shape[0]
    C = [[Fraction(0)] * N for _ in range(M)]
    A = [[Fraction(0)] * N for _ in range(M)]       # sum of |terms|, for the error bound
    for i in range(M):
        for j in range(N):
            terms = [val(int(a_codes[i, k]), int(a_sf[i, k // 16]), ga) *
                     val(int(b_codes[j, k]), int(b_sf[j, k // 16]), gb) for k in range(K)]
            C[i][j] = sum(terms)
            A[i][j] = sum(abs(t) for t in terms)
    return C, A


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (3, 4, 32), (4, 2, 64)])
def test_gemm_matches_exact_rationals(M, N, K):
    g = inputs.rng(100 + M * N * K)
    a = inputs.normal_bf16(g, (M, K)).float().numpy()
    b = inputs.normal_bf16(g, (N, K), 0.02).float().numpy()
    pa, sa, ga = oracle.quantize(a)
    pb, sb, gb = oracle.quantize(b)
    C = oracle.gemm(pa, sa, ga, pb, sb, gb)
    E, A = _exact_gemm(oracle.unpack_codes(pa), sa, ga, oracle.unpack_codes(pb), sb, gb)
    # FP64 dot-product error bound: |C - exact| <= gamma_(K+1) * sum |a_k b_k|
    gamma = (K + 1) * 2.0 ** -53 / (1 - (K + 1) * 2.0 ** -53)
    for i in range(M):
        for j in range(N):
            err = abs(Fraction(float(C[i, j])) - E[i][j])
            assert err <= Fraction(gamma) * A[i][j]


def test_gemm_one_hot_reproduces_rows_of_b():
    # A built in code space: one E2M1 "1.0" (code 2) per row, scale 0x38 (=1), g = 1.
    g = inputs.rng(21)
    N, K = 8, 64
    b = inputs.normal_bf16(g, (N, K), 0.02).float().numpy()
    pb, sb, gb = oracle.quantize(b)
    bhat = oracle.dequantize(pb, sb, gb)
    for kk in (0, 17, 63):
        codes = np.zeros((1, K), np.uint8)
        codes[0, kk] = 2
        sa = np.full((1, K // 16), 0x38, np.uint8)
        C = oracle.gemm(oracle.pack_codes(codes), sa, 1.0, pb, sb, gb)
        assert np.array_equal(C[0], bhat[:, kk])


def test_gemm_transpose_and_operand_order():
    # C(A, B) = C(B, A)^T, and a K=16 product is a single-block dot product.
    g = inputs.rng(22)
    a = inputs.normal_bf16(g, (5, 16)).float().numpy()
    b = inputs.normal_bf16(g, (3, 16)).float().numpy()
    pa, sa, ga = oracle.quantize(a)
    pb, sb, gb = oracle.quantize(b)
    C1 = oracle.gemm(pa, sa, ga, pb, sb, gb)
    C2 = oracle.gemm(pb, sb, gb, pa, sa, ga)
    assert np.array_equal(C1, C2.T)
    ca = oracle.E2M1_TABLE[oracle.unpack_codes(pa)]
    cb = oracle.E2M1_TABLE[oracle.unpack_codes(pb)]
    scale = oracle.e4m3_decode(sa) * oracle.e4m3_decode(sb).T * float(ga) * float(gb)
    dot = (ca @ cb.T) * scale                      # codes dot-product, one block scale pair
    bound = 40 * 2.0 ** -53 * (np.abs(ca) @ np.abs(cb).T) * scale
    assert np.all(np.abs(C1 - dot) <= bound)


# --------------------------------------------------------- routing, MoE -----

def test_route_matches_brute_force():
    g = inputs.rng(31)
    T, E, k = 37, 9, 3
    ids = inputs.uniform_topk(g, T, E, k)
    off, tok, slot = oracle.route(ids, E)
    p = 0
    for e in range(E):
        assert off[e] == p
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    assert tok[p] == t and slot[p] == j
                    p += 1
    assert off[E] == p == T * k


def test_route_empty_experts_and_single_token():
    off, tok, slot = oracle.route(np.array([[3, 1]], np.int32), 5)
    assert list(off) == [0, 0, 1, 1, 2, 2]
    assert list(tok) == [0, 0] and list(slot) == [1, 0]


def test_grouped_single_expert_equals_dense():
    g = inputs.rng(41)
    T, K, N = 7, 64, 16
    x = inputs.normal_bf16(g, (T, K)).float().numpy()
    w = inputs.normal_bf16(g, (N, K), 0.02).float().numpy()
    px, sx, gx = oracle.quantize(x)
    pw, sw, gw = oracle.quantize(w)
    off, tok, slot = oracle.route(np.zeros((T, 1), np.int32), 1)
    xh = oracle.dequantize(px, sx, gx)[tok]
    y = oracle.grouped_gemm(xh, oracle.dequantize(pw, sw, gw)[None], off)
    assert np.array_equal(y, oracle.gemm(px, sx, gx, pw, sw, gw))


def test_combine_one_hot_weights_is_a_gather():
    g = inputs.rng(42)
    T, E, k, N = 6, 4, 2, 5
    ids = inputs.uniform_topk(g, T, E, k)
    off, tok, slot = oracle.route(ids, E)
    y = g.standard_normal((T * k, N))
    w = np.zeros((T, k), np.float32)
    w[:, 1] = 1.0
    out = oracle.combine(y, tok, slot, w, T)
    for t in range(T):
        p = [i for i in range(T * k) if tok[i] == t and slot[i] == 1][0]
        assert np.array_equal(out[t], y[p])


def test_combine_is_linear_in_weights():
    g = inputs.rng(43)
    T, E, k, N = 5, 3, 2, 4
    ids = inputs.uniform_topk(g, T, E, k)
    off, tok, slot = oracle.route(ids, E)
    y = g.standard_normal((T * k, N))
    w1, w2 = inputs.dirichlet_weights(g, T, k), inputs.dirichlet_weights(g, T, k)
    lhs = oracle.combine(y, tok, slot, w1.astype(np.float64) + w2, T)
    rhs = oracle.combine(y, tok, slot, w1, T) + oracle.combine(y, tok, slot, w2, T)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- scale layouts ------

def test_atom_layout_golden_offsets():
    rows, ks = 300, 8
    sf = np.zeros((rows, ks), np.uint8)
    pts = [tuple(map(int, r)) for r in _read("sf_atom_offsets.txt")]
    for i, (r, c, _) in enumerate(pts):
        sf[r, c] = i + 1
    buf = oracle.prepack_scales(sf)
    assert buf.size == 384 * ks
    for i, (r, c, off) in enumerate(pts):
        assert buf[off] == i + 1, (r, c, off)


def test_prepack_is_a_bijection():
    g = inputs.rng(51)
    sf = g.integers(0, 256, (200, 12)).astype(np.uint8)
    buf = oracle.prepack_scales(sf)
    assert np.array_equal(oracle.unprepack_scales(buf, 200, 12), sf)
    # every (row, col) lands on a distinct byte; padding rows stay zero
    sf1 = np.arange(200 * 12).reshape(200, 12)
    pos = np.zeros(buf.size, np.int64)
    for r in range(200):
        for c in range(12):
            one = np.zeros((200, 12), np.uint8)
            one[r, c] = 1
            pos += oracle.prepack_scales(one)
    assert pos.max() == 1 and pos.sum() == sf1.size


def test_grouped_sf_layout_padding():
    off = np.array([0, 3, 3, 133, 140], np.int64)      # counts 3, 0, 130, 7
    R, ks = 140, 4
    sf = (np.arange(R * ks).reshape(R, ks) % 251 + 1).astype(np.uint8)
    buf = oracle.grouped_sf_layout(sf, off)
    assert list(oracle.sf_tiles_per_expert(off)) == [1, 0, 2, 1]
    assert buf.size == 4 * 128 * ks
    # expert 2's local row 129 sits in its second tile (tile 2 overall), row 1 of it
    p = 3 + 129
    base = (1 + 1) * 512
    for c in range(ks):
        assert buf[base + 1 * 16 + c] == sf[p, c]
    # expert 3 starts a fresh tile (tile 3)
    assert buf[3 * 512 + 0 * 16 + 2] == sf[133, 2]


def test_operand_tile_golden_offsets():
    rows, K = 300, 512
    n_kb = K // 256
    for kind, r, col, off in _read("tile_offsets.txt"):
        r, col, off = int(r), int(col), int(off)
        if kind == "b":
            got = oracle.tile_byte_offset(r // 128, r % 128, col // 128, col % 128, n_kb)
        else:
            got = oracle.tile_scale_offset(r // 128, r % 128, col // 16, col % 16, n_kb)
        assert int(got) == off, (kind, r, col, int(got), off)


def test_operand_tiles_bijection_and_swizzle():
    g = inputs.rng(61)
    rows, K = 200, 768
    packed = g.integers(0, 256, (rows, K // 2)).astype(np.uint8)
    sf = g.integers(0, 256, (rows, K // 16)).astype(np.uint8)
    buf = oracle.operand_tiles(packed, sf)
    assert buf.size == 2 * 3 * oracle.TILE_BYTES
    # every byte of the input lands on a distinct position
    pos_b = oracle.tile_byte_offset(np.arange(rows)[:, None] // 128, np.arange(rows)[:, None] % 128,
                                    np.arange(K // 2)[None, :] // 128,
                                    np.arange(K // 2)[None, :] % 128, 3)
    pos_s = oracle.tile_scale_offset(np.arange(rows)[:, None] // 128,
                                     np.arange(rows)[:, None] % 128,
                                     np.arange(K // 16)[None, :] // 16,
                                     np.arange(K // 16)[None, :] % 16, 3)
    allpos = np.concatenate([pos_b.ravel(), pos_s.ravel()])
    assert np.unique(allpos).size == allpos.size
    assert np.array_equal(buf[pos_b], packed) and np.array_equal(buf[pos_s], sf)
    # the scale part of a tile is the atom layout of its 128 rows x 16 scale columns
    tile0_sf = buf[16384:18432]
    assert np.array_equal(tile0_sf, oracle.prepack_scales(sf[:128, :16]))
    # within a tile, a row's 128 bytes are its 8 chunks permuted by XOR with row % 8
    r = 13
    row = buf[r * 128:(r + 1) * 128].reshape(8, 16)
    for j in range(8):
        assert np.array_equal(row[j ^ (r % 8)], packed[r, 16 * j:16 * (j + 1)])


def test_grouped_operand_tiles_layout():
    g = inputs.rng(62)
    off = np.array([0, 3, 3, 133, 140], np.int64)
    R, K = 140, 256
    packed = g.integers(0, 256, (R, K // 2)).astype(np.uint8)
    sf = g.integers(0, 256, (R, K // 16)).astype(np.uint8)
    buf = oracle.grouped_operand_tiles(packed, sf, off)
    assert buf.size == 4 * oracle.TILE_BYTES
    # expert 2, local row 129 -> second tile of expert 2 (tile 2), row 1
    p = 3 + 129
    t = 2 * oracle.TILE_BYTES
    assert np.array_equal(buf[t + 128:t + 256].reshape(8, 16)[0 ^ 1], packed[p, :16])
    assert buf[t + 16384 + 1 * 16 + 0] == sf[p, 0]


def test_grouped_operand_tiles_chunks():
    g = inputs.rng(63)
    off = np.array([0, 70, 70, 75], np.int64)          # counts 70, 0, 5
    R, K = 75, 256
    packed = g.integers(0, 256, (R, K // 2)).astype(np.uint8)
    sf = g.integers(0, 256, (R, K // 16)).astype(np.uint8)
    buf = oracle.grouped_operand_tiles(packed, sf, off, chunk_rows=32)
    assert buf.size == (3 + 1) * oracle.TILE_BYTES       # 70 -> 3 chunks, 5 -> 1 chunk
    # expert 0, local row 40 -> chunk 1 (tile 1), row 8; its scales are in group 0 of the atom
    t = oracle.TILE_BYTES
    assert np.array_equal(buf[t + 8 * 128:t + 9 * 128].reshape(8, 16)[0], packed[40, :16])
    assert buf[t + 16384 + 8 * 16 + 0] == sf[40, 0]
    # expert 2 starts tile 3
    assert buf[3 * t + 16384 + 2 * 16 + 1] == sf[72, 1]
    # chunk_rows = 128 reproduces the 128-row layout
    assert np.array_equal(oracle.grouped_operand_tiles(packed, sf, off),
                          oracle.grouped_operand_tiles(packed, sf, off, chunk_rows=128))


def test_grouped_operand_rows_inverts_the_layout():
    """Reading the tiles back at the same byte positions returns every route's
    codes and scales (chunks of 32 and 128, an empty expert, a ragged K block)."""
    g = inputs.rng(64)
    off = np.array([0, 5, 5, 45, 46], np.int64)
    R, K = 46, 320
    packed = g.integers(0, 256, (R, K // 2)).astype(np.uint8)
    sf = g.integers(0, 256, (R, K // 16)).astype(np.uint8)
    for chunk in (32, 128):
        buf = oracle.grouped_operand_tiles(packed, sf, off, chunk_rows=chunk)
        p2, s2 = oracle.grouped_operand_rows(buf, off, K, chunk)
        assert np.array_equal(p2, packed) and np.array_equal(s2, sf)


def test_silu_closed_forms():
    """sigmoid(ln 3) = 3/4, so SiLU(ln 3) = (3/4) ln 3; SiLU(z) - SiLU(-z) = z
    because sigmoid(-z) = 1 - sigmoid(z); SiLU(0) = 0; SiLU(z) -> z and -> 0
    for large |z| (no overflow warning at the far end)."""
    ln3 = np.log(3.0)
    assert abs(oracle.silu(ln3) - 0.75 * ln3) <= 4 * np.finfo(np.float64).eps
    z = np.linspace(-20.0, 20.0, 41)
    assert np.allclose(oracle.silu(z) - oracle.silu(-z), z, rtol=0, atol=1e-13)
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(800.0) == 800.0 and oracle.silu(-800.0) == 0.0


def test_silu_mul_uses_the_first_half_as_gate():
    """y = [gate | up]: with up = 1 the product is SiLU(gate); swapping the
    halves changes it (a transposed gate/up reading fails here)."""
    gate = np.array([[-2.0, 0.5, 3.0]])
    up = np.array([[1.0, 1.0, 1.0]])
    h = oracle.silu_mul(np.concatenate([gate, up], axis=1))
    assert np.allclose(h, oracle.silu(gate), rtol=0, atol=0)
    h2 = oracle.silu_mul(np.concatenate([up, gate], axis=1))
    assert not np.allclose(h2, h)
    assert np.allclose(h2, oracle.silu(1.0) * gate)


# ------------------------------------------- grouped GEMM across experts ----

def _expert_of_route(off, p):
    """The expert whose route range [off[e], off[e+1]) holds p, by a linear scan."""
    for e in range(len(off) - 1):
        if int(off[e]) <= p < int(off[e + 1]):
            return e
    raise AssertionError(f"route {p} outside every expert range")


def test_grouped_gemm_many_experts_matches_per_route_exact_rationals():
    """Several experts with uneven counts and an empty one: every route's row
    is the exact rational dot product of its decoded activation with the rows
    of its own expert's decoded weight ("The FP4 Frontier", Finding 5: one
    grouped GEMM over all experts).  A wrong expert index or an off-by-one in
    the offset slices changes rows of distinct random weights, so it fails."""
    g = inputs.rng(47)
    E, N, K = 4, 3, 32
    # uneven routing: expert 0 gets 4 routes, expert 1 none, expert 2 one,
    # expert 3 five (tokens 0..4, top-2)
    ids = np.array([[0, 3], [3, 0], [0, 3], [3, 2], [0, 3]], np.int32)
    T = ids.shape[0]
    x = inputs.normal_bf16(g, (T, K)).float().numpy()
    w = inputs.normal_bf16(g, (E, N, K), 0.5).float().numpy()
    off, tok, slot = oracle.route(ids, E)
    assert [int(off[e + 1] - off[e]) for e in range(E)] == [4, 0, 1, 5]
    xh = oracle.dequantize(*oracle.quantize(x))[tok]
    wh = np.stack([oracle.dequantize(*oracle.quantize(w[e])) for e in range(E)])
    y = oracle.grouped_gemm(xh, wh, off)
    gamma = (K + 1) * 2.0 ** -53 / (1 - (K + 1) * 2.0 ** -53)
    for p in range(T * 2):
        e = _expert_of_route(off, p)
        assert ids[tok[p], slot[p]] == e            # the route really belongs to e
        for n in range(N):
            terms = [Fraction(float(xh[p, k])) * Fraction(float(wh[e, n, k])) for k in range(K)]
            exact = sum(terms)
            bound = Fraction(gamma) * sum(abs(t) for t in terms)
            assert abs(Fraction(float(y[p, n])) - exact) <= bound, (p, n)
    # and a neighbouring expert's weights would give a different row
    for p in range(T * 2):
        e = _expert_of_route(off, p)
        for e2 in range(E):
            if e2 != e:
                assert not np.allclose(y[p], xh[p] @ wh[e2].T)


# ------------------------------------------------- global scale rounding ----

def _rne_binary32(q: Fraction) -> float:
    """The binary32 value nearest to the positive rational q (ties to even),
    by integer arithmetic on the exact quotient."""
    assert q > 0
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1                                       # 2^e <= q < 2^(e+1)
    e = max(e, -126)                                 # subnormals share 2^-149 steps
    ulp = Fraction(2) ** (e - 23)
    m = q / ulp                                      # significand in units of ulp
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return float(lo * ulp)


def test_global_scale_is_one_rounding_of_amax_over_2688():
    """g = tensor_amax / (6 * 448) as ONE binary32 division (reading of the
    recipe "global = tensor_amax / (6 * 448)"; 2688 is exact).  The test
    searches amax values where one rounding of the exact quotient and the
    two-step (amax / 6) / 448 disagree, and checks the oracle against the
    exact quotient rounded by integer arithmetic."""
    g = inputs.rng(53)
    cands = g.uniform(1.0, 1000.0, 4000).astype(np.float32)
    found = 0
    for a in cands:
        exact = _rne_binary32(Fraction(float(a)) / 2688)
        two_step = float(np.float32(np.float32(a) / np.float32(6.0)) / np.float32(448.0))
        got = float(oracle.global_scale(np.array([[a, -a / 2]], np.float32)))
        assert got == exact, (float(a), got, exact)
        if two_step != exact:
            found += 1
    assert found >= 10          # the pin separates the two readings on these inputs
