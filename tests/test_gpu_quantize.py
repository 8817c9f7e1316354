"""Quantiser, prepack, routing and dispatch: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_nvfp4_gb300 import inputs
from moe_grouped_gemm_nvfp4_gb300 import nvfp4 as F

pytestmark = pytest.mark.gpu


def _special_matrix(g, rows, cols):
    """N(0,1) plus blocks that hit every E2M1 midpoint, zeros, -0, tiny and huge values."""
    x = g.standard_normal((rows, cols)).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75,
                     -2.5, -3.5, -5.0, -6.0], np.float32)
    if rows >= 4 and cols >= 64:
        x[0, :16] = mids                        # block amax 6 -> d = g * e4m3(s)
        x[1, :16] = 0.0
        x[1, 16:32] = -0.0
        x[2, :16] = mids * np.float32(1e-6)     # subnormal E4M3 scale range
        x[3, 32:48] = mids * np.float32(37.0)
    return inputs.to_bf16(x)


def _cases():
    return [(1, 16), (3, 48), (5, 64), (37, 512), (130, 320), (256, 6144)]


@pytest.mark.parametrize("rows,cols", _cases())
def test_quantize_rowmajor_bit_exact(rows, cols):
    g = inputs.rng(rows * 1000 + cols)
    x = _special_matrix(g, rows, cols)
    packed, scales, gd = F.quantize(x.cuda())
    p_ref, s_ref, g_ref = oracle.quantize(x.float().numpy())
    assert np.float32(gd.item()) == g_ref
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(packed.cpu().numpy(), p_ref)


@pytest.mark.parametrize("rows,cols", [(5, 64), (130, 320), (300, 512)])
def test_quantize_atom_layout_bit_exact(rows, cols):
    g = inputs.rng(7 + rows)
    x = _special_matrix(g, rows, cols)
    packed, scales, gd = F.quantize(x.cuda(), atoms=True)
    p_ref, s_ref, _ = oracle.quantize(x.float().numpy())
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    ref = oracle.prepack_scales(s_ref)
    got = scales.cpu().numpy()
    # padding rows are not written by the quantiser; compare the defined bytes
    mask = oracle.prepack_scales(np.ones_like(s_ref)) == 1
    assert got.size == ref.size
    assert np.array_equal(got[mask], ref[mask])


@pytest.mark.parametrize("dstep,amax,scode", [(1.0, 6.0, 0x78), (1.5, 9.0, 0x7C)])
def test_quantize_e2m1_rounding_at_exact_ties(dstep, amax, scode):
    """With g = 2^-8 and a block maximum `amax`, s = amax / 6 / g is an exact
    E4M3 value and d = dstep, so x = midpoint * dstep makes x / d an exact E2M1
    tie (ties go to the even code); the BF16 neighbours of those x fall just
    either side.  Both signs.  (d = 1.5 puts the quotients at the ties without
    d being a power of two, where a shortcut through 1/d must defer to the
    exact division.)"""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32) * np.float32(dstep)
    bits = inputs.to_bf16(mids).view(torch.int16).numpy().astype(np.int32)
    vals = []
    for b in bits:                                   # the tie and its two BF16 neighbours
        for db in (-1, 0, 1):
            vals.append(np.array([b + db], np.int32).astype(np.int16).view(np.uint16)[0])
    v = torch.from_numpy(np.array(vals, np.uint16).view(np.int16)).view(torch.bfloat16).float()
    v = v.numpy()
    tail = np.array([0.0, -0.0, amax, -amax, 1e-3, -1e-3, 0.1, -0.1], np.float32)
    pool = np.concatenate([v, -v, tail])             # 50 values
    rows = []
    for i in range(0, len(pool), 15):                # 15 values + the block maximum
        blk = np.full(16, 0.0, np.float32)
        chunk = pool[i:i + 15]
        blk[:len(chunk)] = chunk
        blk[15] = amax
        rows.append(blk)
    x = inputs.to_bf16(np.concatenate(rows).reshape(1, -1))
    gg = torch.tensor([2.0 ** -8], dtype=torch.float32, device="cuda")
    packed, scales, _ = F.quantize(x.cuda(), global_scale=gg)
    p_ref, s_ref, _ = oracle.quantize(x.float().numpy(), g=np.float32(2.0 ** -8))
    assert (s_ref == scode).all()                    # d = dstep in every block
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(packed.cpu().numpy(), p_ref)


@pytest.mark.parametrize("gval", [2.0 ** -8, 0.0123, 3.0e-38, 1.0e-39, 5.0e35])
def test_quantize_block_scales_at_e4m3_midpoints(gval):
    """Block maxima b = 3 (2j + 1) 2^k make s = (b / 6) / g an exact midpoint
    between two E4M3 values when g is a power of two (ties go to the even
    code); their BF16 neighbours fall just either side.  Other globals put s
    anywhere, including a global so small (or subnormal, or huge) that every
    block takes the exact division chain."""
    vals = []
    for j in range(8, 16):
        for k in range(-12, 4):
            b = np.float32(3 * (2 * j + 1) * 2.0 ** k)
            bits = inputs.to_bf16(np.array([b], np.float32)).view(torch.int16).numpy()[0]
            for db in (-2, -1, 0, 1, 2):
                vals.append(np.array([bits + db], np.int32).astype(np.int16)[0])
    amaxes = torch.from_numpy(np.array(vals, np.int16)).view(torch.bfloat16).float().numpy()
    g = inputs.rng(1234)
    x = g.standard_normal((len(amaxes), 16)).astype(np.float32) * 0.3 * amaxes[:, None]
    x[:, 5] = amaxes                                 # the block maximum
    x[::2, 5] *= -1.0                                # half of them negative
    xb = inputs.to_bf16(x.reshape(-1, 64)) if x.size % 64 == 0 else inputs.to_bf16(x)
    gg = torch.tensor([gval], dtype=torch.float32, device="cuda")
    packed, scales, _ = F.quantize(xb.cuda(), global_scale=gg)
    p_ref, s_ref, _ = oracle.quantize(xb.float().numpy(), g=np.float32(gval))
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(packed.cpu().numpy(), p_ref)


def test_quantize_strided_rows_and_given_global():
    g = inputs.rng(99)
    base = inputs.normal_bf16(g, (20, 200)).cuda()
    x = base[:, 8:136]                             # ld = 200, cols = 128
    gg = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    packed, scales, _ = F.quantize(x, global_scale=gg)
    p_ref, s_ref, _ = oracle.quantize(x.float().cpu().numpy(), g=np.float32(0.01))
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(packed.cpu().numpy(), p_ref)


def test_quantize_zero_tensor():
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    packed, scales, gd = F.quantize(x)
    assert gd.item() == 0.0
    assert int(scales.abs().sum()) == 0 and int(packed.sum()) == 0


def test_quantize_empty_is_ok():
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    packed, scales, gd = F.quantize(x)
    assert gd.item() == 0.0


def test_prepack_matches_oracle():
    g = inputs.rng(5)
    for rows, kblk in [(1, 4), (128, 8), (300, 12), (4096, 384)]:
        s = g.integers(0, 256, (rows, kblk)).astype(np.uint8)
        out = torch.full((F.nvfp4_atom_scales_bytes(rows, kblk * 16),), 0xAB, dtype=torch.uint8,
                         device="cuda")
        F.nvfp4_prepack_weights(torch.from_numpy(s).cuda(), out)
        assert np.array_equal(out.cpu().numpy(), oracle.prepack_scales(s))


@pytest.mark.parametrize("T,E,k,kind", [(1, 4, 2, "uniform"), (37, 9, 3, "uniform"),
                                        (256, 128, 8, "uniform"), (8192, 128, 8, "zipf")])
def test_route_matches_oracle(T, E, k, kind):
    g = inputs.rng(T + E)
    ids = inputs.uniform_topk(g, T, E, k) if kind == "uniform" else inputs.zipf_topk(g, T, E, k)
    off, tok, slot, pos = F.moe_route(torch.from_numpy(ids).cuda(), E)
    o_ref, t_ref, s_ref = oracle.route(ids, E)
    assert np.array_equal(off.cpu().numpy(), o_ref)
    assert np.array_equal(tok.cpu().numpy(), t_ref)
    assert np.array_equal(slot.cpu().numpy(), s_ref)
    inv = np.empty(T * k, np.int64)
    inv[t_ref.astype(np.int64) * k + s_ref] = np.arange(T * k)
    assert np.array_equal(pos.cpu().numpy(), inv)
    assert F.nvfp4_device_status() == F.NVFP4_OK


def test_route_rejects_bad_ids_on_device():
    ids = torch.tensor([[0, 1], [5, 2]], dtype=torch.int32, device="cuda")
    F.nvfp4_device_status(reset=True)
    off, tok, slot, pos = F.moe_route(ids, 4)
    assert F.nvfp4_last_device_status() == F.NVFP4_ERR_DEVICE_CHECK   # read, not cleared
    assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_DEVICE_CHECK
    assert F.nvfp4_last_device_status() == F.NVFP4_OK
    assert off[-1].item() == 3


def _valid_tile_mask(n_rows_routes, K, off, chunk):
    """Bytes of the grouped tile layout that hold a route's codes or scales."""
    ones_p = np.full((n_rows_routes, K // 2), 1, np.uint8)
    ones_s = np.full((n_rows_routes, K // 16), 1, np.uint8)
    return oracle.grouped_operand_tiles(ones_p, ones_s, off, chunk) == 1


@pytest.mark.parametrize("T,E,k,K", [(13, 6, 2, 128), (256, 128, 8, 6144), (300, 4, 2, 320),
                                     (100, 16, 2, 256)])
def test_dispatch_gather_bit_exact(T, E, k, K):
    g = inputs.rng(T * 7 + K)
    x = inputs.normal_bf16(g, (T, K))
    ids = inputs.uniform_topk(g, T, E, k)
    ids_d = torch.from_numpy(ids).cuda()
    off, tok, slot, pos = F.moe_route(ids_d, E)
    R = T * k
    tiles = torch.zeros(F.nvfp4_grouped_tiles_bytes(R, E, K), dtype=torch.uint8, device="cuda")
    gd = torch.empty(1, dtype=torch.float32, device="cuda")
    F.nvfp4_quantize_dispatch(x.cuda(), pos, k, off, E, R, tiles, gd)
    p_ref, s_ref, g_ref = oracle.quantize(x.float().numpy())
    o_ref, t_ref, _ = oracle.route(ids, E)
    assert np.float32(gd.item()) == g_ref
    chunk = F.nvfp4_grouped_chunk_rows(R, E)
    lay = oracle.grouped_operand_tiles(p_ref[t_ref], s_ref[t_ref], o_ref, chunk)
    mask = _valid_tile_mask(R, K, o_ref, chunk)
    got = tiles.cpu().numpy()[: lay.size]
    assert np.array_equal(got[mask], lay[mask])


def test_dispatch_route_order_input_bit_exact():
    g = inputs.rng(3)
    T, E, k, K = 64, 16, 4, 256
    ids = inputs.uniform_topk(g, T, E, k)
    off, tok, slot, pos = F.moe_route(torch.from_numpy(ids).cuda(), E)
    R = T * k
    h = inputs.normal_bf16(g, (R, K))
    tiles = torch.zeros(F.nvfp4_grouped_tiles_bytes(R, E, K), dtype=torch.uint8, device="cuda")
    gd = torch.empty(1, dtype=torch.float32, device="cuda")
    F.nvfp4_quantize_dispatch(h.cuda(), None, 1, off, E, R, tiles, gd)
    p_ref, s_ref, g_ref = oracle.quantize(h.float().numpy())
    o_ref, _, _ = oracle.route(ids, E)
    chunk = F.nvfp4_grouped_chunk_rows(R, E)
    lay = oracle.grouped_operand_tiles(p_ref, s_ref, o_ref, chunk)
    mask = _valid_tile_mask(R, K, o_ref, chunk)
    assert np.array_equal(tiles.cpu().numpy()[: lay.size][mask], lay[mask])


@pytest.mark.parametrize("rows,K", [(128, 256), (300, 512), (256, 320)])
def test_prepack_weight_tiles_matches_oracle(rows, K):
    g = inputs.rng(rows + K)
    packed = g.integers(0, 256, (rows, K // 2)).astype(np.uint8)
    sf = g.integers(0, 256, (rows, K // 16)).astype(np.uint8)
    out = torch.full((F.nvfp4_operand_tiles_bytes(rows, K),), 0xCD, dtype=torch.uint8,
                     device="cuda")
    F.nvfp4_prepack_weight_tiles(torch.from_numpy(packed).cuda(), torch.from_numpy(sf).cuda(), out)
    assert np.array_equal(out.cpu().numpy(), oracle.operand_tiles(packed, sf))
