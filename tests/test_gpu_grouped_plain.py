"""The grouped GEMM on plain NVFP4 operands (nvfp4_grouped_gemm: packed
activation rows + row-major scales, gathered by route_token inside the call;
packed expert weights + atom-layout scales) against the FP64 oracle, called
through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_nvfp4_gb300 import inputs, moe
from moe_grouped_gemm_nvfp4_gb300 import nvfp4 as F
from parity import bf16_to_np, check_gemm, nan_filled

pytestmark = pytest.mark.gpu


def _oracle_weights(w_bf16):
    return np.stack([oracle.dequantize(*oracle.quantize(w_bf16[e].float().numpy()))
                     for e in range(w_bf16.shape[0])])


def _problem(seed, T, E, k, N, K, rows_of):
    g = inputs.rng(seed)
    ids = inputs.uniform_topk(g, T, E, k)
    wts = inputs.dirichlet_weights(g, T, k)
    x = inputs.normal_bf16(g, (rows_of(T * k, T), K))
    w = inputs.normal_bf16(g, (E, N, K), 0.05)
    return ids, wts, x, w


@pytest.mark.parametrize("T,E,k,N,K", [
    (32, 8, 2, 256, 512),        # 8 routes per expert: 32-route tiles, two weight tiles per unit
    (5, 16, 2, 128, 192),        # most experts empty, partial K block
    (500, 4, 2, 128, 320),       # ~250 routes per expert: 256-route tiles, ragged K block
    (128, 16, 4, 384, 256),      # 32 routes per expert: 64-route tiles
])
def test_plain_gather_matches_oracle(T, E, k, N, K):
    ids, _, x, w = _problem(T * 7 + E + N + K, T, E, k, N, K, lambda R, T: T)
    px, sx, gx = F.quantize(x.cuda())                      # row-major scales
    Wp = moe.quantize_experts_plain(w.cuda())
    off, tok, slot, pos = F.moe_route(torch.from_numpy(ids).cuda(), E)
    R = T * k
    ws = torch.empty(F.nvfp4_grouped_gemm_workspace_bytes(T, k, E, N, K, False),
                     dtype=torch.uint8, device="cuda")
    out = nan_filled((R, N))
    F.nvfp4_grouped_gemm(px, sx, gx, Wp.packed, Wp.sf_atoms, Wp.g, off, E, tok, None, slot,
                         T, k, N, K, out, ws)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    o_off, o_tok, _ = oracle.route(ids, E)
    opx, osx, ogx = oracle.quantize(x.float().numpy())
    ref = oracle.grouped_gemm(oracle.dequantize(opx, osx, ogx)[o_tok], _oracle_weights(w), o_off)
    check_gemm(bf16_to_np(out), ref, "plain gather")
    # the rows the call gathered into the workspace are the token rows, byte for byte
    chunk = F.nvfp4_grouped_chunk_rows(R, E)
    gp, gs = oracle.grouped_operand_rows(ws.cpu().numpy(), o_off, K, chunk)
    assert np.array_equal(gp, px.cpu().numpy()[o_tok])
    assert np.array_equal(gs, sx.cpu().numpy()[o_tok])


def test_plain_route_order_without_gather_matches_oracle():
    T, E, k, N, K = 24, 8, 2, 256, 256
    ids, _, x, w = _problem(501, T, E, k, N, K, lambda R, T: R)     # x already in route order
    px, sx, gx = F.quantize(x.cuda())
    Wp = moe.quantize_experts_plain(w.cuda())
    off, tok, slot, pos = F.moe_route(torch.from_numpy(ids).cuda(), E)
    ws = torch.empty(F.nvfp4_grouped_gemm_workspace_bytes(T, k, E, N, K, False),
                     dtype=torch.uint8, device="cuda")
    out = nan_filled((T * k, N))
    F.nvfp4_grouped_gemm(px, sx, gx, Wp.packed, Wp.sf_atoms, Wp.g, off, E, None, None, None,
                         T, k, N, K, out, ws)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    o_off, _, _ = oracle.route(ids, E)
    opx, osx, ogx = oracle.quantize(x.float().numpy())
    ref = oracle.grouped_gemm(oracle.dequantize(opx, osx, ogx), _oracle_weights(w), o_off)
    check_gemm(bf16_to_np(out), ref, "plain, route order")


@pytest.mark.parametrize("T,E,k,N,K", [(32, 8, 2, 256, 512), (64, 16, 8, 384, 256),
                                       (400, 4, 2, 128, 256)])
def test_plain_combine_matches_oracle(T, E, k, N, K):
    ids, wts, h, w = _problem(T * 11 + E + N + K, T, E, k, N, K, lambda R, T: R)
    ph, sh, gh = F.quantize(h.cuda())
    Wp = moe.quantize_experts_plain(w.cuda())
    off, tok, slot, pos = F.moe_route(torch.from_numpy(ids).cuda(), E)
    ws = torch.empty(F.nvfp4_grouped_gemm_workspace_bytes(T, k, E, N, K, True),
                     dtype=torch.uint8, device="cuda")
    o_off, o_tok, o_slot = oracle.route(ids, E)
    oph, osh, ogh = oracle.quantize(h.float().numpy())
    y = oracle.grouped_gemm(oracle.dequantize(oph, osh, ogh), _oracle_weights(w), o_off)
    ref = oracle.combine(y, o_tok, o_slot, wts, T)
    for call in range(2):                         # the workspace's sums start from zero each call
        out = nan_filled((T, N))
        F.nvfp4_grouped_gemm(ph, sh, gh, Wp.packed, Wp.sf_atoms, Wp.g, off, E, tok,
                             torch.from_numpy(wts).cuda(), slot, T, k, N, K, out, ws)
        torch.cuda.synchronize()
        assert F.nvfp4_device_status() == F.NVFP4_OK
        check_gemm(bf16_to_np(out), ref, f"plain combine, call {call}")


def test_plain_equals_the_tile_entry_point_bit_for_bit():
    """Both forms run the same kernel on the same quantised values, so the
    outputs are identical: operand tiles prepacked offline against weights read
    as row-major codes through the tensor map plus atom-layout scales."""
    T, E, k, N, K = 64, 16, 2, 256, 512
    ids, _, x, w = _problem(777, T, E, k, N, K, lambda R, T: T)
    xd, wd = x.cuda(), w.cuda()
    ids_d = torch.from_numpy(ids).cuda()
    W = moe.quantize_experts(wd)
    Wp = moe.quantize_experts_plain(wd)
    plan = moe.GroupedPlan(W, T, k, "gather")
    ref = plan.run(xd, ids_d).clone()
    px, sx, gx = F.quantize(xd)
    ws = torch.empty(F.nvfp4_grouped_gemm_workspace_bytes(T, k, E, N, K, False),
                     dtype=torch.uint8, device="cuda")
    out = nan_filled((T * k, N))
    F.nvfp4_grouped_gemm(px, sx, gx, Wp.packed, Wp.sf_atoms, Wp.g, plan.expert_offsets, E,
                         plan.route_token, None, plan.route_slot, T, k, N, K, out, ws)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    assert torch.equal(out.view(torch.int16), ref[:T * k].view(torch.int16))


def test_plain_gather_rejects_a_row_outside_a():
    """A gathered token row outside [0, T) is a device-side input error: the
    copy of that route is skipped and the status word says so."""
    T, E, k, N, K = 16, 4, 2, 128, 256
    ids, _, x, w = _problem(888, T, E, k, N, K, lambda R, T: T)
    px, sx, gx = F.quantize(x.cuda())
    Wp = moe.quantize_experts_plain(w.cuda())
    off, tok, slot, pos = F.moe_route(torch.from_numpy(ids).cuda(), E)
    tok[0] = T
    ws = torch.empty(F.nvfp4_grouped_gemm_workspace_bytes(T, k, E, N, K, False),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((T * k, N), dtype=torch.bfloat16, device="cuda")
    F.nvfp4_device_status(reset=True)
    F.nvfp4_grouped_gemm(px, sx, gx, Wp.packed, Wp.sf_atoms, Wp.g, off, E, tok, None, slot,
                         T, k, N, K, out, ws)
    assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_DEVICE_CHECK
