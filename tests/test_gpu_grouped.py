"""MoE grouped GEMM (gather and weighted combine) against the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_nvfp4_gb300 import inputs, moe
from moe_grouped_gemm_nvfp4_gb300 import nvfp4 as F
from parity import bf16_to_np, check_gemm, nan_filled

pytestmark = pytest.mark.gpu


def _weights_host(g, E, N, K):
    return inputs.normal_bf16(g, (E, N, K), 0.02)


def _oracle_weights(w_bf16):
    """Per-expert quantisation in the oracle -> float64 [E, N, K]."""
    E = w_bf16.shape[0]
    out = []
    for e in range(E):
        p, s, gg = oracle.quantize(w_bf16[e].float().numpy())
        out.append(oracle.dequantize(p, s, gg))
    return np.stack(out)


def _routing(g, T, E, k, kind):
    if kind == "zipf":
        return inputs.zipf_topk(g, T, E, k, n_unused=max(1, E // 16))
    ids = inputs.uniform_topk(g, T, E, k)
    return ids


@pytest.mark.parametrize("T,E,k,N,K,kind", [
    (32, 8, 2, 256, 512, "uniform"),
    (5, 16, 2, 128, 192, "uniform"),      # most experts empty, partial K block
    (200, 4, 2, 128, 256, "uniform"),     # experts with > 128 routes (several token tiles)
    (300, 16, 4, 256, 512, "zipf"),       # skewed with empty experts
    (400, 4, 2, 256, 512, "uniform"),     # 256-row token tiles spanning two operand tiles
    (900, 3, 2, 128, 320, "uniform"),     # several 256-row tiles per expert, ragged K block
    (256, 32, 2, 1280, 256, "uniform"),   # more two-tile units than CTAs
])
def test_grouped_gather_matches_oracle(T, E, k, N, K, kind):
    g = inputs.rng(T * 13 + E + N + K)
    x = inputs.normal_bf16(g, (T, K))
    w = _weights_host(g, E, N, K)
    ids = _routing(g, T, E, k, kind)
    W = moe.quantize_experts(w.cuda())
    plan = moe.GroupedPlan(W, T, k, "gather")
    plan.out.view(torch.int16).fill_(0x7FC0)
    out = plan.run(x.cuda(), torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    off, tok, slot = oracle.route(ids, E)
    px, sx, gx = oracle.quantize(x.float().numpy())
    xh = oracle.dequantize(px, sx, gx)[tok]
    ref = oracle.grouped_gemm(xh, _oracle_weights(w), off)
    check_gemm(bf16_to_np(out[: T * k]), ref, "grouped gather")


@pytest.mark.parametrize("T,E,k,N,K", [(32, 8, 2, 256, 512), (64, 16, 8, 384, 256),
                                       (3, 8, 2, 128, 128), (400, 4, 2, 128, 256),
                                       (256, 32, 2, 1280, 256)])   # units > CTAs
def test_grouped_combine_matches_oracle(T, E, k, N, K):
    g = inputs.rng(T * 17 + E + N + K)
    ids = inputs.uniform_topk(g, T, E, k)
    wts = inputs.dirichlet_weights(g, T, k)
    R = T * k
    h = inputs.normal_bf16(g, (R, K))          # route-ordered intermediate
    w = _weights_host(g, E, N, K)
    W = moe.quantize_experts(w.cuda())
    plan = moe.GroupedPlan(W, T, k, "combine")
    off, tok, slot = oracle.route(ids, E)
    ph, sh, gh = oracle.quantize(h.float().numpy())
    y = oracle.grouped_gemm(oracle.dequantize(ph, sh, gh), _oracle_weights(w), off)
    ref = oracle.combine(y, tok, slot, wts, T)
    # twice on one workspace: each call must leave it cleared for the next
    for call in range(2):
        plan.out.view(torch.int16).fill_(0x7FC0)
        out = plan.run(h.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(wts).cuda())
        torch.cuda.synchronize()
        assert F.nvfp4_device_status() == F.NVFP4_OK
        check_gemm(bf16_to_np(out[:T]), ref, f"grouped combine, call {call}")


def test_grouped_rejects_non_monotone_offsets_on_device():
    E, N, K, T, k = 4, 128, 128, 4, 1
    g = inputs.rng(1)
    W = moe.quantize_experts(_weights_host(g, E, N, K).cuda())
    plan = moe.GroupedPlan(W, T, k, "gather")
    x = inputs.normal_bf16(g, (T, K)).cuda()
    plan.route(torch.zeros((T, k), dtype=torch.int32, device="cuda"))
    plan.quantize(x)
    torch.cuda.synchronize()
    F.nvfp4_device_status(reset=True)
    plan.expert_offsets.copy_(torch.tensor([0, 3, 1, 4, 4], dtype=torch.int32))
    plan.gemm()
    assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_DEVICE_CHECK


def _hot_expert_routing(g, T, E):
    """Slot 0 of every token goes to expert 0, slot 1 uniformly to 1..E-1: one
    expert with T routes among experts with few, so narrow token tiles of the
    hot expert start at rows 0, 32, 64 and 96 of their operand tiles."""
    ids = np.empty((T, 2), np.int32)
    ids[:, 0] = 0
    ids[:, 1] = g.integers(1, E, T)
    return ids


@pytest.mark.parametrize("T,E,N,K", [(100, 16, 256, 512), (150, 16, 128, 256),
                                     (150, 8, 128, 256)])     # 32-, 32- and 64-row tiles
def test_grouped_narrow_tiles_hot_expert(T, E, N, K):
    g = inputs.rng(T + 5 * E)
    x = inputs.normal_bf16(g, (T, K))
    w = _weights_host(g, E, N, K)
    ids = _hot_expert_routing(g, T, E)
    W = moe.quantize_experts(w.cuda())
    plan = moe.GroupedPlan(W, T, 2, "gather")
    plan.out.view(torch.int16).fill_(0x7FC0)
    out = plan.run(x.cuda(), torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    off, tok, slot = oracle.route(ids, E)
    px, sx, gx = oracle.quantize(x.float().numpy())
    ref = oracle.grouped_gemm(oracle.dequantize(px, sx, gx)[tok], _oracle_weights(w), off)
    check_gemm(bf16_to_np(out[: 2 * T]), ref, "hot expert gather")
    # the same routing through the weighted combine
    wts = inputs.dirichlet_weights(g, T, 2)
    h = inputs.normal_bf16(g, (2 * T, K))
    plan2 = moe.GroupedPlan(W, T, 2, "combine", routing_from=plan)
    out2 = plan2.run(h.cuda(), None, torch.from_numpy(wts).cuda(), route=False)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    ph, sh, gh = oracle.quantize(h.float().numpy())
    y = oracle.grouped_gemm(oracle.dequantize(ph, sh, gh), _oracle_weights(w), off)
    check_gemm(bf16_to_np(out2[:T]), oracle.combine(y, tok, slot, wts, T), "hot expert combine")


def test_bounded_wait_expires_reports_timeout_and_context_survives():
    """Failure path: a stage that never fills (test hook) makes the MMA wait run
    out; the kernel records NVFP4_ERR_TIMEOUT and returns, and the next call on
    the same context computes the right result."""
    T, E, k, N, K = 16, 4, 2, 128, 256
    g = inputs.rng(9)
    x = inputs.normal_bf16(g, (T, K)).cuda()
    w = _weights_host(g, E, N, K)
    ids = torch.from_numpy(inputs.uniform_topk(g, T, E, k)).cuda()
    W = moe.quantize_experts(w.cuda())
    plan = moe.GroupedPlan(W, T, k, "gather")
    plan.route(ids)
    plan.quantize(x)
    torch.cuda.synchronize()
    F.nvfp4_device_status(reset=True)
    F.nvfp4_set_timeout_ns(20_000_000)                 # 20 ms
    F.nvfp4_debug_set_flags(1)
    try:
        plan.gemm()
        assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_TIMEOUT
    finally:
        F.nvfp4_debug_set_flags(0)
        F.nvfp4_set_timeout_ns(1_000_000_000)
    plan.out.view(torch.int16).fill_(0x7FC0)
    plan.gemm()
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    off, tok, _ = oracle.route(ids.cpu().numpy(), E)
    px, sx, gx = oracle.quantize(x.float().cpu().numpy())
    ref = oracle.grouped_gemm(oracle.dequantize(px, sx, gx)[tok], _oracle_weights(w), off)
    check_gemm(bf16_to_np(plan.out[: T * k]), ref, "after timeout")


def test_layer_step_overlapping_route_and_amax_matches_sequential_calls():
    """DecodeLayer.step runs the amax of x on a side stream beside the routing
    (NVFP4_AMAX_DONE for the dispatch); eagerly and replayed from a CUDA graph
    it must give the bytes the plain sequence route -> quantize -> GEMM gives."""
    T, E, k, K1, N1, K2, N2 = 48, 8, 2, 256, 256, 128, 256
    g = inputs.rng(4242)
    x = inputs.normal_bf16(g, (T, K1)).cuda()
    h = inputs.normal_bf16(g, (T * k, K2)).cuda()
    ids = torch.from_numpy(inputs.uniform_topk(g, T, E, k)).cuda()
    wts = torch.from_numpy(inputs.dirichlet_weights(g, T, k)).cuda()
    W1 = moe.quantize_experts(_weights_host(g, E, N1, K1).cuda())
    W2 = moe.quantize_experts(_weights_host(g, E, N2, K2).cuda())
    ref = moe.GroupedPlan(W1, T, k, "gather")
    ref_out = ref.run(x, ids).clone()
    ref_dn = moe.GroupedPlan(W2, T, k, "combine", routing_from=ref)
    ref_dn_out = ref_dn.run(h, None, wts, route=False).clone()
    layer = moe.DecodeLayer(W1, W2, T, k)
    gu_out, dn_out = layer.step(x, ids, h, wts)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    assert torch.equal(layer.gate_up.a_g, ref.a_g)
    assert torch.equal(gu_out[:T * k], ref_out[:T * k])
    assert torch.equal(dn_out[:T].float(), ref_dn_out[:T].float()) or \
        torch.allclose(dn_out[:T].float(), ref_dn_out[:T].float(), rtol=1e-2, atol=1e-3)
    cap = moe.CapturedStep(layer, x, ids, h, wts)
    gu_out.zero_()
    cap.replay()
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    assert torch.equal(gu_out[:T * k], ref_out[:T * k])
