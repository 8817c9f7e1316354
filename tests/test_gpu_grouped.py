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
    (160, 8, 2, 256, 256, "uniform"),     # 64-row tiles, two weight tiles per unit
    (900, 3, 2, 256, 320, "uniform"),     # 256-row tiles on CTA pairs, ragged K block
    (2000, 16, 2, 512, 256, "zipf"),      # CTA pairs, skewed: hot experts, empty ones, odd tiles
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
                                       (256, 32, 2, 1280, 256),    # units > CTAs
                                       (64, 16, 8, 512, 320)])     # 64-row tiles, weight-tile pairs
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


@pytest.mark.parametrize("T,E,k,N,K", [(16, 4, 2, 128, 256),      # one-SM kernel
                                       (400, 4, 2, 256, 256)])    # 256-route tiles: CTA pairs
def test_bounded_wait_expires_reports_timeout_and_context_survives(T, E, k, N, K):
    """Failure path: a stage that never fills (test hook) makes the MMA wait run
    out; the kernel records NVFP4_ERR_TIMEOUT and returns, and the next call on
    the same context computes the right result."""
    assert F.nvfp4_grouped_chunk_rows(T * k, E) in (32, 128)
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


def test_layer_step_overlapping_route_and_amax_matches_oracle_eager_and_replayed():
    """DecodeLayer.step runs the amax of x on a side stream beside the routing
    (NVFP4_AMAX_DONE for the dispatch).  Eagerly and replayed from a CUDA
    graph, both of its outputs (gate_up in route order, down with the
    weighted combine) must match the FP64 oracle, and gate_up must be the
    bytes the plain sequence route -> quantize -> GEMM gives."""
    T, E, k, K1, N1, K2, N2 = 48, 8, 2, 256, 256, 128, 256
    g = inputs.rng(4242)
    x_h = inputs.normal_bf16(g, (T, K1))
    h_h = inputs.normal_bf16(g, (T * k, K2))
    ids_h = inputs.uniform_topk(g, T, E, k)
    wts_h = inputs.dirichlet_weights(g, T, k)
    w1 = _weights_host(g, E, N1, K1)
    w2 = _weights_host(g, E, N2, K2)
    x, h = x_h.cuda(), h_h.cuda()
    ids, wts = torch.from_numpy(ids_h).cuda(), torch.from_numpy(wts_h).cuda()
    W1 = moe.quantize_experts(w1.cuda())
    W2 = moe.quantize_experts(w2.cuda())
    # oracle: gate_up in route order; down over the route-ordered h, combined
    off, tok, slot = oracle.route(ids_h, E)
    px, sx, gx = oracle.quantize(x_h.float().numpy())
    ref_gu = oracle.grouped_gemm(oracle.dequantize(px, sx, gx)[tok], _oracle_weights(w1), off)
    ph, sh, gh = oracle.quantize(h_h.float().numpy())
    ref_dn = oracle.combine(oracle.grouped_gemm(oracle.dequantize(ph, sh, gh),
                                                _oracle_weights(w2), off), tok, slot, wts_h, T)
    seq = moe.GroupedPlan(W1, T, k, "gather")
    seq_out = seq.run(x, ids).clone()
    layer = moe.DecodeLayer(W1, W2, T, k)
    gu_out, dn_out = layer.step(x, ids, h, wts)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    assert torch.equal(layer.gate_up.a_g, seq.a_g)
    assert torch.equal(gu_out[:T * k], seq_out[:T * k])
    check_gemm(bf16_to_np(gu_out[:T * k]), ref_gu, "eager gate_up")
    check_gemm(bf16_to_np(dn_out[:T]), ref_dn, "eager down + combine")
    cap = moe.CapturedStep(layer, x, ids, h, wts)
    for _ in range(2):                           # two replays, outputs poisoned before each
        gu_out.view(torch.int16).fill_(0x7FC0)
        dn_out.view(torch.int16).fill_(0x7FC0)
        cap.replay()
        torch.cuda.synchronize()
        assert F.nvfp4_device_status() == F.NVFP4_OK
        assert torch.equal(gu_out[:T * k], seq_out[:T * k])
        check_gemm(bf16_to_np(gu_out[:T * k]), ref_gu, "replayed gate_up")
        check_gemm(bf16_to_np(dn_out[:T]), ref_dn, "replayed down + combine")


def test_combine_rejects_a_token_outside_the_batch():
    """A route whose token is T (one past the batch) is a device-side input
    error: the kernel records NVFP4_ERR_DEVICE_CHECK, adds nothing for that
    route and writes no FP32 row past T (the workspace handed in is twice as
    large, its upper half a sentinel); every other route is combined."""
    T, E, k, N, K = 16, 4, 2, 128, 256
    g = inputs.rng(77)
    ids_h = inputs.uniform_topk(g, T, E, k)
    wts_h = inputs.dirichlet_weights(g, T, k)
    h_h = inputs.normal_bf16(g, (T * k, K))
    w = _weights_host(g, E, N, K)
    W = moe.quantize_experts(w.cuda())
    plan = moe.GroupedPlan(W, T, k, "combine")
    plan.route(torch.from_numpy(ids_h).cuda())
    plan.quantize(h_h.cuda())
    torch.cuda.synchronize()
    off, tok, slot = oracle.route(ids_h, E)
    bad = 5                                      # route position whose token goes bad
    t_bad, s_bad = int(tok[bad]), int(slot[bad])
    plan.route_token[bad] = T
    ws = torch.full((2 * T, N), 7.0, dtype=torch.float32, device="cuda")
    out = nan_filled((T, N))
    F.nvfp4_device_status(reset=True)
    F.nvfp4_grouped_gemm_tiles(plan.a_tiles, plan.a_g, W.tiles, W.g, plan.expert_offsets, E, T, k, N,
                         K, plan.route_token, plan.route_slot,
                         torch.from_numpy(wts_h).cuda(), out, ws)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_DEVICE_CHECK
    assert torch.all(ws[T:] == 7.0)
    ph, sh, gh = oracle.quantize(h_h.float().numpy())
    y = oracle.grouped_gemm(oracle.dequantize(ph, sh, gh), _oracle_weights(w), off)
    wts_ref = wts_h.astype(np.float64).copy()
    wts_ref[t_bad, s_bad] = 0.0                  # the rejected route adds nothing
    check_gemm(bf16_to_np(out), oracle.combine(y, tok, slot, wts_ref, T), "bad token dropped")
