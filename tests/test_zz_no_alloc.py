"""The allocation-free combine entry point gives the same result as the
workspace-taking one, call after call.

Some callers cannot allocate device memory when they call a kernel (plugin
interfaces that pass only inputs and outputs, serving loops that forbid the
CUDA allocator after start-up); nvfp4_grouped_gemm_combine_noalloc serves
them from a fixed workspace inside the library.  This file is collected last
so that a run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

from moe_grouped_gemm_nvfp4_gb300 import inputs, moe
from moe_grouped_gemm_nvfp4_gb300 import nvfp4 as F
from parity import bf16_to_np, check_gemm

pytestmark = pytest.mark.gpu


def test_noalloc_combine_matches_workspace_entry_point_twice():
    T, E, k, N, K = 48, 8, 2, 256, 512
    g = inputs.rng(2024)
    ids = inputs.uniform_topk(g, T, E, k)
    wts = torch.from_numpy(inputs.dirichlet_weights(g, T, k)).cuda()
    h = inputs.normal_bf16(g, (T * k, K)).cuda()
    W = moe.quantize_experts(inputs.normal_bf16(g, (E, N, K), 0.02).cuda())
    plan = moe.GroupedPlan(W, T, k, "combine")
    ref = plan.run(h, torch.from_numpy(ids).cuda(), wts).clone()
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    ref_np = bf16_to_np(ref[:T])
    for call in range(2):            # the second call must not see the first call's sums
        out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        out.view(torch.int16).fill_(0x7FC0)
        F.nvfp4_grouped_gemm_combine_noalloc(plan.a_tiles, plan.a_g, W.tiles, W.g,
                                             plan.expert_offsets, E, T, k, N, K,
                                             plan.route_token, plan.route_slot, wts, out)
        torch.cuda.synchronize()
        assert F.nvfp4_device_status() == F.NVFP4_OK
        check_gemm(bf16_to_np(out), ref_np, f"no-alloc call {call}")


def test_noalloc_rejects_shapes_beyond_its_workspace():
    cap = F.nvfp4_noalloc_workspace_floats()
    assert cap == 4 * 1024 * 1024
    z = torch.zeros(64, dtype=torch.uint8, device="cuda")
    gf = torch.ones(1, dtype=torch.float32, device="cuda")
    i32 = torch.zeros(4, dtype=torch.int32, device="cuda")
    N = 6144
    T = cap // N + 1                        # one token row too many
    with pytest.raises(F.NVFP4Error) as ei:
        F.nvfp4_grouped_gemm_combine_noalloc(z, gf, z, gf, i32, 2, T, 1, N, 128, i32, i32, gf, z)
    assert ei.value.status == F.NVFP4_ERR_UNSUPPORTED


def _combine_problem(seed, T=32, E=4, k=2, N=128, K=256):
    g = inputs.rng(seed)
    ids = torch.from_numpy(inputs.uniform_topk(g, T, E, k)).cuda()
    wts = torch.from_numpy(inputs.dirichlet_weights(g, T, k)).cuda()
    h = inputs.normal_bf16(g, (T * k, K)).cuda()
    W = moe.quantize_experts(inputs.normal_bf16(g, (E, N, K), 0.02).cuda())
    plan = moe.GroupedPlan(W, T, k, "combine")
    ref = plan.run(h, ids, wts).clone()
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    return plan, W, wts, ref, (T, E, k, N, K)


def _noalloc(plan, W, wts, out, shape):
    T, E, k, N, K = shape
    F.nvfp4_grouped_gemm_combine_noalloc(plan.a_tiles, plan.a_g, W.tiles, W.g,
                                         plan.expert_offsets, E, T, k, N, K,
                                         plan.route_token, plan.route_slot, wts, out)


def test_noalloc_rejects_a_token_outside_the_batch():
    """A route whose token is T is refused by the device-side check (status
    NVFP4_ERR_DEVICE_CHECK) and adds nothing, so it cannot write past the T
    rows of the library's workspace that the call uses (T * N is far below
    the workspace size, so even an unchecked write would stay inside it).
    The next, valid call gives the workspace entry point's result."""
    plan, W, wts, ref, shape = _combine_problem(91)
    T = shape[0]
    saved = plan.route_token.clone()
    plan.route_token[3] = T
    out = torch.empty((T, shape[3]), dtype=torch.bfloat16, device="cuda")
    F.nvfp4_device_status(reset=True)
    _noalloc(plan, W, wts, out, shape)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_DEVICE_CHECK
    plan.route_token.copy_(saved)
    out.view(torch.int16).fill_(0x7FC0)
    _noalloc(plan, W, wts, out, shape)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    check_gemm(bf16_to_np(out), bf16_to_np(ref[:T]), "no-alloc after a bad token")


def test_noalloc_bounded_wait_expires_then_next_call_is_right():
    """The test hook that leaves each CTA's first stage unfilled reaches this
    entry point too: with a 20 ms limit the call records NVFP4_ERR_TIMEOUT and
    returns; the next call clears the workspace and gives the right sums."""
    plan, W, wts, ref, shape = _combine_problem(92)
    T, N = shape[0], shape[3]
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    F.nvfp4_device_status(reset=True)
    F.nvfp4_set_timeout_ns(20_000_000)
    F.nvfp4_debug_set_flags(1)
    try:
        _noalloc(plan, W, wts, out, shape)
        assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_TIMEOUT
    finally:
        F.nvfp4_debug_set_flags(0)
        F.nvfp4_set_timeout_ns(1_000_000_000)
    out.view(torch.int16).fill_(0x7FC0)
    _noalloc(plan, W, wts, out, shape)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    check_gemm(bf16_to_np(out), bf16_to_np(ref[:T]), "no-alloc after a timeout")
