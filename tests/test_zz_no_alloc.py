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
