"""Decode attention over an NVFP4 KV cache ("The Blackwell architectural
split", The A4Q Kernel) against the FP64 oracle.

Tolerance: the kernel computes scores, exponentials and weighted sums in
binary32 (relative error ~1e-6 of the largest output) and rounds the output
to BF16 (half an ulp), so per element |gpu - ref| <= 0.5 ulp_bf16(ref) +
1e-4 * max|ref|, and normwise <= 4e-3."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_nvfp4_gb300 import attention, inputs
from moe_grouped_gemm_nvfp4_gb300 import nvfp4 as F
from parity import ulp_bf16

pytestmark = pytest.mark.gpu


def _case(seed, B, Hq, Hkv, L, D):
    g = inputs.rng(seed)
    q = inputs.normal_bf16(g, (B, Hq, D))
    k = inputs.normal_bf16(g, (B, Hkv, L, D))
    v = inputs.normal_bf16(g, (B, Hkv, L, D))
    return q, k, v


def _check(got, ref, name):
    assert np.isfinite(got).all(), f"{name}: non-finite output"
    err = np.abs(got - ref)
    allow = 0.5 * ulp_bf16(ref) + 1e-4 * np.abs(ref).max()
    worst = float((err / allow).max())
    nref = np.linalg.norm(ref)
    normwise = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got))
    assert worst <= 1.0, f"{name}: element error {worst:.3f} x allowance"
    assert normwise <= 4e-3, f"{name}: normwise {normwise:.2e}"


@pytest.mark.parametrize("B,Hq,Hkv,L,D,lens", [
    (2, 4, 4, 100, 128, [100, 37]),          # one query head per KV head
    (3, 8, 2, 300, 64, [300, 1, 0]),         # groups of 4, a one-token and an empty sequence
    (1, 16, 2, 1000, 128, [1000]),           # groups of 8, several splits
    (2, 4, 1, 2500, 256, [2500, 1333]),      # ragged split tails
    (1, 4, 1, 700, 512, [700]),              # 512-wide heads
    (4, 2, 1, 64, 512, [64, 3, 33, 17]),
    (2, 8, 8, 4097, 64, [4097, 4096]),       # chunk boundary +- 1
    (2, 8, 2, 333, 128, [333, 200]),         # scale slabs not in 16-byte units
    (4, 16, 2, 5000, 128, [5000, 4999, 2048, 129]),  # several work items per CTA, empty splits
    (2, 8, 1, 1500, 64, [1500, 777]),        # groups of 8 over 64-wide heads, ragged tiles
    (2, 8, 2, 3000, 128, [3000, 2999]),      # groups of 4, a tile of one token
    (2, 8, 4, 1000, 128, [1000, 517]),       # groups of 2 on the tensor cores
    (2, 8, 4, 1000, 256, [1000, 517]),       # 256-wide heads: groups of 2, 4 and 8
    (2, 16, 2, 1500, 256, [1500, 1]),
    (4, 8, 2, 9000, 256, [9000, 8999, 4100, 130]),   # several work items per CTA
    (2, 4, 2, 300, 512, [300, 129]),         # 512-wide heads in groups of 2
    (3, 8, 2, 2000, 512, [2000, 0, 1025]),   # groups of 4, an empty sequence
])
def test_decode_attention_matches_oracle(B, Hq, Hkv, L, D, lens):
    q, k, v = _case(B * 1000 + Hq * 10 + D + L, B, Hq, Hkv, L, D)
    kd, vd = k.cuda(), v.cuda()
    kq = attention.quantize_kv(kd)
    vq = attention.quantize_kv(vd)
    # the oracle quantises the same BF16 cache with its own global
    kf, vf = k.float().numpy(), v.float().numpy()
    gk, gv = oracle.global_scale(kf), oracle.global_scale(vf)
    pk, sk = oracle.quantize_kv(kf, gk)
    pv, sv = oracle.quantize_kv(vf, gv)
    assert np.array_equal(kq[0].cpu().numpy(), pk) and np.array_equal(kq[1].cpu().numpy(), sk)
    assert np.array_equal(vq[0].cpu().numpy(), pv) and np.array_equal(vq[1].cpu().numpy(), sv)
    scale = 1.0 / np.sqrt(D)
    plan = attention.DecodeAttention(B, Hq, Hkv, L, D)
    plan.out.view(torch.int16).fill_(0x7FC0)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = plan.run(q.cuda(), kq, vq, seq, scale)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    ref = oracle.decode_attention(q.float().numpy(), oracle.dequantize_kv(pk, sk, gk),
                                  oracle.dequantize_kv(pv, sv, gv), lens, scale)
    _check(out.float().cpu().numpy().astype(np.float64), ref, f"attention B{B} Hq{Hq} D{D}")
    for b, n in enumerate(lens):
        if n == 0:
            assert not out[b].float().abs().sum().item()


def test_sequence_length_out_of_range_is_reported():
    B, Hq, Hkv, L, D = 2, 2, 1, 64, 64
    q, k, v = _case(5, B, Hq, Hkv, L, D)
    kq, vq = attention.quantize_kv(k.cuda()), attention.quantize_kv(v.cuda())
    plan = attention.DecodeAttention(B, Hq, Hkv, L, D)
    F.nvfp4_device_status(reset=True)
    out = plan.run(q.cuda(), kq, vq, torch.tensor([65, 10], dtype=torch.int32, device="cuda"), 0.125)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_DEVICE_CHECK
    assert not out[0].float().abs().sum().item()          # counted as empty
    assert out[1].float().abs().sum().item() > 0


def test_unsupported_shapes_are_refused():
    q = torch.zeros((1, 8, 512), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, 4, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 1, 4, 32), dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 16, dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(RuntimeError):            # 512-wide heads take groups of at most 4
        F.nvfp4_decode_attention(q, k, s, g, k, s, g, torch.ones(1, dtype=torch.int32,
                                 device="cuda"), 0.1, out, ws)


@pytest.mark.parametrize("D", [128, 512])
def test_rising_and_spiking_scores_move_the_reference_maximum(D):
    """Long splits (L_max 262144 with B 2, Hkv 2: 1024-token splits of 8
    tiles) whose scores rise by about 50 (base 2) along sequence 0 and jump by
    about 70 at a few tokens of sequence 1: for 128-wide heads the tensor-core
    kernel's reference maximum moves inside a split, so O and the sums are
    rescaled there; for 512-wide heads the split's maximum comes from the
    stored scores and every p is at most 1.  Tokens past the first 3000 are
    zero and unread."""
    B, Hq, Hkv, n, L_max = 2, 8, 2, 3000, 262144
    G = Hq // Hkv
    g = inputs.rng(91)
    q = inputs.normal_bf16(g, (B, Hq, D))
    qf = q.float().numpy()
    k = g.standard_normal((B, Hkv, n, D)) * 0.5
    v = g.standard_normal((B, Hkv, n, D))
    for b in range(B):
        for j in range(Hkv):
            u = qf[b, j * G:(j + 1) * G].mean(0)
            u /= np.linalg.norm(u)
            amp = np.linspace(0.0, 6.0, n) if b == 0 else np.zeros(n)
            if b == 1:
                amp[1500:1510] = 8.0
            k[b, j] += 12.0 * amp[:, None] * u[None, :]
    kb = torch.from_numpy(k.astype(np.float32)).to(torch.bfloat16)
    vb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    kd = torch.zeros((B, Hkv, L_max, D), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    kd[:, :, :n] = kb.cuda()
    vd[:, :, :n] = vb.cuda()
    kq, vq = attention.quantize_kv(kd), attention.quantize_kv(vd)
    kf, vf = kb.float().numpy(), vb.float().numpy()
    gk, gv = oracle.global_scale(kf), oracle.global_scale(vf)   # the zero tail leaves amax alone
    assert kq[2].item() == gk and vq[2].item() == gv
    pk, sk = oracle.quantize_kv(kf, gk)
    pv, sv = oracle.quantize_kv(vf, gv)
    assert np.array_equal(kq[0][:, :, :n].cpu().numpy(), pk)
    assert np.array_equal(vq[1][:, :, :n].cpu().numpy(), sv)
    scale = 1.0 / np.sqrt(D)
    plan = attention.DecodeAttention(B, Hq, Hkv, L_max, D)
    plan.out.view(torch.int16).fill_(0x7FC0)
    seq = torch.tensor([n, n], dtype=torch.int32, device="cuda")
    out = plan.run(q.cuda(), kq, vq, seq, scale)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    ref = oracle.decode_attention(qf, oracle.dequantize_kv(pk, sk, gk),
                                  oracle.dequantize_kv(pv, sv, gv), [n, n], scale)
    _check(out.float().cpu().numpy().astype(np.float64), ref, "rising / spiking scores")


@pytest.mark.parametrize("D", [128, 512])
def test_tensor_core_kernel_wait_expires_reports_timeout_and_context_survives(D):
    """Failure path of the tensor-core kernels: with the test hook every CTA's
    producer leaves its first ring stage unfilled, so the expansion's wait can
    only end by its time limit; the kernel records NVFP4_ERR_TIMEOUT, every
    role leaves, the copies in flight are drained, and the next call on the
    same context is correct.  (512-wide heads: both the scores and the values
    kernel take the hook.)"""
    B, Hq, Hkv, L = 2, 8, 2, 1000                        # groups of 4: the tensor-core kernel
    q, k, v = _case(17, B, Hq, Hkv, L, D)
    kq, vq = attention.quantize_kv(k.cuda()), attention.quantize_kv(v.cuda())
    plan = attention.DecodeAttention(B, Hq, Hkv, L, D)
    seq = torch.tensor([L, 611], dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    F.nvfp4_device_status(reset=True)
    F.nvfp4_set_timeout_ns(20_000_000)                 # 20 ms
    F.nvfp4_debug_set_flags(1)
    try:
        plan.run(q.cuda(), kq, vq, seq, 0.125)
        torch.cuda.synchronize()
        assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_TIMEOUT
    finally:
        F.nvfp4_debug_set_flags(0)
        F.nvfp4_set_timeout_ns(1_000_000_000)
    plan.out.view(torch.int16).fill_(0x7FC0)
    out = plan.run(q.cuda(), kq, vq, seq, 0.125)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    kf, vf = k.float().numpy(), v.float().numpy()
    gk, gv = oracle.global_scale(kf), oracle.global_scale(vf)
    pk, sk = oracle.quantize_kv(kf, gk)
    pv, sv = oracle.quantize_kv(vf, gv)
    ref = oracle.decode_attention(q.float().numpy(), oracle.dequantize_kv(pk, sk, gk),
                                  oracle.dequantize_kv(pv, sv, gv), [L, 611], 0.125)
    _check(out.float().cpu().numpy().astype(np.float64), ref, "after timeout")
