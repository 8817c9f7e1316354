"""Grouped GEMM at the full workload sizes, in the launch configuration the
benchmark times, checked on sampled outputs that the oracle computes one by
one (whole experts' weights are quantised by the oracle for their global
scale; only sampled rows and columns are multiplied)."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_nvfp4_gb300 import inputs, moe
from moe_grouped_gemm_nvfp4_gb300 import nvfp4 as F
from parity import bf16_to_np, check_gemm

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _device_weights(E, N, K, seed):
    w = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    for e in range(E):
        w[e] = inputs.device_normal_bf16((N, K), 0.02, seed * 100003 + e, "cuda")
    return w


def _oracle_weight_rows(w_dev, e, cols, sparse=False):
    """Oracle-quantised rows `cols` of expert e (global scale over all of W_e;
    sparse: W_e pruned to 2:4 over element pairs first)."""
    we = w_dev[e].float().cpu().numpy()
    if sparse:
        we = oracle.prune_pairs_2of4(we)
    ge = oracle.global_scale(we)
    p, s, _ = oracle.quantize(we[cols], g=ge)
    return oracle.dequantize(p, s, ge)


def _routing_for(cfg, g):
    if cfg.routing == "zipf":
        return inputs.zipf_topk(g, cfg.T, cfg.E, cfg.topk)
    return inputs.uniform_topk(g, cfg.T, cfg.E, cfg.topk)


def _gate_up_case(cfg, n_route_samples, n_col_samples, experts_pick, sparse=False):
    g = inputs.rng(cfg.seed)
    xf = g.standard_normal((cfg.T, cfg.K), dtype=np.float32)
    if cfg.outliers:
        xf = inputs.add_outliers(g, xf)
    x = inputs.to_bf16(xf)
    ids = _routing_for(cfg, g)
    w = _device_weights(cfg.E, cfg.N, cfg.K, cfg.seed)
    W = moe.quantize_experts_sparse(w) if sparse else moe.quantize_experts(w)
    plan = moe.GroupedPlan(W, cfg.T, cfg.topk, "gather")
    plan.out.view(torch.int16).fill_(0x7FC0)
    out = plan.run(x.cuda(), torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    off, tok, slot = oracle.route(ids, cfg.E)
    assert np.array_equal(plan.expert_offsets.cpu().numpy(), off)
    x_np = x.float().numpy()
    gx = oracle.global_scale(x_np)
    sel = np.random.Generator(np.random.PCG64(cfg.seed + 99))
    cols = np.sort(sel.choice(cfg.N, n_col_samples, replace=False))
    counts = off[1:] - off[:-1]
    for e in experts_pick(counts):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        p = np.arange(lo, hi)
        if p.size > n_route_samples:       # keep the first and last rows of every tile edge
            edges = np.unique(np.clip(np.concatenate([np.arange(0, p.size, 128),
                                                      np.arange(127, p.size, 128)]), 0,
                                      p.size - 1))
            rest = sel.choice(p.size, n_route_samples, replace=False)
            p = p[np.unique(np.concatenate([edges, rest]))]
        px, sx, _ = oracle.quantize(x_np[tok[p]], g=gx)
        ref = oracle.dequantize(px, sx, gx) @ _oracle_weight_rows(w, e, cols, sparse).T
        got = bf16_to_np(out[torch.from_numpy(p).cuda()][:, torch.from_numpy(cols).cuda()])
        check_gemm(got, ref, f"{cfg.name} expert {e} ({hi - lo} routes)")
    # nothing left unwritten anywhere in the route-ordered output
    assert not torch.isnan(out[: cfg.T * cfg.topk]).any().item()


def test_decode_gate_up_full():
    cfg = inputs.CONFIGS["decode_gate_up"]
    _gate_up_case(cfg, 64, 256, lambda c: [int(np.argmax(c)), int(np.argmin(c)), 0, 77])


def test_decode_gate_up_sparse_full():
    """The same workload with the weights pruned to 2:4 and streamed as sparse
    tiles (32-route token tiles, two weight tiles per unit)."""
    cfg = inputs.CONFIGS["decode_gate_up"]
    _gate_up_case(cfg, 64, 256, lambda c: [int(np.argmax(c)), int(np.argmin(c)), 0, 77],
                  sparse=True)


def test_prefill_skewed_full():
    cfg = inputs.CONFIGS["prefill_skewed"]
    g = inputs.rng(cfg.seed)
    ids = _routing_for(cfg, g)
    counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
    assert counts.max() > 1000 and (counts == 0).sum() >= 1     # the workload's skew
    _gate_up_case(cfg, 192, 192,
                  lambda c: [int(np.argmax(c)), int(np.argsort(c)[len(c) // 2]),
                             int(np.argmin(np.where(c > 0, c, 1 << 30)))])


@pytest.mark.parametrize("name,sparse", [("decode_down_256", False), ("decode_down_512", False),
                                         ("decode_down_1024", False), ("decode_down_512", True)])
def test_decode_down_full(name, sparse):
    cfg = inputs.CONFIGS[name]
    g = inputs.rng(cfg.seed)
    ids = inputs.uniform_topk(g, cfg.T, cfg.E, cfg.topk)
    wts = inputs.dirichlet_weights(g, cfg.T, cfg.topk)
    R = cfg.T * cfg.topk
    h = inputs.normal_bf16(g, (R, cfg.K))
    w = _device_weights(cfg.E, cfg.N, cfg.K, cfg.seed)
    W = moe.quantize_experts_sparse(w) if sparse else moe.quantize_experts(w)
    plan = moe.GroupedPlan(W, cfg.T, cfg.topk, "combine")
    plan.out.view(torch.int16).fill_(0x7FC0)
    out = plan.run(h.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(wts).cuda())
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    assert not torch.isnan(out[: cfg.T]).any().item()
    off, tok, slot = oracle.route(ids, cfg.E)
    h_np = h.float().numpy()
    gh = oracle.global_scale(h_np)
    sel = np.random.Generator(np.random.PCG64(cfg.seed + 7))
    tokens = np.sort(sel.choice(cfg.T, 2, replace=False))
    cols = np.sort(sel.choice(cfg.N, 256, replace=False))
    ref = np.zeros((tokens.size, cols.size))
    for i, t in enumerate(tokens):
        for p in np.nonzero(tok == t)[0]:
            e = int(np.searchsorted(off, p, side="right") - 1)
            ph, sh, _ = oracle.quantize(h_np[p:p + 1], g=gh)
            y = oracle.dequantize(ph, sh, gh) @ _oracle_weight_rows(w, e, cols, sparse).T
            ref[i] += np.float64(wts[t, slot[p]]) * y[0]
    got = bf16_to_np(out[torch.from_numpy(tokens).cuda()][:, torch.from_numpy(cols).cuda()])
    check_gemm(got, ref, name + (" sparse" if sparse else ""))


@pytest.mark.parametrize("B,Hq,Hkv,L,D", [
    (16, 32, 8, 16384, 128),     # groups of 4 over 128-wide heads: the pipelined kernel
    (16, 64, 8, 16384, 128),     # groups of 8
    (16, 32, 8, 8192, 256),      # 256-wide heads: the scores and values passes
    (8, 8, 2, 32768, 512),       # 512-wide heads
])
def test_decode_attention_full_size(B, Hq, Hkv, L, D):
    """Decode attention over an NVFP4 KV cache at the benchmark's shapes, in the
    launch configuration it times, checked on sampled (sequence, KV head)
    groups: the oracle takes each cache's global from the whole tensor,
    quantises the sampled groups' rows itself (codes and scales bit-exact
    against the GPU's), and computes their heads' outputs.  Sequence lengths:
    full, ragged (a split boundary's neighbourhood), and a single token."""
    from moe_grouped_gemm_nvfp4_gb300 import attention
    from test_gpu_attention import _check
    G = Hq // Hkv
    dev = "cuda"
    kd = inputs.device_normal_bf16((B, Hkv, L, D), 1.0, 71, dev)
    vd = inputs.device_normal_bf16((B, Hkv, L, D), 1.0, 72, dev)
    q = inputs.device_normal_bf16((B, Hq, D), 1.0, 73, dev)
    kq, vq = attention.quantize_kv(kd), attention.quantize_kv(vd)
    g = inputs.rng(B * 7 + L + D)
    lens = np.full(B, L, dtype=np.int64)
    lens[1] = L // 2 + 1 + int(g.integers(0, 100))
    lens[2] = 1
    scale = 1.0 / np.sqrt(D)
    plan = attention.DecodeAttention(B, Hq, Hkv, L, D, dev)
    plan.out.view(torch.int16).fill_(0x7FC0)
    out = plan.run(q, kq, vq, torch.from_numpy(lens.astype(np.int32)).to(dev), scale)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    gk = oracle.global_scale(kd.float().cpu().numpy())
    gv = oracle.global_scale(vd.float().cpu().numpy())
    assert kq[2].item() == gk and vq[2].item() == gv
    qf = q.float().cpu().numpy()
    outf = out.float().cpu().numpy().astype(np.float64)
    for b, j in ((0, 0), (1, Hkv - 1), (2, Hkv // 2), (B - 1, 1 % Hkv)):
        n = int(lens[b])
        kf = kd[b, j, :n].float().cpu().numpy()
        vf = vd[b, j, :n].float().cpu().numpy()
        pk, sk = oracle.quantize_kv(kf, gk)
        pv, sv = oracle.quantize_kv(vf, gv)
        assert np.array_equal(kq[0][b, j, :n].cpu().numpy(), pk)
        assert np.array_equal(kq[1][b, j, :n].cpu().numpy(), sk)
        assert np.array_equal(vq[0][b, j, :n].cpu().numpy(), pv)
        assert np.array_equal(vq[1][b, j, :n].cpu().numpy(), sv)
        ref = oracle.decode_attention(qf[b:b + 1, j * G:(j + 1) * G],
                                      oracle.dequantize_kv(pk, sk, gk)[None, None],
                                      oracle.dequantize_kv(pv, sv, gv)[None, None], [n], scale)
        _check(outf[b:b + 1, j * G:(j + 1) * G], ref, f"attention B{B} Hq{Hq} D{D} b{b} j{j}")
