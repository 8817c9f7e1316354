"""2:4-sparse NVFP4 weights ("The FP4 Frontier", Finding 6) against the oracle:
pruning and the sparse tile layout bit for bit, the sparse grouped GEMM
(gather and weighted combine, every token-tile width) within the GEMM
tolerance, and equal to the dense grouped GEMM on the same pruned weights."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_nvfp4_gb300 import inputs, moe
from moe_grouped_gemm_nvfp4_gb300 import nvfp4 as F
from parity import bf16_to_np, check_gemm

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def _tie_heavy_bf16(g, shape):
    """Few distinct magnitudes, so equal pair scores are common."""
    pool = np.array([0.0, 0.25, 0.5, 1.0, 1.5, 2.0], np.float32)
    v = g.choice(pool, size=shape) * np.where(g.random(shape) < 0.5, -1.0, 1.0)
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols,ties", [(64, 256, False), (37, 520, True), (1, 8, True),
                                            (300, 1024, False)])
def test_prune_bit_exact(rows, cols, ties):
    g = inputs.rng(rows * 7 + cols)
    w = _tie_heavy_bf16(g, (rows, cols)) if ties else inputs.normal_bf16(g, (rows, cols), 0.02)
    ref = torch.from_numpy(oracle.prune_pairs_2of4(w.float().numpy())).to(torch.bfloat16)
    wd = w.cuda()
    out = torch.full_like(wd, float("nan"))
    F.nvfp4_prune_2of4(wd, out)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), _bits(ref))
    F.nvfp4_prune_2of4(wd, wd)                     # in place
    torch.cuda.synchronize()
    assert np.array_equal(_bits(wd), _bits(ref))


def test_prune_strided_rows():
    g = inputs.rng(5)
    full = inputs.normal_bf16(g, (48, 320))
    view = full[:, 32:288]                          # ld 320, cols 256
    ref = oracle.prune_pairs_2of4(view.float().numpy())
    out = torch.zeros((48, 256), dtype=torch.bfloat16, device="cuda")
    F.nvfp4_prune_2of4(view.cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), _bits(torch.from_numpy(ref).to(torch.bfloat16)))


def _random_sparse_packed(g, rows, half):
    """Packed codes with two random kept bytes per group of four (signed zero
    codes among them)."""
    out = np.zeros((rows, half // 4, 4), np.uint8)
    special = np.array([0x00, 0x08, 0x80, 0x88], np.uint8)
    keep = np.argsort(g.random((rows, half // 4, 4)), axis=-1)[..., :2]
    vals = g.integers(0, 256, size=(rows, half // 4, 2), dtype=np.uint8)
    sp = g.random((rows, half // 4, 2)) < 0.2
    vals[sp] = special[g.integers(0, 4, size=int(sp.sum()))]
    np.put_along_axis(out, keep, vals, axis=-1)
    return out.reshape(rows, half)


@pytest.mark.parametrize("rows,K", [(128, 256), (200, 320), (64, 1024), (384, 6144)])
def test_sparse_tiles_bit_exact(rows, K):
    g = inputs.rng(rows + K)
    packed = _random_sparse_packed(g, rows, K // 2)
    sf = g.integers(0, 127, size=(rows, K // 16), dtype=np.uint8)
    ref = oracle.sparse_operand_tiles(packed, sf)
    tiles = torch.full((F.nvfp4_sparse_tiles_bytes(rows, K),), 0xA5, dtype=torch.uint8,
                       device="cuda")
    F.nvfp4_device_status(reset=True)
    F.nvfp4_prepack_sparse_weight_tiles(torch.from_numpy(packed).cuda(),
                                        torch.from_numpy(sf).cuda(), tiles)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    assert np.array_equal(tiles.cpu().numpy(), ref)


def test_sparse_tiles_reject_three_kept_bytes():
    g = inputs.rng(3)
    packed = _random_sparse_packed(g, 128, 128)
    packed[77, 40:44] = [1, 2, 3, 0]                # three non-zero bytes in one group
    sf = np.ones((128, 16), np.uint8)
    tiles = torch.empty(F.nvfp4_sparse_tiles_bytes(128, 256), dtype=torch.uint8, device="cuda")
    F.nvfp4_device_status(reset=True)
    F.nvfp4_prepack_sparse_weight_tiles(torch.from_numpy(packed).cuda(),
                                        torch.from_numpy(sf).cuda(), tiles)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status(reset=True) == F.NVFP4_ERR_DEVICE_CHECK


def _pruned_oracle_weights(w_bf16):
    """Oracle: prune each expert, quantise with its own global, dequantise."""
    out = []
    for e in range(w_bf16.shape[0]):
        p = oracle.prune_pairs_2of4(w_bf16[e].float().numpy())
        q, s, gg = oracle.quantize(p)
        out.append(oracle.dequantize(q, s, gg))
    return np.stack(out)


def _routing(g, T, E, k, kind):
    if kind == "zipf":
        return inputs.zipf_topk(g, T, E, k, n_unused=max(1, E // 16))
    return inputs.uniform_topk(g, T, E, k)


GATHER_CASES = [
    (32, 8, 2, 256, 512, "uniform"),       # 32-route token tiles
    (5, 16, 2, 128, 192, "uniform"),       # most experts empty, partial K block
    (128, 16, 4, 256, 320, "uniform"),     # 64-route token tiles, ragged K block
    (300, 4, 2, 128, 256, "uniform"),      # 128-route tiles, two token tiles per expert
    (300, 16, 4, 256, 512, "zipf"),        # skewed with empty experts
    (256, 32, 2, 1280, 256, "uniform"),    # more units than CTAs
]


@pytest.mark.parametrize("T,E,k,N,K,kind", GATHER_CASES)
def test_sparse_grouped_gather_matches_oracle(T, E, k, N, K, kind):
    g = inputs.rng(T * 19 + E + N + K)
    x = inputs.normal_bf16(g, (T, K))
    w = inputs.normal_bf16(g, (E, N, K), 0.02)
    ids = _routing(g, T, E, k, kind)
    W = moe.quantize_experts_sparse(w.cuda())
    plan = moe.GroupedPlan(W, T, k, "gather")
    plan.out.view(torch.int16).fill_(0x7FC0)
    out = plan.run(x.cuda(), torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    off, tok, _ = oracle.route(ids, E)
    px, sx, gx = oracle.quantize(x.float().numpy())
    xh = oracle.dequantize(px, sx, gx)[tok]
    ref = oracle.grouped_gemm(xh, _pruned_oracle_weights(w), off)
    check_gemm(bf16_to_np(out[: T * k]), ref, "sparse grouped gather")


@pytest.mark.parametrize("T,E,k,N,K", [(32, 8, 2, 256, 512), (64, 16, 8, 384, 256),
                                       (400, 4, 2, 128, 256), (256, 32, 2, 1280, 256)])
def test_sparse_grouped_combine_matches_oracle(T, E, k, N, K):
    g = inputs.rng(T * 23 + E + N + K)
    ids = inputs.uniform_topk(g, T, E, k)
    wts = inputs.dirichlet_weights(g, T, k)
    h = inputs.normal_bf16(g, (T * k, K))
    w = inputs.normal_bf16(g, (E, N, K), 0.02)
    W = moe.quantize_experts_sparse(w.cuda())
    plan = moe.GroupedPlan(W, T, k, "combine")
    off, tok, slot = oracle.route(ids, E)
    ph, sh, gh = oracle.quantize(h.float().numpy())
    y = oracle.grouped_gemm(oracle.dequantize(ph, sh, gh), _pruned_oracle_weights(w), off)
    ref = oracle.combine(y, tok, slot, wts, T)
    for call in range(2):
        plan.out.view(torch.int16).fill_(0x7FC0)
        out = plan.run(h.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(wts).cuda())
        torch.cuda.synchronize()
        assert F.nvfp4_device_status() == F.NVFP4_OK
        check_gemm(bf16_to_np(out[:T]), ref, f"sparse grouped combine, call {call}")


@pytest.mark.parametrize("T,E,k,N,K", [(32, 8, 2, 256, 512), (128, 16, 4, 256, 320),
                                       (300, 4, 2, 128, 256)])
def test_sparse_equals_dense_on_the_same_pruned_weights(T, E, k, N, K):
    """Expanding in shared memory feeds the MMAs the very operand the dense
    tiles hold, and the K steps accumulate in the same order: equal bits."""
    g = inputs.rng(T + E * 3 + N + K)
    x = inputs.normal_bf16(g, (T, K)).cuda()
    w = inputs.normal_bf16(g, (E, N, K), 0.02).cuda()
    F.nvfp4_prune_2of4(w.view(E * N, K), w.view(E * N, K))
    ids = torch.from_numpy(inputs.uniform_topk(g, T, E, k)).cuda()
    dense = moe.GroupedPlan(moe.quantize_experts(w), T, k, "gather")
    sparse = moe.GroupedPlan(moe.quantize_experts_sparse(w, pruned=True), T, k, "gather")
    a = dense.run(x, ids).clone()
    b = sparse.run(x, ids)
    torch.cuda.synchronize()
    assert F.nvfp4_device_status() == F.NVFP4_OK
    assert torch.equal(a[: T * k].view(torch.int16), b[: T * k].view(torch.int16))
