"""Seeded synthetic inputs for the NVFP4 GEMM and MoE grouped-GEMM workloads.

This module only draws random numbers and lays them out; it holds none of the
NVFP4 arithmetic (no quantisation, no scale formula, no GEMM).  Both the CUDA
path and the CPU oracle take their inputs from here, so that the two see the
same bytes.

Workload shapes follow the small-batch MoE decode and prefill settings the
pages discuss ("The FP4 Frontier", The Context: 16-64 tokens per expert;
"The Tile That Didn't Fit", The Path to Discovery: ~16 tokens per expert):

* activations ~ N(0, 1) in BF16, weights ~ N(0, 0.02) in BF16;
* top-k routing drawn uniformly without replacement per token, or with a
  Zipf(s) expert popularity for the skewed prefill case;
* routing weights ~ Dirichlet(1, ..., 1) per token, FP32;
* prefill activations carry 0.1% outliers scaled by 50.

Small tensors are drawn on the host with numpy's PCG64.  Full-size weight
tensors (gigabytes) are drawn on the device with a seeded torch generator,
expert by expert; `device_normal_bf16` documents that path.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = [
    "Config", "CONFIGS", "rng", "to_bf16", "normal_bf16", "uniform_topk",
    "zipf_topk", "dirichlet_weights", "add_outliers", "device_normal_bf16",
]


def rng(seed: int) -> np.random.Generator:
    """The seeded host generator every small input comes from."""
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """FP32 numpy array -> BF16 CPU tensor (torch's round-to-nearest-even cast)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal_bf16(g: np.random.Generator, shape, sigma: float = 1.0) -> torch.Tensor:
    """N(0, sigma^2) drawn in FP32 on the host, cast to BF16."""
    return to_bf16(g.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def add_outliers(g: np.random.Generator, x: np.ndarray, frac: float = 1e-3,
                 factor: float = 50.0) -> np.ndarray:
    """Multiply a seeded random `frac` of the elements of x (FP32) by `factor`."""
    x = np.array(x, dtype=np.float32, copy=True)
    n = x.size
    k = int(round(frac * n))
    idx = g.choice(n, size=k, replace=False)
    flat = x.reshape(-1)
    flat[idx] *= np.float32(factor)
    return x


def uniform_topk(g: np.random.Generator, T: int, E: int, k: int) -> np.ndarray:
    """Per token, k distinct experts drawn uniformly without replacement: int32 [T, k]."""
    keys = g.random((T, E))
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def zipf_topk(g: np.random.Generator, T: int, E: int, k: int, s: float = 1.1,
              n_unused: int = 8) -> np.ndarray:
    """Skewed routing: expert popularity p_e proportional to rank^-s.

    Ranks come from a seeded permutation of the experts; the `n_unused`
    lowest-ranked experts get p = 0 so that some experts receive no token.
    Each token draws k distinct experts without replacement with
    probabilities p (successive sampling, done with Gumbel top-k keys).
    Returns int32 [T, k].
    """
    ranks = g.permutation(E) + 1                      # rank of each expert, 1..E
    p = ranks.astype(np.float64) ** (-s)
    p[ranks > E - n_unused] = 0.0
    p /= p.sum()
    with np.errstate(divide="ignore"):
        logp = np.log(p)
    gumbel = -np.log(-np.log(g.random((T, E))))
    keys = logp[None, :] + gumbel
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def dirichlet_weights(g: np.random.Generator, T: int, k: int) -> np.ndarray:
    """Routing weights ~ Dirichlet(1, ..., 1) per token: float32 [T, k]."""
    return g.dirichlet(np.ones(k), size=T).astype(np.float32)


def device_normal_bf16(shape, sigma: float, seed: int, device) -> torch.Tensor:
    """N(0, sigma^2) drawn on `device` by a torch generator seeded with `seed`.

    Used for weight tensors too large to draw on the host in reasonable time
    (up to 3.2e9 elements).  The values are reproducible for a given torch
    build and device; the oracle reads them back from the device tensor.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(0.0, sigma, generator=gen)
    return x.to(torch.bfloat16)


@dataclass(frozen=True)
class Config:
    """One workload: a single GEMM (E == 0) or an MoE grouped GEMM."""
    name: str
    kind: str                 # "gemm" | "gate_up" | "down" | "prefill"
    K: int
    N: int
    M: int = 0                # rows of A for a single GEMM
    E: int = 0                # experts
    T: int = 0                # tokens
    topk: int = 0
    seed: int = 0
    sigma_w: float = 0.02
    routing: str = "uniform"  # "uniform" | "zipf"
    outliers: bool = False
    extra: dict = field(default_factory=dict, compare=False, hash=False)


CONFIGS = {
    "tiny_gemm": Config("tiny_gemm", "gemm", K=512, N=256, M=16, seed=0),
    "dense_8192": Config("dense_8192", "gemm", K=8192, N=8192, M=8192, seed=1),
    "decode_gate_up": Config("decode_gate_up", "gate_up", K=6144, N=4096, E=128,
                             T=256, topk=8, seed=2),
    "decode_down_256": Config("decode_down_256", "down", K=2048, N=6144, E=128,
                              T=256, topk=8, seed=3),
    "decode_down_512": Config("decode_down_512", "down", K=2048, N=6144, E=128,
                              T=512, topk=8, seed=3),
    "decode_down_1024": Config("decode_down_1024", "down", K=2048, N=6144, E=128,
                               T=1024, topk=8, seed=3),
    "prefill_skewed": Config("prefill_skewed", "prefill", K=6144, N=4096, E=128,
                             T=8192, topk=8, seed=4, routing="zipf", outliers=True),
}
