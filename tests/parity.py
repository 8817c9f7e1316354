"""Helpers shared by the GPU parity tests (test infrastructure)."""
from __future__ import annotations

import numpy as np
import torch

NAN_BF16 = 0x7FC0


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |x| (8 significant bits)."""
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.exp2(e - 7)


def check_gemm(got: np.ndarray, ref: np.ndarray, name: str = "") -> dict:
    """GEMM tolerance against the FP64 oracle.

    normwise  ||got - ref|| / ||ref|| <= 2e-3
    per element |got - ref| <= 1e-2 * rms(ref) + 0.5 * ulp_bf16(ref)
    (the half-ulp term is the final BF16 rounding that even an exact FP32
    accumulator incurs; without it the 1e-2 * rms bound fails for a perfect
    kernel wherever |C| is about 2 rms or more).
    """
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output (unwritten NaN sentinel?)"
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    nref = float(np.linalg.norm(ref))
    normwise = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got))
    allow = 1e-2 * rms + 0.5 * ulp_bf16(ref)
    worst = float(np.max(err / np.maximum(allow, 1e-300))) if err.size else 0.0
    stats = dict(normwise=normwise, max_abs=float(err.max()) if err.size else 0.0, rms=rms,
                 max_over_allow=worst, literal_max_over_rms=float(err.max() / rms) if rms else 0)
    assert normwise <= 2e-3, f"{name}: normwise {normwise:.3e} > 2e-3 ({stats})"
    assert worst <= 1.0, f"{name}: element error over allowance ({stats})"
    return stats


def nan_filled(shape, dtype=torch.bfloat16, device="cuda") -> torch.Tensor:
    t = torch.empty(shape, dtype=dtype, device=device)
    if dtype == torch.bfloat16:
        t.view(torch.int16).fill_(NAN_BF16)
    else:
        t.fill_(float("nan"))
    return t
