"""Helpers shared by the GPU parity tests (upload inputs, compare with the oracle)."""

from __future__ import annotations

import numpy as np
import torch

from nvfp4_w4a16_moe_skinny_gb300 import workloads as W

# Per-output bound: |y - y_exact| <= 1e-3 * sum|w*x|  (+ the output's own bf16
# rounding, at most 2^-8 |y| by round-to-nearest, for bf16 outputs).
REL_TOL = 1e-3
BF16_HALF_ULP = 2.0 ** -8


def dev():
    return torch.device("cuda", 0)


def upload_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev())


def upload_bf16(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).to(dev())
    return t.view(torch.bfloat16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def check_bound(got: np.ndarray, exact: np.ndarray, abs_scale: np.ndarray, bf16_out: bool, what: str):
    """Assert the per-output bound and return the worst ratio err / allowed."""
    err = np.abs(got - exact)
    allowed = REL_TOL * abs_scale + (BF16_HALF_ULP * np.abs(exact) if bf16_out else 0.0)
    allowed = np.maximum(allowed, 1e-30)
    ratio = err / allowed
    worst = float(ratio.max()) if ratio.size else 0.0
    bad = np.argwhere(ratio > 1.0)
    assert bad.size == 0, (f"{what}: {bad.shape[0]} outputs out of bound, worst ratio {worst:.3g} at "
                           f"{tuple(bad[0])}: got {got[tuple(bad[0])]}, exact {exact[tuple(bad[0])]}")
    return worst


def ragged_weight(n, k, seed):
    return W.weight((n, k), seed)
