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


def oracle_quantize(w: np.ndarray):
    """The oracle's canonical NVFP4 bytes of one fp32 matrix [N, K] or a stack [E, N, K]:
    (nibbles, scales, global scales float32 [E] or scalar)."""
    from oracle import formats as F
    if w.ndim == 2:
        return F.quantize_matrix(w)
    return F.quantize_stack(w)


def upload_oracle_weight(lib, q, gated: bool = False):
    """Repack the oracle's canonical bytes on the GPU into the kernel layout: the kernels
    then read exactly the codes the oracle computes with."""
    nib, sc, g = q
    g = np.atleast_1d(np.asarray(g, np.float32))
    return lib.repack(torch.from_numpy(np.ascontiguousarray(nib)).to(dev()),
                      torch.from_numpy(np.ascontiguousarray(sc)).to(dev()),
                      torch.from_numpy(g).to(dev()), gated=gated)


def assert_gpu_quantizer_matches(lib, w: np.ndarray, q, what: str):
    """The library's GPU quantizer gives the oracle's bytes for this matrix (stack)."""
    nib, sc, g = lib.quantize(upload_f32(w))
    onib, osc, og = q
    assert np.array_equal(np.atleast_1d(g.cpu().numpy()), np.atleast_1d(np.asarray(og, np.float32))), what
    assert np.array_equal(sc.cpu().numpy(), osc), f"{what}: scale codes differ"
    assert np.array_equal(nib.cpu().numpy(), onib), f"{what}: element codes differ"
