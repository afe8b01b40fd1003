"""The skinny NVFP4 W4A16 product (oracle; test infrastructure only).

gemma-cuda-hybrid README, "Everything it has / Inference engine": every M<=16
GEMM (verify dense, both lm_heads, draft linears) computes y[M, N] = x . W^T
with NVFP4 weights and 16-bit activations, fp32 accumulation, bf16 out.

Here the product is taken exactly in float64 on the dequantized weights (the
definition, with numpy's matmul as the library primitive; it is pinned by a
triple loop in the tests).  The per-output tolerance quantity sum_k |w*x| is
returned beside it.
"""

from __future__ import annotations

import numpy as np

from .formats import dequantize_matrix, bf16_round


def gemm_fp64(w_hat: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y[m, n] = sum_k w_hat[n, k] * x[m, k] in float64."""
    return np.asarray(x, np.float64) @ np.asarray(w_hat, np.float64).T


def abs_gemm_fp64(w_hat: np.ndarray, x: np.ndarray) -> np.ndarray:
    """sum_k |w_hat[n, k] * x[m, k]|, the scale of the per-output error bound."""
    return np.abs(np.asarray(x, np.float64)) @ np.abs(np.asarray(w_hat, np.float64)).T


def nvfp4_gemm(nib, scales, g, x):
    """Reference for the library's dense call: returns (y_exact, y_bf16, sum|w*x|)."""
    w_hat = dequantize_matrix(nib, scales, g)
    y = gemm_fp64(w_hat, x)
    return y, bf16_round(y), abs_gemm_fp64(w_hat, x)
