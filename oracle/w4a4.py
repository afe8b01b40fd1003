"""W4A4 NVFP4 verify products (oracle; test infrastructure only).

The pages do not describe this variant; it is the "next" row that quantizes the
activations as well as the weights, so that both operands of every product are
NVFP4 values.  Readings taken where nothing fixes the choice:

- The activations use the weights' recipe (gemma-cuda-hybrid README,
  "Everything it has / Inference engine": E2M1 codes, an E4M3 scale per 16
  consecutive values along K, an FP32 global scale), with the codes decided on
  exact quotients exactly as for the weights (formats.quantize_matrix).
- The global scale is per token row, g_m = fp32(amax_k |x[m, k]| / (448 * 6)):
  each row is quantized as a matrix of its own, so a token's codes do not
  depend on the other tokens of the batch.
- The product is the exact sum over the dequantized operands,
  y[m, n] = sum_k w_hat[n, k] * x_hat[m, k]; the tolerance quantity is
  sum_k |w_hat * x_hat| (the quantization error of x is part of the definition,
  not of the error).
"""

from __future__ import annotations

import numpy as np

from .formats import bf16_round, dequantize_matrix, quantize_matrix
from .gemm import abs_gemm_fp64, gemm_fp64


def quantize_activations(x: np.ndarray):
    """Per-row NVFP4 quantization of fp32 activations [m, K]: (codes u8 [m, K/2],
    scales u8 [m, K/16], global scales fp32 [m])."""
    x = np.asarray(x, np.float32)
    m, k = x.shape
    codes = np.empty((m, k // 2), np.uint8)
    scales = np.empty((m, k // 16), np.uint8)
    g = np.empty((m,), np.float32)
    for i in range(m):
        c, s, gi = quantize_matrix(x[i:i + 1])
        codes[i], scales[i], g[i] = c[0], s[0], gi
    return codes, scales, g


def dequantize_activations(codes, scales, g) -> np.ndarray:
    """x_hat [m, K] in float64: row m dequantized with its own global scale."""
    return np.stack([dequantize_matrix(codes[i:i + 1], scales[i:i + 1], g[i])[0] for i in range(codes.shape[0])])


def w4a4_gemm(nib, scales, g, xq):
    """The W4A4 dense product: (y_exact, y_bf16, sum |w_hat * x_hat|) for the weight
    (nib, scales, g) and quantized activations xq = (codes, scales, g)."""
    w_hat = dequantize_matrix(nib, scales, g)
    x_hat = dequantize_activations(*xq)
    y = gemm_fp64(w_hat, x_hat)
    return y, bf16_round(y), abs_gemm_fp64(w_hat, x_hat)
