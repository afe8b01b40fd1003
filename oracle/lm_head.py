"""NVFP4 lm_head with a greedy per-row argmax (oracle; test infrastructure only).

gemma-cuda-hybrid README: "Headline numbers" (greedy decoding is bit-exact),
"Everything it has / Inference engine" (both lm_heads go through the M<=16
NVFP4 GEMM; the tied embedding is quantized to NVFP4 for a 4x lighter
lm_head), "What it is" (262,144-entry vocabulary).

Per token row m: logits = W_hat . x_m exactly in float64, computed over vocab
chunks (a full float64 dequantisation of a 262,144 x 2,816 matrix would need
5.9 GB); the result is the largest logit and the lowest index that reaches it.
The softcap of TensorSharp docs/models/gemma4.md, "4.8 Logit softcap", is
monotone and is not applied: the raw maximum logit is returned.
"""

from __future__ import annotations

import numpy as np

from .formats import dequantize_matrix


def lm_head_argmax(nib, scales, g, x, chunk_rows: int = 8192, row_lo: int = 0, row_hi=None):
    """Returns dict(max [M], argmax [M], second [M] (2nd-largest logit), tol_scale [M]
    (sum|w*x| of the winning row), logits_of(rows) helper not included)."""
    x = np.asarray(x, np.float64)
    m = x.shape[0]
    n = nib.shape[0] if row_hi is None else row_hi
    best = np.full(m, -np.inf)
    best_i = np.full(m, -1, dtype=np.int64)
    second = np.full(m, -np.inf)
    best_abs = np.zeros(m)
    for lo in range(row_lo, n, chunk_rows):
        hi = min(n, lo + chunk_rows)
        w = dequantize_matrix(nib[lo:hi], scales[lo:hi], g)
        logits = x @ w.T                              # [M, rows]
        absl = np.abs(x) @ np.abs(w).T
        for t in range(m):
            row = logits[t]
            j = int(np.argmax(row))                   # first (lowest) index of the max
            v = row[j]
            # second-largest over this chunk (value only)
            if row.size > 1:
                part = np.partition(row, -2)[-2:]
                c2 = part[0] if part[1] == v else part[1]
                c2 = min(c2, v)
            else:
                c2 = -np.inf
            if v > best[t]:
                second[t] = max(best[t], c2)
                best[t], best_i[t], best_abs[t] = v, lo + j, absl[t, j]
            else:
                second[t] = max(second[t], v)
    return dict(max=best, argmax=best_i.astype(np.int32), second=second, tol_scale=best_abs)


def logits_rows(nib, scales, g, x, rows):
    """Exact logits of selected vocab rows: returns (logits [M, R], sum|w*x| [M, R])."""
    rows = np.asarray(rows, dtype=np.int64)
    w = dequantize_matrix(nib[rows], scales[rows], g)
    x = np.asarray(x, np.float64)
    return x @ w.T, np.abs(x) @ np.abs(w).T
