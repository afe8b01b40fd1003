"""The step before the MoE routing and the step after the lm_head (oracle; test
infrastructure only).  The GPU path for these is not built yet.

TensorSharp docs/models/gemma4.md, "4.6 MoE", step 2: router matmul, then an
unweighted RMSNorm, then a multiply by the learned scale ffn_gate_inp.scale; the
result is the router logits that the top-k takes.  Same page, "4.8 Logit
softcap": tanh(logits / cap) * cap when the final-logit softcap is positive.

Readings: the learned scale is one entry per expert (broadcast over tokens); the
RMSNorm epsilon is 1e-6 (the pages give none); the router weight is an NVFP4
matrix like every other weight of the path, so the router matmul is the skinny
GEMM with N = n_experts.  The softcap is monotone: it changes the returned maximum
logit and the sampling keys, not the greedy argmax.
"""

from __future__ import annotations

import numpy as np

from .formats import dequantize_matrix

RMS_EPS = 1e-6


def rmsnorm_unweighted(v, eps: float = RMS_EPS):
    """v / sqrt(mean(v^2) + eps) over the last axis, float64."""
    v = np.asarray(v, np.float64)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)


def router_logits(x, nib, scales, g, expert_scale, eps: float = RMS_EPS):
    """logits[m, e] = rmsnorm_unweighted(W_hat . x_m)[e] * expert_scale[e]."""
    raw = np.asarray(x, np.float64) @ dequantize_matrix(nib, scales, g).T
    return rmsnorm_unweighted(raw, eps) * np.asarray(expert_scale, np.float64)


def softcap(logits, cap: float):
    """cap * tanh(logits / cap) for cap > 0; the logits unchanged otherwise."""
    logits = np.asarray(logits, np.float64)
    return cap * np.tanh(logits / cap) if cap > 0 else logits
