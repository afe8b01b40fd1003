"""MoE FFN layer with NVFP4 experts (oracle; test infrastructure only).

Sources (page title, section):

* TensorSharp docs/models/gemma4.md, "3.2 Per-layer (MoE)" and "4.6 MoE": the
  router produces logits, experts are chosen by top-k over the softmax, each
  chosen expert runs a gated FFN over its fused gate+up weight and its down
  weight, and the branch is the probability-weighted sum of the experts.
* Same page, "3.1 Per-layer (dense)": the fused gate+up matmul yields
  [gate || up] (gate rows first), then g = GELU(gate), then down(g * up).
* Same page, "14. Optimization opportunities / Completed (Expert-batched
  FFN)": the layer runs as grouped gate[+up] / down products over stacked 3-D
  expert weights with a fused GEGLU and an expert aggregation.
* TensorFold issue #1048, "Steps", step 2: the activation is GELU-tanh.
* gemma-cuda-hybrid README, "What it is": 128 experts, top-8 + 1 shared.

Readings where the pages leave a step open: top-8 is taken on the raw logits (descending,
ties to the lower expert id) and the softmax runs over the 8 chosen logits;
this picks the same set as softmax-then-top-k and equals renormalising the
chosen softmax weights.  The shared expert has the same shape as a routed
expert and is added with weight 1.  The intermediate h = gelu_tanh(gate) * up
is rounded to bf16 (it is the 16-bit activation of the down projection); the
expert sum is exact and the layer output is rounded to bf16 once.
"""

from __future__ import annotations

import math

import numpy as np

from .formats import dequantize_matrix, bf16_round


def route_topk(logits: np.ndarray, top_k: int, softmax_all: bool = False, expert_scale=None):
    """Per token: ids of the top_k largest logits (ties -> lower id) and their weights.

    Default: the softmax over the top_k chosen logits.  softmax_all: the literal
    topK(softmax(logits)) of TensorSharp docs/models/gemma4.md, "3.2 Per-layer
    (MoE)" -- the softmax over all experts' logits, read at the chosen experts
    (not renormalised).  expert_scale [E]: each weight times its expert's scale
    (a per-expert down-projection scale folded into the routing weights, same
    page, "14. Optimization opportunities").
    A NaN logit counts as -inf; -inf logits are chosen last, lowest id first, and a
    token whose logits are all -inf gets weight 0 on every slot.
    Returns (ids int32 [M, top_k] in descending-logit order, probs float64 [M, top_k]).
    """
    l = np.asarray(logits, dtype=np.float64)
    l = np.where(np.isnan(l), -np.inf, l)          # a NaN logit counts as -inf
    order = np.argsort(-l, axis=1, kind="stable")[:, :top_k]
    chosen = np.take_along_axis(l, order, axis=1)
    top = chosen[:, :1]
    none = np.isneginf(top)                        # every logit -inf: weight 0 everywhere
    shift = np.where(none, 0.0, top)
    z = np.where(none, 0.0, np.exp(chosen - shift))
    if softmax_all:
        den = np.sum(np.exp(l - shift), axis=1, keepdims=True)
    else:
        den = np.sum(z, axis=1, keepdims=True)
    probs = np.where(none, 0.0, z / np.where(none, 1.0, den))
    if expert_scale is not None:
        probs = probs * np.asarray(expert_scale, np.float64)[order]
    return order.astype(np.int32), probs


def group_by_expert(ids: np.ndarray, n_experts: int):
    """Stable grouping of the (token, slot) pairs by expert.

    Pair index p = t * top_k + r.  Returns (counts [E], offsets [E+1],
    sorted_pairs [M*top_k]): expert e's pairs are sorted_pairs[offsets[e]:offsets[e+1]]
    in ascending p.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=n_experts).astype(np.int32)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    sorted_pairs = np.argsort(flat, kind="stable").astype(np.int32)
    return counts, offsets, sorted_pairs


def gelu_tanh(z):
    """0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))) in float64."""
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z ** 3)))


def expert_ffn(wgu_hat: np.ndarray, wd_hat: np.ndarray, x: np.ndarray):
    """One expert on token rows x [T, d].

    wgu_hat [2I, d] (rows 0..I-1 gate, I..2I-1 up), wd_hat [d, I].
    Returns (h_bf16 [T, I], d_out [T, d] exact, sum|Wd*h| [T, d]).
    """
    inter = wgu_hat.shape[0] // 2
    gu = np.asarray(x, np.float64) @ wgu_hat.T
    h = gelu_tanh(gu[:, :inter]) * gu[:, inter:]
    hb = bf16_round(h)
    d_out = hb @ wd_hat.T
    d_abs = np.abs(hb) @ np.abs(wd_hat).T
    return hb, d_out, d_abs


def moe_layer(x, logits, top_k, gate_up, down, shared_gate_up=None, shared_down=None, softmax_all=False,
              expert_scale=None):
    """The whole MoE FFN layer.

    gate_up = (nib [E, 2I, d/2], scales [E, 2I, d/16], g [E]); down likewise for [E, d, I];
    shared_* = (nib, scales, g) of one matrix or None.
    Returns a dict with ids, probs, offsets, sorted_pairs, out (exact), out_bf16,
    tol_scale (sum_r p * sum_j |Wd h| + shared term) and h for every pair.
    """
    x = np.asarray(x, np.float64)
    m, d = x.shape
    n_exp = gate_up[0].shape[0]
    ids, probs = route_topk(logits, top_k, softmax_all, expert_scale)
    counts, offsets, sorted_pairs = group_by_expert(ids, n_exp)
    out = np.zeros((m, d))
    tol = np.zeros((m, d))
    h_all = {}
    for e in range(n_exp):
        pairs = sorted_pairs[offsets[e]:offsets[e + 1]]
        if pairs.size == 0:
            continue
        toks = pairs // top_k
        wgu = dequantize_matrix(gate_up[0][e], gate_up[1][e], gate_up[2][e])
        wd = dequantize_matrix(down[0][e], down[1][e], down[2][e])
        hb, dd, da = expert_ffn(wgu, wd, x[toks])
        for i, p in enumerate(pairs):
            t, r = divmod(int(p), top_k)
            out[t] += probs[t, r] * dd[i]
            tol[t] += probs[t, r] * da[i]
            h_all[int(p)] = hb[i]
    if shared_gate_up is not None:
        wgu = dequantize_matrix(*shared_gate_up)
        wd = dequantize_matrix(*shared_down)
        hb, dd, da = expert_ffn(wgu, wd, x)
        out += dd
        tol += da
        for t in range(m):
            h_all[m * top_k + t] = hb[t]
    return dict(ids=ids, probs=probs, counts=counts, offsets=offsets,
                sorted_pairs=sorted_pairs, out=out, out_bf16=bf16_round(out),
                tol_scale=tol, h=h_all)
