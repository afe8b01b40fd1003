"""GPU parity: the router normalisation (row f2) -- router logits from the hidden state
through the C ABI (moe_router_logits: the NVFP4 router matmul, the unweighted RMSNorm,
the learned per-expert scale; TensorSharp docs/models/gemma4.md, "4.6 MoE", step 2)
against the FP64 oracle, and the top-k taken on them."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as OM
from oracle import router as OR
from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
from tests.gpu_helpers import upload_bf16, upload_f32, upload_oracle_weight

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _case(lib, m, n_exp=W.N_EXPERTS, d=W.HIDDEN, seed=0):
    w = W.weight((n_exp, d), W.seed_of("router", n_exp, d, "w", seed))
    scale = (0.5 + np.abs(W.normal_f32((n_exp,), W.seed_of("router", n_exp, "scale", seed)))).astype(np.float32)
    xb, xf = W.activations((m, d), W.seed_of("router", m, d, "x", seed))
    q = F.quantize_matrix(w)
    logits = lib.router_logits(upload_oracle_weight(lib, q), upload_bf16(xb), upload_f32(scale), EPS)
    torch.cuda.synchronize()
    return logits.cpu().numpy().astype(np.float64), q, scale, xf.astype(np.float64)


def _bound(q, scale, xf):
    """Per-logit bound: the GEMM's 1e-3 * sum|w*x| carried through the RMSNorm (the norm
    moves by at most the largest raw error) and the scale, plus fp32 rounding."""
    w_hat = F.dequantize_matrix(*q)
    raw = xf @ w_hat.T
    a = np.abs(xf) @ np.abs(w_hat).T
    delta = 1e-3 * a
    big = delta.max(axis=1, keepdims=True)
    rms = np.sqrt(np.mean(raw ** 2, axis=1, keepdims=True) + EPS)
    ref = OR.router_logits(xf, *q, scale, EPS)
    tol = scale * (delta + np.abs(raw) * big / rms) / (rms - big) + 1e-5 * np.abs(ref) + 1e-7
    return ref, tol


@pytest.mark.parametrize("m", [1, 3, 8, 15, 16])
def test_router_logits_match_oracle(lib, m):
    got, q, scale, xf = _case(lib, m)
    ref, tol = _bound(q, scale, xf)
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"m={m}: worst {np.max(err / tol):.3g} x bound"
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [1, 15])
def test_router_logits_then_topk(lib, m):
    """The top-8 ids taken on the GPU logits (moe_route_topk) equal the oracle's top-8 on
    exact logits, except where the oracle's 8th and 9th logits lie within the bound."""
    got, q, scale, xf = _case(lib, m, seed=1)
    ref, tol = _bound(q, scale, xf)
    ids, probs, _, _ = lib.route_topk(torch.from_numpy(got.astype(np.float32)).cuda(), W.TOP_K)
    torch.cuda.synchronize()
    oids, _ = OM.route_topk(ref, W.TOP_K)
    for t in range(m):
        srt = np.sort(ref[t])[::-1]
        if srt[W.TOP_K - 1] - srt[W.TOP_K] > 2 * tol[t].max():
            assert set(ids[t].cpu().numpy().tolist()) == set(oids[t].tolist()), t
    assert lib.device_error() == 0


def test_router_logits_without_scale_is_unit_rms(lib):
    """gate_scale = NULL: every row of logits has mean square mean/(mean + eps), i.e. 1
    up to eps and fp32 rounding."""
    m, n_exp, d = 4, 64, 512
    w = W.weight((n_exp, d), 91)
    xb, _ = W.activations((m, d), 92)
    logits = lib.router_logits(upload_oracle_weight(lib, F.quantize_matrix(w)), upload_bf16(xb), None, EPS)
    torch.cuda.synchronize()
    ms = np.mean(logits.cpu().numpy().astype(np.float64) ** 2, axis=1)
    assert np.all(np.abs(ms - 1.0) < 1e-4), ms
