"""GPU parity: MoE router (top-k, softmax, grouping) and the grouped NVFP4 expert FFN vs the oracle."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as OM
from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
from tests.gpu_helpers import bf16_to_f64, check_bound, dev, upload_bf16, upload_f32

pytestmark = pytest.mark.gpu

PROB_TOL = 4e-6   # fp32 softmax over <= 32 terms vs float64: a few ulps of 1


def _route(lib, logits, top_k):
    ids, probs, offsets, pairs = lib.route_topk(upload_f32(logits), top_k)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), probs.cpu().numpy(), offsets.cpu().numpy(), pairs.cpu().numpy()


@pytest.mark.parametrize("m,e,k", [(1, 128, 8), (15, 128, 8), (16, 128, 8), (512, 128, 8), (37, 64, 4),
                                   (3, 1024, 32), (100, 40, 1)])
def test_route_topk_bit_exact(lib, m, e, k):
    logits = W.normal_f32((m, e), W.seed_of("route-test", m, e, k))
    ids, probs, offsets, pairs = _route(lib, logits, k)
    oids, oprobs = OM.route_topk(logits, k)
    counts, ooffsets, opairs = OM.group_by_expert(oids, e)
    assert np.array_equal(ids, oids)
    assert np.array_equal(offsets, ooffsets)
    assert np.array_equal(pairs, opairs)
    assert np.max(np.abs(probs - oprobs)) <= PROB_TOL


@pytest.mark.parametrize("m,e,k,softmax_all,scaled", [(1, 128, 8, True, False), (15, 128, 8, True, True),
                                                       (15, 128, 8, False, True), (100, 40, 3, True, True),
                                                       (512, 128, 8, True, True)])
def test_route_weight_options(lib, m, e, k, softmax_all, scaled):
    """The softmax over all experts (not renormalised) and a per-expert scale folded
    into the weights: ids and grouping unchanged and bit-exact, weights as the oracle's
    (one CTA for m <= 32, the split router above)."""
    logits = W.normal_f32((m, e), W.seed_of("route-opt", m, e, k))
    scale = (0.5 + np.abs(W.normal_f32((e,), W.seed_of("route-scale", e)))).astype(np.float32) if scaled else None
    ids, probs, offsets, pairs = lib.route_topk(upload_f32(logits), k, softmax_all=softmax_all,
                                                expert_scale=upload_f32(scale) if scaled else None)
    torch.cuda.synchronize()
    oids, oprobs = OM.route_topk(logits, k, softmax_all, scale)
    _, ooffsets, opairs = OM.group_by_expert(oids, e)
    assert np.array_equal(ids.cpu().numpy(), oids)
    assert np.array_equal(offsets.cpu().numpy(), ooffsets)
    assert np.array_equal(pairs.cpu().numpy(), opairs)
    # fp32 exp and a sum over up to 128 terms against float64: a few 1e-6 relative
    assert np.max(np.abs(probs.cpu().numpy() - oprobs) / np.maximum(oprobs, 1e-30)) <= 2e-5


def test_moe_layer_with_weight_options(lib):
    """The whole layer on routing weights from the variants: softmax over all experts
    and per-expert scales, for a decode batch and a prefill chunk."""
    scale = (0.5 + np.abs(W.normal_f32((8,), 77))).astype(np.float32)
    for m in (5, 40):
        got, ref, _ = _moe_case(lib, m, 128, 64, 8, 3, True, "moe-small", softmax_all=True, expert_scale=scale)
        check_bound(got, ref["out"], ref["tol_scale"], True, f"moe weight options m={m}")
    assert lib.device_error() == 0


def test_route_ties_go_to_lower_id(lib):
    logits = np.zeros((4, 128), np.float32)
    logits[0, [3, 77, 9, 100]] = 2.0          # four-way tie at the top
    logits[1, :] = -1.0                        # everything tied
    logits[2, ::2] = 1.0
    logits[3] = W.normal_f32((128,), 5)
    logits[3, 50] = logits[3, 60] = logits[3].max() + 1
    ids, probs, offsets, pairs = _route(lib, logits, 8)
    oids, _ = OM.route_topk(logits, 8)
    assert np.array_equal(ids, oids)
    assert ids[0, :4].tolist() == [3, 9, 77, 100]
    assert ids[1].tolist() == list(range(8))
    assert ids[3, :2].tolist() == [50, 60]


def _stack_q(mats):
    qs = [F.quantize_matrix(w) for w in mats]
    return np.stack([q[0] for q in qs]), np.stack([q[1] for q in qs]), np.array([q[2] for q in qs], np.float32)


_EXPERTS = {}


def _experts(lib, case, shared):
    """Host fp32 expert stacks and their GPU-prepared weights, cached per shape (the
    weights do not depend on m)."""
    key = (case.d, case.inter, case.n_experts, case.tag, shared)
    if key not in _EXPERTS:
        _EXPERTS.clear()
        gu = np.stack([case.gate_up(e) for e in range(case.n_experts)])
        dn = np.stack([case.down(e) for e in range(case.n_experts)])
        wgu = lib.prepare(upload_f32(gu), gated=True)
        wdn = lib.prepare(upload_f32(dn))
        sgu = sdn = None
        if shared:
            sgu = lib.prepare(upload_f32(case.gate_up(-1)), gated=True)
            sdn = lib.prepare(upload_f32(case.down(-1)))
        _EXPERTS[key] = (gu, dn, wgu, wdn, sgu, sdn)
    return _EXPERTS[key]


def _moe_case(lib, m, d, inter, n_exp, top_k, shared, tag, logits=None, rows=None, softmax_all=False,
              expert_scale=None):
    """Run the layer on the GPU for all m tokens; the oracle computes the tokens in
    `rows` (all by default) -- a token's output depends on its own x and logits only."""
    case = W.MoECase(m=m, d=d, inter=inter, n_experts=n_exp, top_k=top_k, tag=tag)
    gu, dn, wgu, wdn, sgu, sdn = _experts(lib, case, shared)
    xb, xf = case.x()
    if logits is None:
        logits = case.logits()
    x = upload_bf16(xb)
    scale_dev = upload_f32(expert_scale) if expert_scale is not None else None
    ids, probs, offsets, pairs = lib.route_topk(upload_f32(logits), top_k, softmax_all=softmax_all,
                                                expert_scale=scale_dev)
    out = lib.moe_ffn(x, top_k, probs, offsets, pairs, wgu, wdn, sgu, sdn)
    torch.cuda.synchronize()
    got = bf16_to_f64(out)
    if rows is not None:
        rows = np.asarray(rows)
        xf, logits, got = xf[rows], logits[rows], got[rows]
    # oracle: quantize only the experts the (sampled) routing uses, plus the shared one
    oids, _ = OM.route_topk(logits, top_k)
    used = sorted(set(oids.reshape(-1).tolist()))  # (the options change the weights, not the ids)
    gq = [None] * n_exp
    dq = [None] * n_exp
    for e in used:
        gq[e] = F.quantize_matrix(gu[e])
        dq[e] = F.quantize_matrix(dn[e])
    zero_g = (np.zeros_like(gq[used[0]][0]), np.zeros_like(gq[used[0]][1]), np.float32(0))
    zero_d = (np.zeros_like(dq[used[0]][0]), np.zeros_like(dq[used[0]][1]), np.float32(0))
    gq = [q if q is not None else zero_g for q in gq]
    dq = [q if q is not None else zero_d for q in dq]
    gate_up = (np.stack([q[0] for q in gq]), np.stack([q[1] for q in gq]), np.array([q[2] for q in gq]))
    down = (np.stack([q[0] for q in dq]), np.stack([q[1] for q in dq]), np.array([q[2] for q in dq]))
    sh_gu = F.quantize_matrix(case.gate_up(-1)) if shared else None
    sh_dn = F.quantize_matrix(case.down(-1)) if shared else None
    ref = OM.moe_layer(xf.astype(np.float64), logits, top_k, gate_up, down, sh_gu, sh_dn, softmax_all, expert_scale)
    return got, ref, (ids, offsets, pairs)


@pytest.mark.parametrize("m", [1, 2, 5, 8, 9, 15, 16, 17, 33, 64, 100])
@pytest.mark.parametrize("shared", [True, False])
def test_moe_small(lib, m, shared):
    """m <= 16: one segment per expert; m > 16 (prefill): each expert's pairs in
    blocks of 32, the last one ragged, and the shared expert in blocks of 32 tokens."""
    got, ref, (ids, offsets, pairs) = _moe_case(lib, m, 128, 64, 8, 3, shared, "moe-small")
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    check_bound(got, ref["out"], ref["tol_scale"], True, f"moe small m={m} shared={shared}")


def test_moe_ragged_and_concentrated(lib):
    """Every token routed to the same two experts: the largest per-expert token groups (16),
    with row-block counts (16 and 12) that do not divide the 16 warps of a CTA."""
    m, n_exp, top_k = 16, 6, 2
    logits = np.full((m, n_exp), -5.0, np.float32)
    logits[:, 4] = 3.0
    logits[:, 1] = 2.0
    got, ref, _ = _moe_case(lib, m, 192, 128, n_exp, top_k, True, "moe-conc", logits=logits)
    assert ref["counts"][4] == m and ref["counts"][1] == m
    check_bound(got, ref["out"], ref["tol_scale"], True, "moe concentrated")


def test_moe_prefill_concentrated(lib):
    """Every one of 40 tokens routed to the same two experts: each gets blocks of 32
    and 8 pairs, and the shared expert blocks of 32 and 8 tokens."""
    m, n_exp, top_k = 40, 6, 2
    logits = np.full((m, n_exp), -5.0, np.float32)
    logits[:, 2] = 3.0
    logits[:, 5] = 2.0
    got, ref, _ = _moe_case(lib, m, 192, 128, n_exp, top_k, True, "moe-conc", logits=logits)
    assert ref["counts"][2] == m and ref["counts"][5] == m
    check_bound(got, ref["out"], ref["tol_scale"], True, "moe prefill concentrated")
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [1, 15])
def test_moe_config2_full_size(lib, m):
    got, ref, _ = _moe_case(lib, m, W.HIDDEN, W.INTER, W.N_EXPERTS, W.TOP_K, True, "moe")
    check_bound(got, ref["out"], ref["tol_scale"], True, f"moe config2 m={m}")
    assert lib.device_error() == 0


def test_moe_workspace_reused_across_shapes(lib):
    """One workspace serves calls of different m: a 15-token call fills h and the
    down outputs, then a 1-token call (which splits K and needs zeroed arrival
    counters) and a 15-token call again must still match the oracle."""
    _moe_case(lib, 15, W.HIDDEN, W.INTER, W.N_EXPERTS, W.TOP_K, True, "moe")
    for m in (1, 15):
        got, ref, _ = _moe_case(lib, m, W.HIDDEN, W.INTER, W.N_EXPERTS, W.TOP_K, True, "moe")
        check_bound(got, ref["out"], ref["tol_scale"], True, f"moe reused workspace m={m}")
    assert lib.device_error() == 0


def test_moe_prefill_config4_full_size(lib):
    """The M=512 prefill chunk through the full-size layer: all 512 tokens run on the
    GPU; the oracle checks a sample of tokens spread over the chunk (first, last and
    seeded picks, so that their pairs fall in first, middle and ragged last blocks)."""
    m = 512
    rng = np.random.default_rng(W.seed_of("prefill-sample", m))
    rows = sorted(set([0, 1, m // 2, m - 1] + rng.choice(m, 4, replace=False).tolist()))
    got, ref, (ids, offsets, pairs) = _moe_case(lib, m, W.HIDDEN, W.INTER, W.N_EXPERTS, W.TOP_K, True, "moe",
                                                rows=rows)
    check_bound(got, ref["out"], ref["tol_scale"], True, f"moe prefill m={m} rows={rows}")
    # the grouping is bit-exact for the whole chunk
    case = W.MoECase(m=m, d=W.HIDDEN, inter=W.INTER, n_experts=W.N_EXPERTS, top_k=W.TOP_K, tag="moe")
    oids, _ = OM.route_topk(case.logits(), W.TOP_K)
    counts, ooffsets, opairs = OM.group_by_expert(oids, W.N_EXPERTS)
    assert np.array_equal(offsets.cpu().numpy(), ooffsets)
    assert np.array_equal(pairs.cpu().numpy(), opairs)
    assert counts.max() > 16          # experts span several 16-pair blocks
    assert lib.device_error() == 0
