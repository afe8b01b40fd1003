"""GPU parity: MoE router (top-k, softmax, grouping) and the grouped NVFP4 expert FFN vs the oracle."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as OM
from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
from tests.gpu_helpers import (assert_gpu_quantizer_matches, bf16_to_f64, check_bound, dev, upload_bf16,
                               upload_f32, upload_oracle_weight)

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
        for forward in (False, True):
            got, ref, (ids, _, _) = _moe_case(lib, m, 128, 64, 8, 3, True, "moe-small", softmax_all=True,
                                              expert_scale=scale, forward=forward)
            assert np.array_equal(ids.cpu().numpy(), ref["ids"])
            check_bound(got, ref["out"], ref["tol_scale"], True, f"moe weight options m={m} forward={forward}")
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [4, 40])
def test_route_nan_and_neginf_logits(lib, m):
    """NaN logits count as -inf and -inf experts are chosen last, lowest id first: every
    id is a valid, distinct expert and the grouping stays a permutation of the pairs; a
    token whose logits are all NaN or -inf gets weight 0 (one-CTA and split routers)."""
    logits = W.normal_f32((m, 128), W.seed_of("route-nan", m))
    logits[0, [1, 5, 9]] = np.nan
    logits[1, 4:] = -np.inf
    logits[2, :] = np.nan
    logits[3, ::2] = -np.inf
    logits[3, 1::4] = np.nan
    for softmax_all in (False, True):
        ids, probs, offsets, pairs = lib.route_topk(upload_f32(logits), 8, softmax_all=softmax_all)
        torch.cuda.synchronize()
        oids, oprobs = OM.route_topk(logits, 8, softmax_all)
        _, ooffsets, opairs = OM.group_by_expert(oids, 128)
        assert np.array_equal(ids.cpu().numpy(), oids)
        assert np.array_equal(offsets.cpu().numpy(), ooffsets)
        assert np.array_equal(pairs.cpu().numpy(), opairs)
        p = probs.cpu().numpy()
        assert np.all(np.isfinite(p))
        assert np.all(p[oprobs == 0] == 0)
        assert np.max(np.abs(p - oprobs)) <= 2e-5


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


_EXPERTS = {}


def _experts(lib, case, shared):
    """The layer's weights quantized by the oracle (per-expert stacks and the shared
    expert), and the same bytes repacked on the GPU for the kernels; cached per shape
    (the weights do not depend on m).  The GPU quantizer is checked against the
    oracle's bytes on the expert stacks on the way."""
    key = (case.d, case.inter, case.n_experts, case.tag, shared)
    if key not in _EXPERTS:
        _EXPERTS.clear()
        gu = np.stack([case.gate_up(e) for e in range(case.n_experts)])
        dn = np.stack([case.down(e) for e in range(case.n_experts)])
        qgu, qdn = F.quantize_stack(gu), F.quantize_stack(dn)
        assert_gpu_quantizer_matches(lib, gu, qgu, f"gate_up stack {gu.shape}")
        assert_gpu_quantizer_matches(lib, dn, qdn, f"down stack {dn.shape}")
        del gu, dn
        wgu = upload_oracle_weight(lib, qgu, gated=True)
        wdn = upload_oracle_weight(lib, qdn)
        qsgu = qsdn = sgu = sdn = None
        if shared:
            qsgu, qsdn = F.quantize_matrix(case.gate_up(-1)), F.quantize_matrix(case.down(-1))
            sgu = upload_oracle_weight(lib, qsgu, gated=True)
            sdn = upload_oracle_weight(lib, qsdn)
        torch.cuda.synchronize()
        _EXPERTS[key] = (qgu, qdn, qsgu, qsdn, wgu, wdn, sgu, sdn)
    return _EXPERTS[key]


def _moe_case(lib, m, d, inter, n_exp, top_k, shared, tag, logits=None, rows=None, softmax_all=False,
              expert_scale=None, forward=False):
    """Run the layer on the GPU for all m tokens; the oracle computes the tokens in
    `rows` (all by default) -- a token's output depends on its own x and logits only.
    Kernels and oracle use the same (oracle-quantized) weight bytes.  forward: the
    one-call moe_forward instead of moe_route_topk_ex then moe_ffn_grouped."""
    case = W.MoECase(m=m, d=d, inter=inter, n_experts=n_exp, top_k=top_k, tag=tag)
    qgu, qdn, qsgu, qsdn, wgu, wdn, sgu, sdn = _experts(lib, case, shared)
    xb, xf = case.x()
    if logits is None:
        logits = case.logits()
    x = upload_bf16(xb)
    scale_dev = upload_f32(expert_scale) if expert_scale is not None else None
    if forward:
        out, (ids, probs, offsets, pairs) = lib.moe_forward(x, upload_f32(logits), top_k, wgu, wdn, sgu, sdn,
                                                            softmax_all=softmax_all, expert_scale=scale_dev)
    else:
        ids, probs, offsets, pairs = lib.route_topk(upload_f32(logits), top_k, softmax_all=softmax_all,
                                                    expert_scale=scale_dev)
        out = lib.moe_ffn(x, top_k, probs, offsets, pairs, wgu, wdn, sgu, sdn)
    torch.cuda.synchronize()
    got = bf16_to_f64(out)
    if rows is not None:
        rows = np.asarray(rows)
        xf, logits, got = xf[rows], logits[rows], got[rows]
    ref = OM.moe_layer(xf.astype(np.float64), logits, top_k, qgu, qdn, qsgu, qsdn, softmax_all, expert_scale)
    return got, ref, (ids, offsets, pairs)


@pytest.mark.parametrize("forward", [False, True])
@pytest.mark.parametrize("m", [1, 2, 5, 8, 9, 15, 16, 17, 33, 64, 100])
@pytest.mark.parametrize("shared", [True, False])
def test_moe_small(lib, m, shared, forward):
    """m <= 16: one segment per expert; m > 16 (prefill): each expert's pairs in
    blocks of 32, the last one ragged, and the shared expert in blocks of 32 tokens.
    Through moe_forward as well."""
    got, ref, (ids, offsets, pairs) = _moe_case(lib, m, 128, 64, 8, 3, shared, "moe-small", forward=forward)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(pairs.cpu().numpy(), ref["sorted_pairs"])
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


@pytest.mark.parametrize("m", [1, 15, 16])
def test_moe_forward_config2_full_size(lib, m):
    """The full-size layer through moe_forward: every output element against the
    oracle, the routing bit-exact."""
    got, ref, (ids, offsets, pairs) = _moe_case(lib, m, W.HIDDEN, W.INTER, W.N_EXPERTS, W.TOP_K, True, "moe",
                                                forward=True)
    check_bound(got, ref["out"], ref["tol_scale"], True, f"moe_forward config2 m={m}")
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(pairs.cpu().numpy(), ref["sorted_pairs"])
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
    """The M=512 prefill chunk through the full-size layer: every one of the 512 tokens
    is compared element by element with the oracle (which dequantizes each expert once
    and applies it to the tokens routed to it), and the grouping is bit-exact."""
    m = 512
    got, ref, (ids, offsets, pairs) = _moe_case(lib, m, W.HIDDEN, W.INTER, W.N_EXPERTS, W.TOP_K, True, "moe")
    assert got.shape == (m, W.HIDDEN)
    check_bound(got, ref["out"], ref["tol_scale"], True, f"moe prefill m={m}")
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(pairs.cpu().numpy(), ref["sorted_pairs"])
    assert ref["counts"].max() > 32   # experts span several 32-pair blocks, the last one ragged
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [1, 2, 4, 8, 15, 16, 40])
def test_moe_forward_equals_route_then_ffn(lib, m):
    """moe_forward (one call) gives the same bytes as moe_route_topk followed by
    moe_ffn_grouped, and the same routing, for decode batches and a prefill chunk."""
    mc = W.MoECase(m=m, d=256, inter=128, n_experts=16, top_k=4, tag="forward")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev())  # noqa: E731
    gu = lib.prepare(up(np.stack([mc.gate_up(e) for e in range(16)])), gated=True)
    dn = lib.prepare(up(np.stack([mc.down(e) for e in range(16)])))
    sgu, sdn = lib.prepare(up(mc.gate_up(-1)), gated=True), lib.prepare(up(mc.down(-1)))
    xb, _ = mc.x()
    x = upload_bf16(xb)
    logits = up(mc.logits())
    ids, probs, offs, pairs = lib.route_topk(logits, 4)
    ref = lib.moe_ffn(x, 4, probs, offs, pairs, gu, dn, sgu, sdn).clone()
    out, (ids2, probs2, offs2, pairs2) = lib.moe_forward(x, logits, 4, gu, dn, sgu, sdn)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2) and torch.equal(probs, probs2) and torch.equal(offs, offs2)
    assert torch.equal(pairs, pairs2)
    assert torch.equal(out, ref)
    assert lib.device_error() == 0


def test_moe_forward_special_logits_and_options(lib):
    """moe_forward on NaN / -inf logits (a NaN counts as -inf; an all-NaN token gets
    weight 0) and with the softmax over all experts and per-expert scales: the same
    routing and bytes as moe_route_topk_ex followed by moe_ffn_grouped."""
    m, e, k = 6, 16, 4
    mc = W.MoECase(m=m, d=256, inter=128, n_experts=e, top_k=k, tag="forward-special")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev())  # noqa: E731
    gu = lib.prepare(up(np.stack([mc.gate_up(i) for i in range(e)])), gated=True)
    dn = lib.prepare(up(np.stack([mc.down(i) for i in range(e)])))
    xb, _ = mc.x()
    x = upload_bf16(xb)
    lg = mc.logits().copy()
    lg[0, [1, 5, 9]] = np.nan
    lg[1, 3:] = -np.inf
    lg[2, :] = np.nan
    lg[3, ::2] = -np.inf
    logits = up(lg)
    scale = up(0.5 + np.abs(W.normal_f32((e,), 91)))
    for softmax_all, es in ((False, None), (True, None), (False, scale), (True, scale)):
        ids, probs, offs, pairs = lib.route_topk(logits, k, softmax_all=softmax_all, expert_scale=es)
        ref = lib.moe_ffn(x, k, probs, offs, pairs, gu, dn).clone()
        out, (ids2, probs2, offs2, pairs2) = lib.moe_forward(x, logits, k, gu, dn, softmax_all=softmax_all,
                                                             expert_scale=es)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids2) and torch.equal(offs, offs2) and torch.equal(pairs, pairs2)
        assert torch.equal(probs, probs2)
        assert torch.equal(out, ref)
    assert lib.device_error() == 0


@pytest.mark.parametrize("m,n_exp,top_k,d,inter", [(16, 1024, 32, 128, 64), (1, 1024, 32, 256, 128),
                                                   (16, 512, 16, 128, 64)])
@pytest.mark.parametrize("forward", [False, True])
def test_moe_many_experts(lib, m, n_exp, top_k, d, inter, forward):
    """Decode batches routed over many experts: up to 512 pairs over 1,024 experts (513
    segments with the shared expert, several per CTA), top-32 routing with the widest
    router instance, against the oracle element by element and the grouping bit-exact."""
    got, ref, (ids, offsets, pairs) = _moe_case(lib, m, d, inter, n_exp, top_k, True, "moe-many", forward=forward)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(pairs.cpu().numpy(), ref["sorted_pairs"])
    assert (np.diff(ref["offsets"]) > 0).sum() > min(n_exp, m * top_k) // 2  # many active experts
    check_bound(got, ref["out"], ref["tol_scale"], True, f"moe many experts m={m} e={n_exp} k={top_k}")
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [1, 5, 16, 40])
@pytest.mark.parametrize("forward", [False, True])
def test_moe_odd_chunk_counts(lib, m, forward):
    """Odd chunk and group counts (the MoE calls take d and I in multiples of 64):
    d = 320 (five 64-column chunks for gate+up, five 64-row groups for down) and
    I = 192 (three chunks for down, six gated groups), decode batches and a prefill
    chunk."""
    got, ref, (ids, offsets, pairs) = _moe_case(lib, m, 320, 192, 8, 3, True, "moe-odd", forward=forward)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    check_bound(got, ref["out"], ref["tol_scale"], True, f"moe odd chunk counts m={m}")
    assert lib.device_error() == 0


@pytest.mark.parametrize("m,top_k,n_exp", [(2048, 8, 128), (4096, 4, 128), (4096, 4, 16)])
def test_moe_prefill_max_pairs(lib, m, top_k, n_exp):
    """Prefill chunks at the calls' limit of 16,384 (token, slot) pairs, over 128 experts
    (about 128 pairs each) and over 16 (about 1,024 each, 32 blocks per expert): every
    token against the oracle, the grouping bit-exact."""
    got, ref, (ids, offsets, pairs) = _moe_case(lib, m, 128, 64, n_exp, top_k, True, "moe-max")
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(pairs.cpu().numpy(), ref["sorted_pairs"])
    check_bound(got, ref["out"], ref["tol_scale"], True, f"moe prefill max pairs m={m} k={top_k} e={n_exp}")
    assert lib.device_error() == 0
