"""Pins for the oracle's GEMM, router, grouping, expert FFN, MoE layer, lm_head and layout (CPU)."""

import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import formats as F
from oracle import gemm as G
from oracle import layout as L
from oracle import lm_head as LM
from oracle import moe as MO
from nvfp4_w4a16_moe_skinny_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _q(rng, n, k, std=0.02):
    return F.quantize_matrix((std * rng.standard_normal((n, k))).astype(np.float32))


# ------------------------------------------------------------------ GEMM

def test_gemm_matches_triple_loop():
    rng = np.random.default_rng(0)
    nib, sc, g = _q(rng, 24, 64)
    x = rng.standard_normal((3, 64))
    y, yb, ya = G.nvfp4_gemm(nib, sc, g, x)
    w = F.dequantize_matrix(nib, sc, g)
    for m in range(3):
        for n in range(24):
            s = 0.0
            a = 0.0
            for k in range(64):
                s += w[n, k] * x[m, k]
                a += abs(w[n, k] * x[m, k])
            assert math.isclose(y[m, n], s, rel_tol=1e-13, abs_tol=1e-15)
            assert math.isclose(ya[m, n], a, rel_tol=1e-13, abs_tol=1e-15)
    assert np.array_equal(yb, F.bf16_round(y))


def test_gemm_one_hot_picks_a_column():
    rng = np.random.default_rng(1)
    nib, sc, g = _q(rng, 40, 96)
    w = F.dequantize_matrix(nib, sc, g)
    for k in (0, 17, 95):
        x = np.zeros((1, 96))
        x[0, k] = 1.0
        y, _, _ = G.nvfp4_gemm(nib, sc, g, x)
        assert np.array_equal(y[0], w[:, k])


# ------------------------------------------------------------------ router / grouping

def test_route_topk_brute_force_and_ties():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((6, 128)).astype(np.float32)
    logits[0, 5] = logits[0, 9] = logits[0, 77] = 5.0          # planted three-way tie at the top
    logits[1, :] = 0.0                                          # all equal: ids 0..7
    ids, probs = MO.route_topk(logits, 8)
    for m in range(6):
        brute = sorted(range(128), key=lambda e: (-float(logits[m, e]), e))[:8]
        assert ids[m].tolist() == brute
    assert ids[0, :3].tolist() == [5, 9, 77]
    assert ids[1].tolist() == list(range(8))
    assert np.allclose(probs.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    # softmax over the chosen 8 equals the renormalised slice of the full softmax
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, ids.astype(np.int64), axis=1)
    assert np.allclose(probs, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=0)
    assert np.all(np.diff(probs, axis=1) <= 0)


def test_route_weight_options_closed_forms():
    """softmax_all: with logits ln 1 .. ln 4 the softmax over all four experts is
    1/10 .. 4/10, so the top-2 weights are 0.4 and 0.3 (not renormalised); the
    default renormalises the chosen two to 4/7 and 3/7; an expert scale multiplies
    the weight of its expert only; with top_k = E both readings coincide."""
    logits = np.log(np.array([[1.0, 2.0, 3.0, 4.0]]))
    ids, p_all = MO.route_topk(logits, 2, softmax_all=True)
    assert ids.tolist() == [[3, 2]]
    assert np.allclose(p_all, [[0.4, 0.3]], rtol=1e-14)
    _, p_renorm = MO.route_topk(logits, 2)
    assert np.allclose(p_renorm, [[4 / 7, 3 / 7]], rtol=1e-14)
    _, p_scaled = MO.route_topk(logits, 2, softmax_all=True, expert_scale=[1.0, 1.0, 0.5, 2.0])
    assert np.allclose(p_scaled, [[0.8, 0.15]], rtol=1e-14)
    rng = np.random.default_rng(9)
    l = rng.standard_normal((5, 6))
    assert np.allclose(MO.route_topk(l, 6, softmax_all=True)[1], MO.route_topk(l, 6)[1], rtol=1e-12)


def test_route_nan_and_neginf_logits():
    """A NaN logit counts as -inf: -inf experts are chosen after every finite one, lowest
    id first (brute force over (value, id) with NaN read as -inf), each id is valid and
    distinct, their weights are 0 (exp(-inf) = 0), and a token whose logits are all -inf
    or NaN gets weight 0 on every slot (both weight readings)."""
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((4, 16))
    logits[0, [2, 7]] = np.nan
    logits[1, 3:] = -np.inf                       # three finite, then the rest -inf
    logits[2, :] = np.nan
    logits[3, ::2] = -np.inf
    logits[3, 1::4] = np.nan
    for softmax_all in (False, True):
        ids, probs = MO.route_topk(logits, 6, softmax_all)
        for m in range(4):
            key = np.where(np.isnan(logits[m]), -np.inf, logits[m])
            brute = sorted(range(16), key=lambda e: (-key[e], e))[:6]
            assert ids[m].tolist() == brute
            assert len(set(ids[m].tolist())) == 6
            fin = np.isfinite(key[ids[m]])
            assert np.all(probs[m][~fin] == 0.0)
        assert ids[1, 3:].tolist() == [3, 4, 5]
        assert ids[2].tolist() == [0, 1, 2, 3, 4, 5] and np.all(probs[2] == 0.0)
        # row 1: every finite logit is chosen, so both readings sum to 1
        assert np.isclose(probs[1].sum(), 1.0, rtol=0, atol=1e-15)


def test_grouping_brute_force():
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(16, 4, replace=False) for _ in range(9)]).astype(np.int32)
    counts, offsets, pairs = MO.group_by_expert(ids, 16)
    flat = ids.reshape(-1)
    for e in range(16):
        brute = [p for p in range(flat.size) if flat[p] == e]
        assert pairs[offsets[e]:offsets[e + 1]].tolist() == brute
        assert counts[e] == len(brute)
    assert offsets[0] == 0 and offsets[-1] == flat.size


def test_gelu_tanh_identities():
    z = np.linspace(-12, 12, 4001)
    gz = MO.gelu_tanh(z)
    assert MO.gelu_tanh(0.0) == 0.0
    assert np.allclose(gz - MO.gelu_tanh(-z), z, rtol=0, atol=1e-12)
    # 0.5 (1 + tanh u) = sigmoid(2u): an independent evaluation through scipy's expit
    u = math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)
    assert np.allclose(gz, z * scipy.special.expit(2 * u), rtol=1e-13, atol=1e-15)
    assert np.allclose(MO.gelu_tanh(np.array([30.0, -30.0])), [30.0, 0.0], atol=1e-12)


# ------------------------------------------------------------------ expert FFN / MoE layer

def _brute_expert(wgu, wd, x):
    inter = wgu.shape[0] // 2
    d = wd.shape[0]
    out = np.zeros(d)
    h = np.zeros(inter)
    for i in range(inter):
        gsum = sum(wgu[i, j] * x[j] for j in range(x.size))
        usum = sum(wgu[inter + i, j] * x[j] for j in range(x.size))
        zz = gsum
        gel = zz * scipy.special.expit(2 * math.sqrt(2 / math.pi) * (zz + 0.044715 * zz ** 3))
        h[i] = float(F.bf16_round(gel * usum))
    for r in range(d):
        out[r] = sum(wd[r, i] * h[i] for i in range(inter))
    return out


def test_moe_layer_reduces_to_single_expert():
    """One dominant logit makes p one-hot (exp(-1000) == 0 in float64); with the shared
    expert absent the layer is exactly one expert FFN, checked by brute force."""
    rng = np.random.default_rng(4)
    e_cnt, d, inter, m = 6, 32, 16, 3
    gu = [_q(rng, 2 * inter, d, 0.5) for _ in range(e_cnt)]
    dn = [_q(rng, d, inter, 0.5) for _ in range(e_cnt)]
    gate_up = (np.stack([q[0] for q in gu]), np.stack([q[1] for q in gu]), np.array([q[2] for q in gu]))
    down = (np.stack([q[0] for q in dn]), np.stack([q[1] for q in dn]), np.array([q[2] for q in dn]))
    x = W.bf16_bits_to_f32(W.to_bf16_bits(rng.standard_normal((m, d)).astype(np.float32))).astype(np.float64)
    logits = rng.standard_normal((m, e_cnt)).astype(np.float32)
    winners = [2, 5, 0]
    for t, e in enumerate(winners):
        logits[t, e] = 1000.0
    res = MO.moe_layer(x, logits, 3, gate_up, down)
    for t, e in enumerate(winners):
        assert res["ids"][t, 0] == e and res["probs"][t, 0] == 1.0
        wgu = F.dequantize_matrix(gate_up[0][e], gate_up[1][e], gate_up[2][e])
        wd = F.dequantize_matrix(down[0][e], down[1][e], down[2][e])
        ref = _brute_expert(wgu, wd, x[t])
        assert np.allclose(res["out"][t], ref, rtol=1e-12, atol=1e-12)


def test_moe_shared_expert_adds_with_weight_one():
    rng = np.random.default_rng(8)
    e_cnt, d, inter, m = 4, 32, 16, 2
    gu = [_q(rng, 2 * inter, d, 0.5) for _ in range(e_cnt)]
    dn = [_q(rng, d, inter, 0.5) for _ in range(e_cnt)]
    gate_up = (np.stack([q[0] for q in gu]), np.stack([q[1] for q in gu]), np.array([q[2] for q in gu]))
    down = (np.stack([q[0] for q in dn]), np.stack([q[1] for q in dn]), np.array([q[2] for q in dn]))
    sgu, sdn = _q(rng, 2 * inter, d, 0.5), _q(rng, d, inter, 0.5)
    x = rng.standard_normal((m, d))
    logits = rng.standard_normal((m, e_cnt)).astype(np.float32)
    a = MO.moe_layer(x, logits, 2, gate_up, down)
    b = MO.moe_layer(x, logits, 2, gate_up, down, sgu, sdn)
    ref = np.stack([_brute_expert(F.dequantize_matrix(*sgu), F.dequantize_matrix(*sdn), x[t]) for t in range(m)])
    assert np.allclose(b["out"] - a["out"], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ lm_head

def test_lm_head_argmax_brute_force_planted_max_and_ties():
    rng = np.random.default_rng(6)
    vocab, d, m = 300, 64, 3
    w = (0.02 * rng.standard_normal((vocab, d))).astype(np.float32)
    w[123] = w[200] = 0.5 * np.sign(rng.standard_normal(d)).astype(np.float32)   # identical rows
    nib, sc, g = F.quantize_matrix(w)
    x = rng.standard_normal((m, d))
    x[0] = F.dequantize_matrix(nib, sc, g)[123]        # token 0 aligns with the planted rows
    res = LM.lm_head_argmax(nib, sc, g, x, chunk_rows=64)
    wh = F.dequantize_matrix(nib, sc, g)
    full = x @ wh.T
    for t in range(m):
        order = sorted(range(vocab), key=lambda n: (-full[t, n], n))
        assert res["argmax"][t] == order[0]
        assert res["max"][t] == full[t, order[0]]
        assert res["second"][t] == full[t, order[1]]
    assert res["argmax"][0] == 123                      # tie with row 200 goes to the lower index


# ------------------------------------------------------------------ layout

def test_layout_round_trip_and_padding():
    rng = np.random.default_rng(7)
    for (n, k, gated) in [(16, 64, False), (40, 80, False), (64, 128, True), (128, 16, True), (200, 320, False)]:
        nib = rng.integers(0, 256, (2, n, k // 2), dtype=np.uint8)
        sc = rng.integers(0, 127, (2, n, k // 16), dtype=np.uint8)
        buf = L.repack(nib, sc, gated)
        assert buf.size == L.repacked_bytes(n, k, 2)
        nib2, sc2 = L.unrepack(buf, n, k, 2, gated)
        assert np.array_equal(nib, nib2) and np.array_equal(sc, sc2)
        used = np.zeros(buf.size, bool)
        per = L.repacked_bytes(n, k, 1)
        kcc = L.padded_dims(n, k)[1] // 64
        dest = L.row_permutation(n, gated)
        for e in range(2):
            used[e * per + L.nibble_byte_offset(np.repeat(dest, k // 2), np.tile(np.arange(k // 2), n), kcc)] = True
            used[e * per + L.scale_byte_offset(np.repeat(dest, k // 16), np.tile(np.arange(k // 16), n), kcc)] = True
        assert not buf[~used].any()                     # padding is zero
        assert used.sum() == 2 * (n * k // 2 + n * k // 16)   # the mapping is injective


def test_layout_hand_checked_positions():
    """Byte positions worked out by hand from the layout specification (version 2)."""
    # tile (group 0, chunk 0, block 0): lane 0 word 0 = (row0,c0-1), (row8,c0-1), (row0,c8-9), (row8,c8-9)
    assert L.nibble_byte_offset(0, 0, 2) == 0
    assert L.nibble_byte_offset(8, 0, 2) == 1
    assert L.nibble_byte_offset(0, 4, 2) == 2
    assert L.nibble_byte_offset(8, 4, 2) == 3
    # lane 1 (g=0, t=1) starts at byte 16 with columns 2-3
    assert L.nibble_byte_offset(0, 1, 2) == 16
    # k-tile 1 (columns 16..31) of lane 0 is the next word
    assert L.nibble_byte_offset(0, 8, 2) == 4
    # row 1 is g = 1 -> lane 4 -> byte 64
    assert L.nibble_byte_offset(1, 0, 2) == 64
    # rows 16..31 are block 1 of group 0: the next tile of the same chunk
    assert L.nibble_byte_offset(16, 0, 2) == 576
    assert L.nibble_byte_offset(48, 0, 2) == 3 * 576
    # columns 64..127 are chunk 1: after the 4 tiles of chunk 0
    assert L.nibble_byte_offset(0, 32, 2) == 4 * 576
    # rows 64.. are group 1: after both chunks (2 x 4 tiles) of group 0
    assert L.nibble_byte_offset(64, 0, 2) == 8 * 576
    # scales: row 0 group 0 at 512, row 8 group 0 at 513, row 0 group 1 at 514, row 1 at 520
    assert [int(L.scale_byte_offset(r, gg, 2)) for r, gg in [(0, 0), (8, 0), (0, 1), (1, 0), (0, 4), (16, 0)]] == \
        [512, 513, 514, 520, 4 * 576 + 512, 576 + 512]
    # gated: gate row 9 -> block 1 row 1; up row 9 -> block 1 row 9
    perm = L.row_permutation(32, True)
    assert perm[9] == 17 and perm[16 + 9] == 25 and perm[0] == 0 and perm[16] == 8
    assert L.repacked_bytes(40, 80) == 4 * 2 * 576        # 40 rows pad to one 64-row group; 80 cols to 2 chunks


# ------------------------------------------------------------------ shapes printed on the pages

def test_model_constants_match_pages():
    vals = {}
    for line in open(os.path.join(GOLDEN, "model_constants.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            key, v = line.split()
            vals[key] = int(v)
    assert W.HIDDEN == vals["hidden"]
    assert W.N_EXPERTS == vals["n_experts"]
    assert W.TOP_K == vals["top_k"]
    assert W.VOCAB == vals["vocab"]
    assert 15 in W.DECODE_M and 15 == vals["draft_tokens"] + 1
    assert L.TILE_COLS % vals["scale_group"] == 0
