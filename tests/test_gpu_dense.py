"""GPU parity: quantizer, repack, dense skinny GEMM and lm_head argmax vs the FP64 oracle.

All compute runs through the C ABI (libnvfp4skinny.so); the oracle runs on the host.
"""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as OG
from oracle import layout as OL
from oracle import lm_head as OLM
from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
from tests.gpu_helpers import (assert_gpu_quantizer_matches, bf16_to_f64, check_bound, dev, oracle_quantize,
                               upload_bf16, upload_f32, upload_oracle_weight)
from tests.test_oracle_formats import _near_midpoint_matrix

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ quantizer
# The GPU quantizer and the oracle both decide every code as the round-to-nearest-even
# code of the exact quotient (bmax / (6 g) for a scale, w / (e4m3(s) g) for an
# element); the oracle is pinned to a brute force over exact rationals.

@pytest.mark.parametrize("n,k,seed", [(512, 256, 0), (40, 80, 1), (33, 16, 2), (16, 1024, 3)])
def test_quantizer_bit_exact(lib, n, k, seed):
    w = W.weight((n, k), seed) if seed else W.DenseCase.tiny().w()
    nib, sc, g = lib.quantize(upload_f32(w))
    onib, osc, og = F.quantize_matrix(w)
    assert g.item() == float(og)
    assert np.array_equal(sc.cpu().numpy(), osc)
    assert np.array_equal(nib.cpu().numpy(), onib)


def test_quantizer_special_values(lib):
    """Zero and underflowing blocks, sign of zero, and exact E2M1 ties: with amax =
    2688 * 2^-10 the global scale is exactly 2^-10 and a block whose maximum is
    6 * 2^-10 gets scale 1, so w / (scale * g) hits the rounding midpoints exactly."""
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((32, 64)) * 0.1).astype(np.float32)
    w[2, 0] = 2688.0 * 2.0 ** -10                    # global max -> g = 2^-10
    w[0, :16] = 0.0                                  # zero block
    w[1, 16:32] = 1e-12                              # block below the scale range
    w[3, :] = -w[3, :]
    w[4, 5] = -1e-9                                  # -tiny next to large values: code 8
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    w[5, :16] = np.concatenate([ties, -ties]) * np.float32(2.0 ** -10)
    nib, sc, g = lib.quantize(upload_f32(w))
    onib, osc, og = F.quantize_matrix(w)
    assert g.item() == float(og)
    assert np.array_equal(sc.cpu().numpy(), osc)
    assert np.array_equal(nib.cpu().numpy(), onib)
    z_nib, z_sc, z_g = lib.quantize(torch.zeros((16, 32), device=dev()))
    assert z_g.item() == 0.0 and not z_nib.any().item() and not z_sc.any().item()


def test_quantizer_near_midpoints(lib):
    """Block maxima and elements on, and one fp32 step either side of, the exact rounding
    midpoints under a global scale with a full 24-bit significand: the GPU codes are the
    exact quotients' codes (IEEE fp32 quotients would pick other codes for some)."""
    w = _near_midpoint_matrix()
    nib, sc, g = lib.quantize(upload_f32(w))
    onib, osc, og = F.quantize_matrix(w)
    assert g.item() == float(og)
    assert np.array_equal(sc.cpu().numpy(), osc)
    assert np.array_equal(nib.cpu().numpy(), onib)


def test_quantizer_stacked(lib):
    w = np.stack([W.weight((32, 128), 100 + e) * (e + 1) for e in range(3)])
    nib, sc, g = lib.quantize(upload_f32(w))
    for e in range(3):
        onib, osc, og = F.quantize_matrix(w[e])
        assert g[e].item() == float(og)
        assert np.array_equal(sc[e].cpu().numpy(), osc)
        assert np.array_equal(nib[e].cpu().numpy(), onib)


# ------------------------------------------------------------------ repack

@pytest.mark.parametrize("e,n,k,gated", [(1, 16, 64, False), (2, 40, 80, False), (1, 1000, 320, False),
                                         (3, 64, 128, True), (2, 128, 16, True), (1, 1408, 2816, True)])
def test_repack_bytes_bit_exact(lib, e, n, k, gated):
    rng = np.random.default_rng(n * 7 + k)
    nib = rng.integers(0, 256, (e, n, k // 2), dtype=np.uint8)
    sc = rng.integers(0, 127, (e, n, k // 16), dtype=np.uint8)
    wt = lib.repack(torch.from_numpy(nib).to(dev()), torch.from_numpy(sc).to(dev()),
                    torch.ones(e, device=dev()), gated=gated)
    assert wt.data.numel() == OL.repacked_bytes(n, k, e)
    assert np.array_equal(wt.data.cpu().numpy(), OL.repack(nib, sc, gated))


def test_device_and_host_repack_agree(lib):
    """The device repack and the host repack give the same bytes on a stacked gated
    weight with negative scales."""
    rng = np.random.default_rng(17)
    e, n, k = 3, 256, 704
    nib = rng.integers(0, 256, (e, n, k // 2), dtype=np.uint8)
    sc = rng.integers(0, 256, (e, n, k // 16), dtype=np.uint8)
    wt = lib.repack(torch.from_numpy(nib).to(dev()), torch.from_numpy(sc).to(dev()), torch.ones(e, device=dev()),
                    gated=True)
    assert np.array_equal(wt.data.cpu().numpy(), lib.repack_host(nib, sc, gated=True))


def test_repack_folds_negative_scales(lib):
    rng = np.random.default_rng(5)
    n, k = 32, 64
    nib = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    sc = rng.integers(1, 127, (n, k // 16), dtype=np.uint8)
    sc[::3, 1] |= 0x80                                   # some negative scales
    wt = lib.repack(torch.from_numpy(nib).to(dev()), torch.from_numpy(sc).to(dev()), torch.ones(1, device=dev()))
    nib2, sc2 = OL.unrepack(wt.data.cpu().numpy(), n, k)
    assert not (sc2 & 0x80).any()
    assert np.array_equal(F.dequantize_matrix(nib2[0], sc2[0], 1.0), F.dequantize_matrix(nib, sc, 1.0))


# ------------------------------------------------------------------ dense GEMM

def _dense(lib, m, n, k, w_seed, x_seed):
    w = W.weight((n, k), w_seed)
    xb, _ = W.activations((m, k), x_seed)
    nib, sc, g = F.quantize_matrix(w)
    wt = upload_oracle_weight(lib, (nib, sc, g))
    y = lib.gemm(wt, upload_bf16(xb))
    torch.cuda.synchronize()
    exact, _, absy = OG.nvfp4_gemm(nib, sc, g, W.bf16_bits_to_f32(xb).astype(np.float64))
    return bf16_to_f64(y), exact, absy


def test_tiny_gemm_config0(lib):
    """The 512 x 256 matrix quantized by the oracle; the kernel reads the oracle's bytes."""
    case = W.DenseCase.tiny()
    w = case.w()
    xb, xf = case.x()
    nib, sc, g = F.quantize_matrix(w)
    wt = upload_oracle_weight(lib, (nib, sc, g))
    y = lib.gemm(wt, upload_bf16(xb))
    torch.cuda.synchronize()
    exact, _, absy = OG.nvfp4_gemm(nib, sc, g, xf.astype(np.float64))
    check_bound(bf16_to_f64(y), exact, absy, True, "tiny gemm")
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", list(range(1, 17)))
@pytest.mark.parametrize("n,k", [(40, 80), (1000, 320), (272, 1088)])
def test_gemm_ragged_all_m(lib, m, n, k):
    got, exact, absy = _dense(lib, m, n, k, 1000 + n + k, 2000 + m)
    check_bound(got, exact, absy, True, f"gemm m={m} n={n} k={k}")


@pytest.mark.parametrize("m,n,k", [(1, 512, 16384), (16, 512, 16384), (7, 1000, 12288), (3, 136, 32768)])
def test_gemm_long_k(lib, m, n, k):
    """Long rows: the planner splits K 10-16 ways (five rounds of partials per tile at
    M=16), a 32,768-column row at M=3, a ragged N at M=7."""
    got, exact, absy = _dense(lib, m, n, k, 3000 + n + k, 4000 + m)
    check_bound(got, exact, absy, True, f"gemm long k m={m} n={n} k={k}")
    assert lib.device_error() == 0


def _wide_range_case(m, n, k, small_exp, big_cols_weight):
    """x rows with 2^10 at every 64th column and +-2^small_exp * (1 + j/128) elsewhere;
    the weight's columns under the large values are zero unless big_cols_weight."""
    rng = np.random.default_rng(77)
    w = W.weight((n, k), 4242)
    big = np.arange(k) % 64 == 0
    if not big_cols_weight:
        w[:, big] = 0.0
    frac = rng.integers(0, 128, size=(m, k)) / 128.0
    sign = np.where(rng.random((m, k)) < 0.5, -1.0, 1.0)
    x = (sign * (1.0 + frac) * 2.0 ** small_exp).astype(np.float32)
    x[:, big] = 2.0 ** 10
    xb = W.to_bf16_bits(x)
    assert np.array_equal(W.bf16_bits_to_f32(xb), x)      # every value is a bf16
    nib, sc, g = F.quantize_matrix(w)
    return (nib, sc, g), xb, x


@pytest.mark.parametrize("m", [1, 5, 8, 16])
def test_gemm_activation_dynamic_range(lib, m):
    """The tensor-core and CUDA-core paths take the bf16 activations as f16 after a
    per-row power-of-two rescale that puts the row maximum (over the staged columns)
    in [2^14, 2^15).  A bf16 value 2^31 or less below the maximum keeps every bit; one
    more than 2^38 below it falls under f16's smallest subnormal and is dropped.
    (a) Small values 2^30 below the large ones, the weights under the large values
    zero, so the result is made of the small values alone: within the bound.
    (b) The same rows with the small values 2^50 below: they are dropped, and the
    result is exactly zero (the documented limit of the f16 operands).
    (c) 2^50 of range with the large values weighted: within the bound, since the
    dropped terms are below 2^-38 of the largest term."""
    n, k = 192, 1024
    for small_exp, weighted, what in ((-20, False, "a"), (-40, False, "b"), (-40, True, "c")):
        q, xb, x = _wide_range_case(m, n, k, small_exp, weighted)
        wt = upload_oracle_weight(lib, q)
        y = bf16_to_f64(lib.gemm(wt, upload_bf16(xb)))
        torch.cuda.synchronize()
        exact, _, absy = OG.nvfp4_gemm(*q, x.astype(np.float64))
        if what == "b":
            assert np.all(y == 0.0) and np.all(exact != 0.0), "values 2^50 below the row maximum were not dropped"
        else:
            check_bound(y, exact, absy, True, f"dynamic range case {what} m={m}")
    assert lib.device_error() == 0


_DENSE_FULL = {}


def _dense_full(lib, n):
    """The config-1 weight of N rows: the oracle's bytes repacked on the GPU for the
    kernel, after checking that the GPU quantizer gives the same bytes at full size."""
    if n not in _DENSE_FULL:
        _DENSE_FULL.clear()
        w = W.DenseCase.sweep(1, n).w()
        q = oracle_quantize(w)
        assert_gpu_quantizer_matches(lib, w, q, f"config1 n={n}")
        _DENSE_FULL[n] = (upload_oracle_weight(lib, q), q)
        torch.cuda.synchronize()
    return _DENSE_FULL[n]


@pytest.mark.parametrize("n", [4096, 14336])
@pytest.mark.parametrize("m", [1, 4, 15, 16])
def test_gemm_config1_full_size(lib, m, n):
    case = W.DenseCase.sweep(m, n)
    wt, (nib, sc, g) = _dense_full(lib, n)
    xb, xf = case.x()
    y = lib.gemm(wt, upload_bf16(xb))
    torch.cuda.synchronize()
    exact, _, absy = OG.nvfp4_gemm(nib, sc, g, xf.astype(np.float64))
    check_bound(bf16_to_f64(y), exact, absy, True, f"config1 m={m} n={n}")
    assert lib.device_error() == 0


def test_gemm_repeat_calls_stable(lib):
    """Back-to-back calls on one workspace (split-K counters stay consistent)."""
    case = W.DenseCase.sweep(16, 4096)
    w = case.w()
    xb, _ = case.x()
    wt = lib.prepare(upload_f32(w))
    x = upload_bf16(xb)
    first = lib.gemm(wt, x).clone()
    for _ in range(5):
        again = lib.gemm(wt, x)
        assert torch.equal(again, first)


# ------------------------------------------------------------------ lm_head

def _lm(lib, m, vocab, k, w_seed, x_seed, plant=None):
    w = W.weight((vocab, k), w_seed)
    xb, xf = W.activations((m, k), x_seed)
    if plant is not None:
        row, tok = plant
        w[row] = np.sign(xf[tok]).astype(np.float32) * 0.05
    wt = lib.prepare(upload_f32(w))
    mx, idx = lib.lm_head_argmax(wt, upload_bf16(xb))
    torch.cuda.synchronize()
    nib, sc, g = F.quantize_matrix(w)
    ref = OLM.lm_head_argmax(nib, sc, g, xf.astype(np.float64))
    return mx.cpu().numpy(), idx.cpu().numpy(), ref, (nib, sc, g, xf)


def _check_argmax(mx, idx, ref, parts, what):
    nib, sc, g, xf = parts
    for t in range(len(idx)):
        lg, la = OLM.logits_rows(nib, sc, g, xf[t:t + 1].astype(np.float64), [idx[t], ref["argmax"][t]])
        tol = 1e-3 * max(la[0, 0], la[0, 1])
        gap = ref["max"][t] - ref["second"][t]
        if gap > 2 * tol:
            assert idx[t] == ref["argmax"][t], f"{what}: token {t} argmax {idx[t]} != {ref['argmax'][t]}"
        else:   # a near-tie: the returned row must be a valid maximiser within the bound
            assert ref["max"][t] - lg[0, 0] <= 2 * tol, f"{what}: token {t} near-tie row not maximal"
        assert abs(mx[t] - lg[0, 0]) <= tol, f"{what}: token {t} max logit {mx[t]} vs {lg[0, 0]}"


@pytest.mark.parametrize("m", [1, 3, 7, 8, 15, 16])
@pytest.mark.parametrize("vocab,k", [(3000, 256), (1037, 2816), (1, 64), (17, 16), (64, 4096)])
def test_lm_head_small(lib, m, vocab, k):
    mx, idx, ref, parts = _lm(lib, m, vocab, k, 300 + vocab, 400 + m)
    _check_argmax(mx, idx, ref, parts, f"lm_head m={m} vocab={vocab}")


def test_lm_head_planted_max_and_tie(lib):
    m, vocab, k = 4, 2048, 256
    w = W.weight((vocab, k), 77)
    xb, xf = W.activations((m, k), 78)
    w[1500] = np.sign(xf[2]).astype(np.float32) * 0.05   # token 2: planted winner
    w[700] = w[1500]                                     # identical row, lower index: must win the tie
    wt = lib.prepare(upload_f32(w))
    mx, idx = lib.lm_head_argmax(wt, upload_bf16(xb))
    torch.cuda.synchronize()
    assert idx[2].item() == 700
    nib, sc, g = F.quantize_matrix(w)
    ref = OLM.lm_head_argmax(nib, sc, g, xf.astype(np.float64))
    assert ref["argmax"][2] == 700
    assert np.array_equal(idx.cpu().numpy(), ref["argmax"])


@pytest.mark.parametrize("m", [3, 9])
def test_lm_head_nan_token_row(lib, m):
    """A token row of NaN activations makes every logit of that token NaN, which counts
    as -inf: the result is (-inf, row 0); the other tokens are unaffected (CUDA-core and
    tensor-core paths)."""
    vocab, k = 2048, 256
    w = W.weight((vocab, k), 91)
    xb, xf = W.activations((m, k), 92)
    xb = xb.copy()
    xb[1, :] = 0x7FC0                       # bf16 quiet NaN
    q = F.quantize_matrix(w)
    wt = upload_oracle_weight(lib, q)
    mx, idx = lib.lm_head_argmax(wt, upload_bf16(xb))
    torch.cuda.synchronize()
    assert idx[1].item() == 0 and mx[1].item() == float("-inf")
    keep = [t for t in range(m) if t != 1]
    ref = OLM.lm_head_argmax(*q, xf[keep].astype(np.float64))
    _check_argmax(mx.cpu().numpy()[keep], idx.cpu().numpy()[keep], ref, (*q, xf[keep]), "lm_head NaN row")
    assert lib.device_error() == 0


@pytest.fixture(scope="module")
def lm_head_full(lib):
    """The full 262,144 x 2,816 lm_head quantized by the oracle; the kernel reads the
    oracle's bytes (repacked on the GPU).  The GPU quantizer's bytes for the whole
    matrix are checked equal to the oracle's on the way."""
    case = W.LMHeadCase(m=1)
    w = case.w_rows(0, case.vocab)
    q = oracle_quantize(w)
    assert_gpu_quantizer_matches(lib, w, q, "lm_head 262144x2816")
    wt = upload_oracle_weight(lib, q)
    torch.cuda.synchronize()
    nib, sc, g = q
    return wt, nib, sc, g


@pytest.mark.parametrize("m", [1, 15])
def test_lm_head_config3_full_size(lib, lm_head_full, m):
    wt, nib, sc, g = lm_head_full
    assert wt.global_scale.item() == float(g)
    xb, xf = W.LMHeadCase(m=m).x()
    mx, idx = lib.lm_head_argmax(wt, upload_bf16(xb))
    torch.cuda.synchronize()
    ref = OLM.lm_head_argmax(nib, sc, g, xf.astype(np.float64), chunk_rows=16384)
    _check_argmax(mx.cpu().numpy(), idx.cpu().numpy(), ref, (nib, sc, g, xf), f"lm_head full m={m}")
    assert lib.device_error() == 0
