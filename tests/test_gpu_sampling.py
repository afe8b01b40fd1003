"""GPU parity: lm_head temperature sampling by the Gumbel-max rule vs the oracle.

The kernel adds Philox4x32-10 Gumbel noise to logit / T in the lm_head epilogue and
keeps the per-row maximum; the oracle does the same in float64 with exact logits.
The index must match the oracle's exactly unless the oracle's top-2 keys are closer
than twice the error bound (then the chosen row must be a maximiser within it)."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import lm_head as OLM
from oracle import sampling as OS
from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
from tests.gpu_helpers import upload_bf16, upload_f32, upload_oracle_weight

pytestmark = pytest.mark.gpu

NOISE_TOL = 1e-5   # fp32 -logf(-logf(u)) against float64, |g| < 17 for u in (2^-25, 1 - 2^-25)


def _check_sample(key, tok, ref, parts, t_temp, seed, what, softcap=0.0):
    nib, sc, g, xf = parts
    for t in range(len(tok)):
        rows = [int(tok[t]), int(ref["index"][t])]
        lg, la = OLM.logits_rows(nib, sc, g, xf[t:t + 1].astype(np.float64), rows)
        lg = OS.softcap_logits(lg, softcap)     # the cap's slope is at most 1: the logit bound carries over
        if t_temp > 0:
            keys = lg[0] / t_temp + OS.noise(np.array(rows), np.array([t]), seed)[0]
            tol = 1e-3 * max(la[0, 0], la[0, 1]) / t_temp + NOISE_TOL + 1e-6 * softcap / t_temp
        else:
            keys = lg[0]
            tol = 1e-3 * max(la[0, 0], la[0, 1]) + 1e-6 * softcap
        gap = ref["key"][t] - ref["second"][t]
        if gap > 2 * tol:
            assert rows[0] == rows[1], f"{what}: token {t} sampled {rows[0]} != {rows[1]} (gap {gap:.3g})"
        else:   # a near-tie of keys: the chosen row must be a maximiser within the bound
            assert ref["key"][t] - keys[0] <= 2 * tol, f"{what}: token {t} near-tie row not maximal"
        assert abs(key[t] - keys[0]) <= tol, f"{what}: token {t} key {key[t]} vs {keys[0]}"


def _run(lib, wt, xb, t_temp, seed):
    key, tok = lib.lm_head_sample(wt, upload_bf16(xb), t_temp, seed)
    torch.cuda.synchronize()
    return key.cpu().numpy(), tok.cpu().numpy()


@pytest.mark.parametrize("m", [1, 3, 8, 15, 16])
@pytest.mark.parametrize("t_temp", [0.5, 1.0, 3.0])
def test_sample_small_vocab(lib, m, t_temp):
    vocab, k = 3000, 256                      # 3000 rows: a ragged last 64-row group
    w = W.weight((vocab, k), 5000 + m)
    xb, xf = W.activations((m, k), 5100 + m)
    wt = lib.prepare(upload_f32(w))
    seed = (m * 1_000_003 + int(t_temp * 10)) | (1 << 40)
    key, tok = _run(lib, wt, xb, t_temp, seed)
    nib, sc, g = F.quantize_matrix(w)
    ref = OS.lm_head_sample(nib, sc, g, xf.astype(np.float64), t_temp, seed)
    _check_sample(key, tok, ref, (nib, sc, g, xf), t_temp, seed, f"sample m={m} T={t_temp}")
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [1, 15])
@pytest.mark.parametrize("t_temp", [0.0, 1.0])
def test_softcap_on_the_logits(lib, m, t_temp):
    """The final-logit softcap (cap 30) in the lm_head epilogue: weights scaled so the
    logits reach the cap's curved range; the greedy index, the sampled index and the
    returned keys follow the oracle's capped logits."""
    vocab, k, cap = 3000, 256, 30.0
    w = W.weight((vocab, k), 5600 + m) * 25.0
    xb, xf = W.activations((m, k), 5700 + m)
    q = F.quantize_matrix(w)
    wt = upload_oracle_weight(lib, q)
    seed = 777 + m
    key, tok = lib.lm_head_sample(wt, upload_bf16(xb), t_temp, seed, softcap=cap)
    torch.cuda.synchronize()
    ref = OS.lm_head_sample(*q, xf.astype(np.float64), t_temp, seed, softcap=cap)
    assert np.max(np.abs(ref["key"])) > 0.5 * cap         # the cap bends the winning logits
    _check_sample(key.cpu().numpy(), tok.cpu().numpy(), ref, (*q, xf), t_temp, seed,
                  f"softcap m={m} T={t_temp}", softcap=cap)
    assert lib.device_error() == 0


def test_sample_temperature_zero_is_the_greedy_argmax(lib):
    m, vocab, k = 8, 2048, 256
    wt = lib.prepare(upload_f32(W.weight((vocab, k), 5200)))
    xb, _ = W.activations((m, k), 5201)
    mx, idx = lib.lm_head_argmax(wt, upload_bf16(xb))
    key, tok = lib.lm_head_sample(wt, upload_bf16(xb), 0.0, 12345)
    torch.cuda.synchronize()
    assert torch.equal(tok, idx) and torch.equal(key, mx)


def test_sample_frequencies_follow_softmax(lib):
    """The GPU's own noise, checked against the Gumbel-max property: over many seeds,
    16 token rows with the same activation pick vocabulary row n with probability
    softmax(logits / T)[n] (64 rows, T = 2: a wide distribution)."""
    vocab, k, m, t_temp, seeds = 64, 64, 16, 2.0, 250
    w = W.weight((vocab, k), 5300) * 10.0
    xb1, xf1 = W.activations((1, k), 5301)
    xb = np.repeat(xb1, m, axis=0)
    wt = lib.prepare(upload_f32(w))
    x = upload_bf16(xb)
    counts = np.zeros(vocab)
    for s in range(seeds):
        _, tok = lib.lm_head_sample(wt, x, t_temp, 0xABC000 + s)
        counts += np.bincount(tok.cpu().numpy(), minlength=vocab)
    nib, sc, g = F.quantize_matrix(w)
    logits = (xf1.astype(np.float64) @ F.dequantize_matrix(nib, sc, g).T)[0]
    p = np.exp(logits / t_temp - np.max(logits / t_temp))
    p /= p.sum()
    draws = seeds * m
    sigma = np.sqrt(p * (1 - p) / draws)
    assert np.all(np.abs(counts / draws - p) < 5 * sigma + 1e-9), (counts / draws, p)
    assert lib.device_error() == 0


def test_sample_seeds_differ_and_repeat(lib):
    m, vocab, k = 16, 512, 128
    wt = lib.prepare(upload_f32(W.weight((vocab, k), 5400) * 0.1))   # nearly flat logits
    xb, _ = W.activations((m, k), 5401)
    a = _run(lib, wt, xb, 1.0, 1)
    b = _run(lib, wt, xb, 1.0, 1)
    c = _run(lib, wt, xb, 1.0, 2)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[0], b[0])   # deterministic in the seed
    assert not np.array_equal(a[1], c[1])                              # another seed, other draws


def test_sample_rejects_bad_temperature(lib):
    wt = lib.prepare(upload_f32(W.weight((128, 64), 5500)))
    xb, _ = W.activations((1, 64), 5501)
    for bad in (-1.0, float("nan"), float("inf")):
        with pytest.raises(Exception):
            lib.lm_head_sample(wt, upload_bf16(xb), bad, 1)


def test_sample_config3_full_size(lib):
    case = W.LMHeadCase(m=15)
    w = case.w_rows(0, case.vocab)
    wt = lib.prepare(upload_f32(w))
    nib, sc, g = F.quantize_matrix(w)
    del w
    xb, xf = case.x()
    seed = 0x5EED_0000_0001
    key, tok = _run(lib, wt, xb, 1.0, seed)
    ref = OS.lm_head_sample(nib, sc, g, xf.astype(np.float64), 1.0, seed, chunk_rows=16384)
    _check_sample(key, tok, ref, (nib, sc, g, xf), 1.0, seed, "sample full m=15")
    assert lib.device_error() == 0
