"""Pins of the sampling oracle (CPU): the Philox4x32-10 generator against its published
known-answer vectors, the Gumbel transform against its closed form, and the Gumbel-max
rule against its defining property -- the sampled index is distributed as
softmax(logits / T) -- plus the chunked lm_head sampler against a one-shot computation."""

import os

import numpy as np
import pytest

from oracle import formats as F
from oracle import sampling as OS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answer_vectors():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(h, 16) for h in r]
        out = OS.philox4x32_10(np.array(v[:4], np.uint64), np.array(v[4:6], np.uint64))
        assert [int(o) for o in out] == v[6:10]


def test_gumbel_is_the_inverse_cdf():
    words = np.array([0, 1, 2 ** 31, 2 ** 32 - 1, 123456789], np.uint64)   # g stays finite at both ends
    u = OS.uniform_open(words)
    assert np.all(u > 0) and np.all(u < 1)
    g = OS.gumbel(words)
    assert np.allclose(np.exp(-np.exp(-g)), u, rtol=1e-12)          # the Gumbel CDF at g is u
    assert OS.uniform_open(np.array([0], np.uint64))[0] == 0.5 * 2.0 ** -23          # smallest u
    assert OS.uniform_open(np.array([2 ** 32 - 1], np.uint64))[0] == 1 - 0.5 * 2.0 ** -23  # largest u
    # every u is exactly representable in fp32 (24 significant bits)
    us = OS.uniform_open(np.array([0, 1 << 9, 2 ** 31, 2 ** 32 - 1, 0xDEADBEEF], np.uint64))
    assert np.array_equal(us.astype(np.float32).astype(np.float64), us)
    half = OS.gumbel(np.array([2 ** 31], np.uint64))[0]               # u = (2^22 + 0.5) / 2^23
    assert half == pytest.approx(-np.log(-np.log(0.5 + 2.0 ** -24)), abs=1e-12)
    assert half == pytest.approx(-np.log(np.log(2.0)), abs=1e-6)


def test_gumbel_max_samples_softmax_of_logits_over_t():
    logits = np.array([1.0, 0.5, -0.3, 2.0, 0.0])
    t = 0.8
    draws = 60000
    g = OS.noise(np.arange(5), np.arange(draws), seed=0x1234_5678_9ABC)   # [draws, 5]
    picks = np.argmax(logits / t + g, axis=1)
    freq = np.bincount(picks, minlength=5) / draws
    p = np.exp(logits / t - np.max(logits / t))
    p /= p.sum()
    sigma = np.sqrt(p * (1 - p) / draws)
    assert np.all(np.abs(freq - p) < 5 * sigma), (freq, p)


def test_noise_depends_on_row_token_and_seed():
    a = OS.noise(np.arange(8), np.arange(3), 7)
    assert a.shape == (3, 8)
    assert not np.allclose(a, OS.noise(np.arange(8), np.arange(3), 8))
    assert np.array_equal(a[:, 4:], OS.noise(np.arange(4, 8), np.arange(3), 7))   # row-addressed
    assert len(np.unique(a)) == a.size


def test_chunked_sampler_matches_one_shot_and_low_t_is_greedy():
    rng = np.random.default_rng(3)
    w = (0.02 * rng.standard_normal((300, 64))).astype(np.float32)
    nib, sc, g = F.quantize_matrix(w)
    x = rng.standard_normal((4, 64))
    logits = x @ F.dequantize_matrix(nib, sc, g).T
    res = OS.lm_head_sample(nib, sc, g, x, 0.7, seed=99, chunk_rows=64)
    keys = OS.sample_keys(logits, 0.7, 99)
    assert np.array_equal(res["index"], np.argmax(keys, axis=1))
    assert np.allclose(res["key"], keys.max(axis=1))
    srt = np.sort(keys, axis=1)
    assert np.allclose(res["second"], srt[:, -2])
    cold = OS.lm_head_sample(nib, sc, g, x, 1e-7, seed=99, chunk_rows=64)
    assert np.array_equal(cold["index"], np.argmax(logits, axis=1))
