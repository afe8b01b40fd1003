"""Temperature sampling from the lm_head by the Gumbel-max rule (oracle; test
infrastructure only).

gemma-cuda-hybrid README, "Server (SERVE=1 ./build/forward)": lossless temperature
sampling by Gumbel-max, where temperature 0 reduces to exact greedy decoding.
Gumbel-max: with independent standard Gumbel noise g_n, the index
argmax_n (logit_n / T + g_n) is distributed as softmax(logit / T).

The pages do not name the noise generator.  Both sides use the counter-based
Philox4x32-10 generator (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
easy as 1, 2, 3", SC 2011), written here from its definition: ten rounds of two
32x32->64-bit multiplies by the fixed multipliers, the high halves crossed and
XORed with the round key and the other words, the key bumped by the Weyl
constants between rounds.  The draw for vocabulary row n of token m under a
64-bit seed is word 0 of Philox(counter = (n, m, 0, 0), key = (seed low, seed
high)); u = ((word >> 9) + 0.5) / 2^23 -- the top 23 bits, so that u (a 24-bit
odd multiple of 2^-24) is exact in fp32 as well and lies strictly inside (0, 1)
-- and g = -log(-log u).
"""

from __future__ import annotations

import numpy as np

from .formats import dequantize_matrix

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9  # golden ratio
PHILOX_W1 = 0xBB67AE85  # sqrt(3) - 1
MASK32 = 0xFFFFFFFF


def _mulhilo(a, m):
    p = a.astype(np.uint64) * np.uint64(m)
    return (p >> np.uint64(32)).astype(np.uint64), (p & np.uint64(MASK32)).astype(np.uint64)


def philox4x32_10(counter, key):
    """counter: uint32 array [..., 4]; key: uint32 array [..., 2] (broadcast).
    Returns uint32 [..., 4]."""
    c = np.asarray(counter, np.uint64) & np.uint64(MASK32)
    k = np.asarray(key, np.uint64) & np.uint64(MASK32)
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k0, k1 = k[..., 0].copy(), k[..., 1].copy()
    for r in range(10):
        if r > 0:
            k0 = (k0 + np.uint64(PHILOX_W0)) & np.uint64(MASK32)
            k1 = (k1 + np.uint64(PHILOX_W1)) & np.uint64(MASK32)
        hi0, lo0 = _mulhilo(c0, PHILOX_M0)
        hi1, lo1 = _mulhilo(c2, PHILOX_M1)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniform_open(word):
    """uint32 -> a float in (0, 1): ((word >> 9) + 0.5) / 2^23 (exact in fp32 and fp64)."""
    w = np.asarray(word, np.uint64) >> np.uint64(9)
    return (w.astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel(word):
    """Standard Gumbel noise from a uint32 draw: -log(-log(u))."""
    return -np.log(-np.log(uniform_open(word)))


def noise(rows, tokens, seed):
    """g[token, row] for the given vocabulary rows and token indices under `seed`."""
    rows = np.asarray(rows, np.uint64)
    tokens = np.asarray(tokens, np.uint64)
    n, t = np.meshgrid(rows, tokens)  # [tokens, rows]
    ctr = np.stack([n, t, np.zeros_like(n), np.zeros_like(n)], axis=-1)
    key = np.array([seed & MASK32, (seed >> 32) & MASK32], np.uint64)
    return gumbel(philox4x32_10(ctr, key)[..., 0])


def softcap_logits(logits, cap):
    """cap * tanh(logits / cap) for cap > 0, else the logits (the same rule as router.softcap)."""
    from .router import softcap
    return softcap(logits, cap)


def sample_keys(logits, temperature, seed, row0=0):
    """keys[m, n] = logits[m, n] / T + g(row0 + n, m); float64."""
    logits = np.asarray(logits, np.float64)
    m, n = logits.shape
    return logits / temperature + noise(np.arange(row0, row0 + n), np.arange(m), seed)


def lm_head_sample(nib, scales, g, x, temperature, seed, chunk_rows: int = 8192, softcap: float = 0.0):
    """Per token row: the index of the largest key logit/T + Gumbel noise (ties to
    the lower index), that key, the second-largest key, and tol_scale (sum|w*x| of
    the winning row, for the logit's error bound).  The logits are exact float64
    products of the dequantized weights and x; softcap > 0 replaces each logit l
    by softcap * tanh(l / softcap) first (TensorSharp docs/models/gemma4.md, "4.8
    Logit softcap").  temperature 0: the key is the (capped) logit itself, no
    noise -- the greedy argmax."""
    x = np.asarray(x, np.float64)
    m = x.shape[0]
    n = nib.shape[0]
    best = np.full(m, -np.inf)
    best_i = np.full(m, -1, dtype=np.int64)
    second = np.full(m, -np.inf)
    best_abs = np.zeros(m)
    for lo in range(0, n, chunk_rows):
        hi = min(n, lo + chunk_rows)
        w = dequantize_matrix(nib[lo:hi], scales[lo:hi], g)
        logits = softcap_logits(x @ w.T, softcap)
        keys = sample_keys(logits, temperature, seed, row0=lo) if temperature > 0 else logits
        absl = np.abs(x) @ np.abs(w).T
        for t in range(m):
            row = keys[t]
            j = int(np.argmax(row))  # first (lowest) index of the max
            v = row[j]
            top2 = np.partition(row, -2)[-2] if row.size > 1 else -np.inf
            if v > best[t]:
                second[t] = max(best[t], top2)
                best[t], best_i[t], best_abs[t] = v, lo + j, absl[t, j]
            else:
                second[t] = max(second[t], v)
    return dict(index=best_i, key=best, second=second, tol_scale=best_abs)
