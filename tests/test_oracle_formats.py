"""Pins for the oracle's NVFP4 codecs and quantizer (CPU only).

Each check ties the oracle to something other than itself: the published E2M1
table, torch's independent float8_e4m3fn decoder/encoder, brute-force nearest
search, and exact round trips on values built to be representable.
"""

import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def test_e2m1_table_matches_published_table():
    rows = _load_table("e2m1_table.txt")
    codes = np.array([int(r[0]) for r in rows])
    vals = np.array([float(r[1]) for r in rows])
    got = F.e2m1_value(codes)
    assert np.array_equal(got, vals)
    # the sign of zero is kept (code 8 is -0)
    assert np.signbit(got[8]) and not np.signbit(got[0])


def test_e4m3_all_256_codes_match_torch():
    codes = np.arange(256)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_value(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan], ref[~nan])
    assert F.e4m3_value(0x7E) == 448.0 and F.e4m3_value(1) == 2.0 ** -9


def test_e4m3_encode_round_trip_and_midpoints():
    codes = np.arange(0x7F)                       # all finite non-negative codes
    vals = F.e4m3_value(codes)
    assert np.array_equal(F.e4m3_encode_nonneg(vals), codes.astype(np.uint8))
    # exact midpoints between neighbours go to the even code
    mids = (vals[:-1] + vals[1:]) / 2
    enc = F.e4m3_encode_nonneg(mids).astype(int)
    lo = codes[:-1]
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(enc, expect)
    # saturation above the largest finite value
    assert np.all(F.e4m3_encode_nonneg(np.array([448.0, 460.0, 464.0, 1e4, 3e38])) == 0x7E)


def test_e4m3_encode_matches_torch_on_random_fp32():
    rng = np.random.default_rng(11)
    t = np.concatenate([
        rng.uniform(0, 448, 20000),
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 20000)),
        rng.uniform(0, 2.0 ** -6, 5000),
    ]).astype(np.float32)
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode_nonneg(t), ref)


def _e2m1_brute(v):
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    out = []
    for x in np.asarray(v, np.float64):
        a = min(abs(x), 6.0)
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        out.append(code | (8 if np.signbit(x) else 0))
    return np.array(out, np.uint8)


def test_e2m1_encode_brute_force_and_ties():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.uniform(-8, 8, 20000), rng.uniform(-1, 1, 5000),
                        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, 7.0, -100.0])])
    v = v.astype(np.float32)
    assert np.array_equal(F.e2m1_encode(v), _e2m1_brute(v))
    ties = F.e2m1_encode(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))
    assert list(F.e2m1_value(ties)) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert F.e2m1_encode(np.array([-1e-30]))[0] == 8       # -tiny keeps its sign: -0
    assert F.e2m1_encode(np.array([7.0, -9.0])).tolist() == [7, 15]


def _representable_matrix(rng, n, k, g_exp=-10):
    """W whose exact NVFP4 encoding is known: g = 2^g_exp, every block has an element of
    magnitude 6 so its scale is recovered, and one block sits at the global max."""
    g = np.float32(2.0 ** g_exp)
    s_codes = rng.integers(1, 0x7F, size=(n, k // 16)).astype(np.uint8)
    s_codes[0, 0] = 0x7E                                   # 448: fixes amax = 2688 g
    q = rng.integers(0, 16, size=(n, k)).astype(np.uint8)
    q.reshape(n, k // 16, 16)[:, :, 5] = np.where(rng.random((n, k // 16)) < 0.5, 7, 15)
    w = F.e2m1_value(q).reshape(n, k // 16, 16) * F.e4m3_value(s_codes)[:, :, None] * float(g)
    return w.reshape(n, k).astype(np.float32), q, s_codes, g


def test_quantize_exact_round_trip_on_representable_values():
    rng = np.random.default_rng(5)
    w, q, s_codes, g = _representable_matrix(rng, 24, 128)
    nib, sc, g2 = F.quantize_matrix(w)
    assert g2 == g
    assert np.array_equal(sc, s_codes)
    assert np.array_equal(F.unpack_nibbles(nib), q)
    assert np.array_equal(F.dequantize_matrix(nib, sc, g2), w.astype(np.float64))


def test_quantize_special_cases():
    z = np.zeros((4, 32), np.float32)
    nib, sc, g = F.quantize_matrix(z)
    assert g == 0 and not nib.any() and not sc.any()
    w = np.zeros((2, 32), np.float32)
    w[0, 3] = 1.0
    w[1, 20] = 1e-12          # far below the block-scale range: whole block flushes to zero
    nib, sc, g = F.quantize_matrix(w)
    assert g == np.float32(1.0) / np.float32(2688.0)
    assert sc[0, 0] == 0x7E and F.unpack_nibbles(nib)[0, 3] == 7      # 448 * 6 * g = 1
    assert sc[1, 1] == 0 and not F.unpack_nibbles(nib)[1].any()


def test_quantize_error_bound_random():
    """Every element is within half an E2M1 step of its block scale (RNE), saturation aside."""
    rng = np.random.default_rng(9)
    w = (0.02 * rng.standard_normal((64, 256))).astype(np.float32)
    nib, sc, g = F.quantize_matrix(w)
    wh = F.dequantize_matrix(nib, sc, g)
    step = F.e4m3_value(sc).repeat(16, axis=1) * float(g)     # scale * g per element
    assert np.all(np.abs(wh - w) <= 1.0 * step + 1e-12)        # max E2M1 gap is 2 -> half is 1
    assert np.max(np.abs(wh - w)) < 0.2 * np.max(np.abs(w))


def test_dequantize_matches_triple_loop():
    rng = np.random.default_rng(2)
    w = rng.standard_normal((8, 48)).astype(np.float32)
    nib, sc, g = F.quantize_matrix(w)
    table = {int(r[0]): float(r[1]) for r in _load_table("e2m1_table.txt")}
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref = np.zeros((8, 48))
    for n in range(8):
        for k in range(48):
            byte = int(nib[n, k // 2])
            code = (byte >> 4) if k % 2 else (byte & 0xF)
            ref[n, k] = table[code] * e4[int(sc[n, k // 16])] * float(g)
    assert np.array_equal(F.dequantize_matrix(nib, sc, g), ref)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(10000) * 10.0 ** rng.integers(-6, 6, 10000),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)])])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.bf16_round(x), ref)


# ------------------------------------------------------------------ exact-quotient quantizer

def _exact_nearest(x, grid_vals, grid_codes):
    """Nearest grid value to the exact rational x >= 0, ties to the even code (brute force)."""
    best, best_d = None, None
    for v, c in zip(grid_vals, grid_codes):
        d = abs(x - v)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best


def _quantize_brute_exact(w):
    """The quantizer written over exact rationals: g = fp32(amax / 2688); per block the
    E4M3 code nearest to bmax / (6 g), ties to even, saturating at 448; per element the
    E2M1 code nearest to |w| / (e4m3(s) g), ties to even, saturating at 6, sign kept."""
    from fractions import Fraction as Fr
    w = np.asarray(w, np.float32)
    n, k = w.shape
    amax = np.max(np.abs(w))
    g = np.float32(np.float32(amax) / np.float32(2688.0))   # one correctly rounded fp32 division
    e4_codes = list(range(0x7F))
    e4_vals = [Fr(float(F.e4m3_value(c))) for c in e4_codes]
    e2_codes = list(range(8))
    e2_vals = [Fr(float(F.e2m1_value(c))) for c in e2_codes]
    gq = Fr(float(g))
    sc = np.zeros((n, k // 16), np.uint8)
    q = np.zeros((n, k), np.uint8)
    for r in range(n):
        for j in range(k // 16):
            blk = [Fr(float(x)) for x in w[r, 16 * j:16 * j + 16]]
            t = max(abs(x) for x in blk) / (6 * gq)
            c = 0x7E if t >= 448 else _exact_nearest(t, e4_vals, e4_codes)
            sc[r, j] = c
            s = e4_vals[c]
            for i, x in enumerate(blk):
                if s == 0:
                    continue
                v = abs(x) / (s * gq)
                code = 7 if v >= 6 else _exact_nearest(v, e2_vals, e2_codes)
                q[r, 16 * j + i] = code | (8 if np.signbit(w[r, 16 * j + i]) else 0)
    return q, sc, g


def _near_midpoint_matrix():
    """Blocks whose maxima, and elements, sit on or one fp32 step either side of the
    exact rounding midpoints, under a global scale with a full 24-bit significand."""
    amax = np.float32(1.2345678)
    g = np.float64(np.float32(amax / np.float32(2688.0)))
    rows = []
    e4 = F.e4m3_value(np.arange(0x7F))
    e2 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for c in (9, 30, 37, 50, 61, 77, 100, 117):          # midpoints between codes c and c + 1
        mid = (e4[c] + e4[c + 1]) / 2 * 6 * g            # exact real bmax of the midpoint
        for bmax in (np.nextafter(np.float32(mid), np.float32(0)), np.float32(mid),
                     np.nextafter(np.float32(mid), np.float32(10))):
            row = np.zeros(16, np.float32)
            row[0] = bmax
            # elements near E2M1 midpoints of the scale this block should get
            s = e4[c] if bmax < mid else (e4[c + 1] if bmax > mid else e4[c + (c % 2)])
            for i, (a, b) in enumerate(zip(e2[:-1], e2[1:])):
                m2 = np.float32((a + b) / 2 * s * g)
                row[1 + 2 * i] = np.nextafter(m2, np.float32(0)) if i % 2 else m2
                row[2 + 2 * i] = -np.nextafter(m2, np.float32(10))
            rows.append(row)
    w = np.stack(rows)
    w[0, 15] = amax                                       # fixes the global maximum
    return w


def test_quantize_matches_exact_rational_brute_force():
    """The oracle's quantizer equals the quantizer written over exact rationals, on
    random blocks and on blocks planted at the rounding midpoints."""
    rng = np.random.default_rng(17)
    rand = (0.02 * rng.standard_normal((6, 64))).astype(np.float32)
    for w in (rand, _near_midpoint_matrix()):
        nib, sc, g = F.quantize_matrix(w)
        q_ref, sc_ref, g_ref = _quantize_brute_exact(w)
        assert g == g_ref
        assert np.array_equal(sc, sc_ref)
        assert np.array_equal(F.unpack_nibbles(nib), q_ref)


def test_exact_quotients_differ_from_fp32_quotients_on_planted_midpoints():
    """The planted blocks have teeth: deciding on IEEE fp32 quotients ((bmax / 6) / g and
    w / fp32(s * g)) picks other codes for some of them than the exact quotients."""
    w = _near_midpoint_matrix()
    nib, sc, g = F.quantize_matrix(w)
    blocks = w.reshape(w.shape[0], -1, 16)
    bmax = np.max(np.abs(blocks), axis=2).astype(np.float32)
    t32 = (bmax / np.float32(6.0)).astype(np.float32) / g
    sc32 = F.e4m3_encode_nonneg(t32.astype(np.float32))
    den32 = (F.e4m3_value(sc).astype(np.float32) * g).astype(np.float32)
    q32 = F.e2m1_encode((blocks / den32[:, :, None]).astype(np.float32)).reshape(w.shape)
    diff = int(np.sum(sc32 != sc)) + int(np.sum(q32 != F.unpack_nibbles(nib)))
    assert diff > 0
