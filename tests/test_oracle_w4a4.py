"""Pins for the W4A4 oracle (activations quantized to NVFP4 per token row) (CPU)."""

import math

import numpy as np

from oracle import formats as F
from oracle import gemm as G
from oracle import w4a4 as A

E4M3_448 = 0x7E  # the largest finite E4M3 code


def _representable_rows(rng, m, k, g_exp=-10):
    """Rows x = e2m1(q) * e4m3(s) * 2^g_exp in which every 16-block holds a +-6 and
    one block of each row has s = 448, so that the row's amax is 2688 * 2^g_exp:
    the global scale is exactly 2^g_exp, each block's scale is exactly s, and
    every element is an E2M1 value times s * g."""
    g = 2.0 ** g_exp
    q = rng.integers(0, 16, size=(m, k))
    s = rng.integers(0x20, 0x70, size=(m, k // 16))
    s[:, 0] = E4M3_448
    for b in range(k // 16):
        q[:, 16 * b + rng.integers(0, 16)] = rng.choice([7, 15], size=m)  # +-6 in every block (codes 7 / 15)
    x = F.e2m1_value(q.astype(np.uint8)) * np.repeat(F.e4m3_value(s.astype(np.uint8)), 16, axis=1) * g
    assert np.all(np.abs(x).max(axis=1) == 2688 * g)
    return x.astype(np.float32), q, s


def test_representable_rows_round_trip_exactly():
    rng = np.random.default_rng(3)
    x, q, s = _representable_rows(rng, 5, 128)
    codes, scales, g = A.quantize_activations(x)
    assert np.all(g == np.float32(2.0 ** -10))
    assert np.array_equal(scales, s.astype(np.uint8))
    # codes equal up to the sign of zero (+0 and -0 both dequantize to 0)
    got = F.unpack_nibbles(codes)
    zero = F.e2m1_value(q.astype(np.uint8)) == 0
    assert np.array_equal(np.where(zero, 0, got), np.where(zero, 0, q))
    assert np.array_equal(A.dequantize_activations(codes, scales, g), x.astype(np.float64))


def test_w4a4_equals_w4a16_on_representable_activations():
    """When x is already an NVFP4 value per row, quantizing it changes nothing, so
    the W4A4 product equals the W4A16 product on the same x."""
    rng = np.random.default_rng(4)
    x, _, _ = _representable_rows(rng, 3, 256)
    wq = F.quantize_matrix((0.02 * rng.standard_normal((40, 256))).astype(np.float32))
    xq = A.quantize_activations(x)
    y4, _, a4 = A.w4a4_gemm(*wq, xq)
    y16, _, a16 = G.nvfp4_gemm(*wq, x.astype(np.float64))
    assert np.array_equal(y4, y16) and np.array_equal(a4, a16)


def test_each_row_has_its_own_global_scale():
    """Scaling one token's row does not change another row's codes, scales or global
    scale (a batch-wide global scale would)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    c0, s0, g0 = A.quantize_activations(x)
    x2 = x.copy()
    x2[1] *= 1000.0
    c1, s1, g1 = A.quantize_activations(x2)
    for r in (0, 2, 3):
        assert np.array_equal(c0[r], c1[r]) and np.array_equal(s0[r], s1[r]) and g0[r] == g1[r]
    assert g1[1] != g0[1]


def test_power_of_two_row_scaling_scales_only_the_global_scale():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 96)).astype(np.float32)
    c0, s0, g0 = A.quantize_activations(x)
    c1, s1, g1 = A.quantize_activations(x * np.float32(32.0))
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
    assert np.array_equal(g1, g0 * np.float32(32.0))


def test_dequantized_activations_within_half_an_e2m1_step():
    """|x_hat - x| <= S * (half the E2M1 spacing at |x| / S), S = e4m3(scale) * g:
    0.25 below 2, 0.5 below 4, 1 above (which also covers a block whose scale
    rounded down and saturates at 6)."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((6, 256)) * np.exp(rng.standard_normal((6, 1)))).astype(np.float32)
    codes, scales, g = A.quantize_activations(x)
    xh = A.dequantize_activations(codes, scales, g)
    S = np.repeat(F.e4m3_value(scales), 16, axis=1) * g[:, None].astype(np.float64)
    r = np.abs(x.astype(np.float64)) / np.where(S == 0, 1.0, S)
    half = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0))
    assert np.all(np.abs(xh - x) <= half * S + 1e-30)
    assert np.any(xh != x)  # random data is not representable


def test_w4a4_gemm_matches_triple_loop():
    rng = np.random.default_rng(8)
    wq = F.quantize_matrix((0.02 * rng.standard_normal((12, 48))).astype(np.float32))
    xq = A.quantize_activations(rng.standard_normal((2, 48)).astype(np.float32))
    y, _, ya = A.w4a4_gemm(*wq, xq)
    w = F.dequantize_matrix(*wq)
    xv = F.e2m1_value(F.unpack_nibbles(xq[0]))
    xs = np.repeat(F.e4m3_value(xq[1]), 16, axis=1)
    for m in range(2):
        for n in range(12):
            s = a = 0.0
            for k in range(48):
                xk = float(xv[m, k]) * float(xs[m, k]) * float(xq[2][m])
                s += w[n, k] * xk
                a += abs(w[n, k] * xk)
            assert math.isclose(y[m, n], s, rel_tol=1e-13, abs_tol=1e-18)
            assert math.isclose(ya[m, n], a, rel_tol=1e-13, abs_tol=1e-18)


def test_zero_row_quantizes_to_zero():
    x = np.zeros((2, 32), np.float32)
    x[1, 3] = 1.5
    codes, scales, g = A.quantize_activations(x)
    assert g[0] == 0 and not codes[0].any() and not scales[0].any()
    assert g[1] == np.float32(1.5 / 2688.0)
