"""NVFP4 codecs and the offline quantizer (oracle; test infrastructure only).

Format (gemma-cuda-hybrid README, "Everything it has / Inference engine":
"E2M1 weights + E4M3 group-16 scales + FP32 global"; and "Why it's
NVIDIA-only ... / NVFP4-specific": "E2M1 + E4M3-block-scale + FP32-global
dequant, ... the group-16 scale handling"):

    w_hat[n, k] = e2m1(q[n, k]) * e4m3(s[n, k // 16]) * g

Readings where the pages are silent:

* E2M1 code c = sign<<3 | exp<<1 | man, bias 1, one subnormal (0.5), no
  inf/NaN, so the magnitudes are {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E4M3 is the "fn" variant: bias 7, subnormals m/8 * 2^-6, max 448, codes
  0x7F/0xFF are NaN, no infinities.
* Global scale g = fp32(amax / (448 * 6)) is the dequant multiplier: an FP32
  number, the correctly rounded quotient.
* Block scale code = E4M3 round-to-nearest-even, saturating at 448, of the
  exact quotient t = bmax / (6 g); element code = E2M1 round-to-nearest-even,
  saturating at 6, of the exact quotient v = w / (e4m3(scale) * g).  Both are
  computed as one float64 division whose divisor (6 g, or e4m3(scale) * g, at
  most 28 significant bits) is exact.  The grids' midpoints have at most 5
  significant bits, and a quotient of fp32 values that is not a midpoint lies
  at least 2^-32 (relative) away from every midpoint, far beyond the 2^-53 of
  one float64 rounding: so the rounded quotient takes the same code decision
  as the exact real one.
* A block whose scale decodes to 0 gets all-zero codes (no division).
* An all-zero matrix gets g = 0 and all-zero codes and scales.
* Canonical packing: element 2i in the low nibble, 2i+1 in the high nibble of
  byte i along K; row-major [N, K/2] nibbles and [N, K/16] scales.
"""

from __future__ import annotations

import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0


# --------------------------------------------------------------------------- decode

def e2m1_value(code) -> np.ndarray:
    """Value of a 4-bit E2M1 code (array-friendly), from the bit fields."""
    c = np.asarray(code, dtype=np.int64) & 0xF
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m * 0.5, (e - 1).astype(np.int64)))
    return sign * mag


def e4m3_value(code) -> np.ndarray:
    """Value of an 8-bit E4M3 ("fn") code; 0x7F and 0xFF decode to NaN."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = (m / 8.0) * 2.0 ** -6
    nrm = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    mag = np.where(e == 0, sub, nrm)
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# --------------------------------------------------------------------------- encode

def e4m3_encode_nonneg(t) -> np.ndarray:
    """Round non-negative finite values to the E4M3 grid, ties to even, saturate at 448.

    Exact for the float64 value given: scaling by a power of two is exact and
    ``np.rint`` rounds half to even, so the code is the RNE code of that value.
    """
    t = np.minimum(np.asarray(t, dtype=np.float64), E4M3_MAX)
    code = np.zeros(t.shape, dtype=np.int64)
    small = t < 2.0 ** -6
    # subnormal range: units of 2^-9; a result of 8 is the smallest normal (code 8)
    code[small] = np.rint(t[small] * 2.0 ** 9).astype(np.int64)
    big = ~small
    if np.any(big):
        tb = t[big]
        _, ex = np.frexp(tb)                 # tb = f * 2^ex, f in [0.5, 1)
        e = ex.astype(np.int64) - 1          # tb in [2^e, 2^(e+1))
        q = np.rint(np.ldexp(tb, 3 - e))     # mantissa in units of 2^(e-3): [8, 16]
        carry = q >= 16
        e = np.where(carry, e + 1, e)
        q = np.where(carry, 8, q)
        code[big] = ((e + 7) << 3) | (q.astype(np.int64) - 8)
    return code.astype(np.uint8)


def e2m1_encode(v) -> np.ndarray:
    """Round finite values to the E2M1 grid, ties to even, saturate at +-6; keeps the sign bit.

    The magnitude code is the number of grid midpoints below |v|: midpoint i lies
    between magnitude codes i and i + 1 and counts when |v| exceeds it, or equals
    it and code i + 1 is even (round half to even).  Past the last midpoint the
    code is 7 (6.0), which is the saturation.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    mags = e2m1_value(np.arange(8))
    code = np.zeros(a.shape, dtype=np.uint8)
    for i in range(7):
        mid = (mags[i] + mags[i + 1]) / 2
        if (i + 1) % 2 == 0:
            code += a >= mid
        else:
            code += a > mid
    code |= np.signbit(v).astype(np.uint8) << 3
    return code


# --------------------------------------------------------------------------- quantizer

def global_scale(w: np.ndarray) -> np.float32:
    """g = fp32(amax|W|) / fp32(448 * 6), one IEEE fp32 division."""
    amax = np.float32(np.max(np.abs(w.astype(np.float32)))) if w.size else np.float32(0)
    return np.float32(amax / np.float32(E4M3_MAX * E2M1_MAX))


def quantize_matrix(w: np.ndarray, chunk_rows: int = 4096):
    """Quantize one fp32 matrix [N, K] (K % 16 == 0) to canonical NVFP4.

    Returns (nibbles uint8 [N, K/2], scales uint8 [N, K/16], g float32).  Rows are
    processed in chunks only to bound host memory; every row is independent once
    g is known.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    if k % 16:
        raise ValueError("K must be a multiple of 16")
    g = global_scale(w)
    if g == 0:
        return (np.zeros((n, k // 2), np.uint8), np.zeros((n, k // 16), np.uint8), np.float32(0))
    nib = np.empty((n, k // 2), np.uint8)
    sc = np.empty((n, k // 16), np.uint8)
    for lo in range(0, n, chunk_rows):
        hi = min(n, lo + chunk_rows)
        nib[lo:hi], sc[lo:hi] = _quantize_rows(w[lo:hi], g)
    return nib, sc, g


def _quantize_rows(w: np.ndarray, g: np.float32):
    n, k = w.shape
    g64 = np.float64(g)
    blocks = w.astype(np.float64).reshape(n, k // 16, 16)
    bmax = np.max(np.abs(blocks), axis=2)
    t = bmax / (E2M1_MAX * g64)                     # exact divisor; decision = the exact quotient's
    s_code = e4m3_encode_nonneg(t)
    s_val = e4m3_value(s_code)
    denom = s_val * g64                             # exact (at most 28 significant bits)
    safe = np.where(denom == 0, 1.0, denom)
    v = blocks / safe[:, :, None]
    q = e2m1_encode(v)
    q = np.where((s_val == 0)[:, :, None], np.uint8(0), q).reshape(n, k)
    nib = (q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)
    return nib.astype(np.uint8), s_code.reshape(n, k // 16)


def quantize_stack(w: np.ndarray):
    """Quantize stacked matrices [E, N, K]; one global scale per matrix."""
    outs = [quantize_matrix(w[e]) for e in range(w.shape[0])]
    nib = np.stack([o[0] for o in outs])
    sc = np.stack([o[1] for o in outs])
    g = np.array([o[2] for o in outs], dtype=np.float32)
    return nib, sc, g


def unpack_nibbles(nib: np.ndarray) -> np.ndarray:
    """Canonical [.., N, K/2] bytes -> [.., N, K] codes (low nibble first)."""
    lo = nib & 0xF
    hi = (nib >> 4) & 0xF
    out = np.empty(nib.shape[:-1] + (nib.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def dequantize_matrix(nib: np.ndarray, scales: np.ndarray, g) -> np.ndarray:
    """w_hat = e2m1(q) * e4m3(s) * g in float64 (exact: at most 30 significant bits)."""
    q = unpack_nibbles(nib)
    n, k = q.shape
    wq = e2m1_value(q).reshape(n, k // 16, 16)
    s = e4m3_value(scales)[:, :, None]
    return (wq * s * np.float64(g)).reshape(n, k)


def bf16_round(x) -> np.ndarray:
    """Round values to bf16 (round to nearest, ties to even) and return them as float64.

    Used where the method itself rounds to bf16 (the GEMM and MoE outputs, and
    the A16 intermediate of the expert FFN).  The exact float64 value is rounded
    once to 8 significant bits; inputs are finite and inside bf16's normal range.
    """
    x64 = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x64)                          # x = m * 2^e, |m| in [0.5, 1)
    r = np.rint(np.ldexp(m, 8))                   # 8 significant bits, ties to even
    out = np.ldexp(r, (e - 8).astype(np.int64))
    return np.where(np.isfinite(x64), out, x64)
