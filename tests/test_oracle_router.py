"""Pins of the router-normalisation and softcap oracle (CPU): closed forms and the
defining properties of an unweighted RMSNorm and of a tanh softcap, and the router
logits against the RMSNorm of a plain product."""

import numpy as np
import pytest

from oracle import formats as F
from oracle import router as OR


def test_rmsnorm_closed_forms():
    v = np.array([[3.0, 4.0]])                         # mean square 12.5
    assert np.allclose(OR.rmsnorm_unweighted(v, 0.0), v / np.sqrt(12.5), rtol=1e-15)
    out = OR.rmsnorm_unweighted(v)                     # with eps: mean(out^2) = ms / (ms + eps)
    assert np.mean(out ** 2) == pytest.approx(12.5 / (12.5 + 1e-6), rel=1e-14)
    rng = np.random.default_rng(4)
    w = rng.standard_normal((3, 128))
    assert np.allclose(OR.rmsnorm_unweighted(7.5 * w, 0.0), OR.rmsnorm_unweighted(w, 0.0), rtol=1e-13)
    assert np.array_equal(np.sign(OR.rmsnorm_unweighted(w)), np.sign(w))
    assert np.allclose(OR.rmsnorm_unweighted(np.zeros((1, 4))), 0.0)   # eps keeps a zero row finite


def test_softcap_properties():
    cap = 30.0
    assert OR.softcap(np.array([cap * np.arctanh(0.5)]), cap)[0] == pytest.approx(15.0, rel=1e-14)
    grid = np.linspace(-200, 200, 4001)
    s = OR.softcap(grid, cap)
    assert np.all(np.abs(s) < cap)                     # bounded by the cap
    assert np.all(np.diff(s) > 0)                      # monotone: the argmax is unchanged
    assert np.allclose(s, -OR.softcap(-grid, cap))     # odd
    assert OR.softcap(np.array([1e-4]), cap)[0] == pytest.approx(1e-4, rel=1e-8)   # slope 1 at 0
    assert np.array_equal(OR.softcap(grid, 0.0), grid)  # cap <= 0: off


def test_router_logits_match_rmsnorm_of_the_product():
    rng = np.random.default_rng(5)
    w = (0.02 * rng.standard_normal((128, 256))).astype(np.float32)
    nib, sc, g = F.quantize_matrix(w)
    x = rng.standard_normal((4, 256))
    scale = 0.5 + rng.random(128)
    raw = x @ F.dequantize_matrix(nib, sc, g).T
    ms = np.mean(raw ** 2, axis=1, keepdims=True)
    ref = raw / np.sqrt(ms + 1e-6) * scale
    assert np.allclose(OR.router_logits(x, nib, sc, g, scale), ref, rtol=1e-13)
    # one-hot rows pick single activations: the logits are those entries, normalised
    x1 = np.zeros((1, 256))
    x1[0, :128] = rng.standard_normal(128)
    eye = np.zeros((128, 256), np.float32)
    eye[np.arange(128), np.arange(128)] = 1.0
    n1, s1, g1 = F.quantize_matrix(eye)
    got = OR.router_logits(x1, n1, s1, g1, np.ones(128))
    assert np.allclose(got, OR.rmsnorm_unweighted(x1[:, :128]), rtol=1e-12)
