"""GPU parity of the W4A4 products (row f4): the activation quantizer bit-exact against
the oracle, the dense GEMM and the lm_head argmax on NVFP4 activations within the
bound of the exact product over both dequantized operands."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import lm_head as OLM
from oracle import w4a4 as A
from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
from tests.gpu_helpers import bf16_to_f64, check_bound, dev, oracle_quantize, upload_bf16, upload_oracle_weight

pytestmark = pytest.mark.gpu


def _quantize_both(lib, xb):
    """The GPU's NVFP4 activations and the oracle's, checked byte for byte."""
    xf = W.bf16_bits_to_f32(xb)
    got = lib.quantize_act(upload_bf16(xb))
    torch.cuda.synchronize()
    ref = A.quantize_activations(xf)
    assert np.array_equal(got[2].cpu().numpy(), ref[2]), "global scales differ"
    assert np.array_equal(got[1].cpu().numpy(), ref[1]), "scale codes differ"
    assert np.array_equal(got[0].cpu().numpy(), ref[0]), "element codes differ"
    return got, ref


@pytest.mark.parametrize("m,k", [(1, 64), (5, 2816), (15, 4096), (16, 512), (40, 256)])
def test_quantize_act_bit_exact(lib, m, k):
    xb, _ = W.activations((m, k), 5000 + m + k)
    _quantize_both(lib, xb)


def test_quantize_act_special_rows(lib):
    """A zero row (g = 0, zero codes), a row with planted E2M1 ties at g = 2^-10,
    negative values and a lone maximum."""
    m, k = 4, 64
    x = np.zeros((m, k), np.float32)
    x[1, 0] = 2688.0 * 2.0 ** -10
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32) * np.float32(2.0 ** -10)
    x[1, 16:32] = np.concatenate([ties, -ties])
    x[2] = -(np.arange(k, dtype=np.float32) / np.float32(16.0))
    x[3, 7] = 1.0
    xb = W.to_bf16_bits(x)
    assert np.array_equal(W.bf16_bits_to_f32(xb), x)
    got, ref = _quantize_both(lib, xb)
    assert ref[2][0] == 0 and not got[0][0].any().item()


@pytest.mark.parametrize("m", [1, 2, 5, 8, 9, 15, 16])
@pytest.mark.parametrize("n,k", [(40, 80), (1000, 320), (272, 1088)])
def test_gemm_w4a4_matches_oracle(lib, m, n, k):
    wq = oracle_quantize(W.weight((n, k), 6000 + n + k))
    xb, _ = W.activations((m, k), 7000 + m)
    got, ref = _quantize_both(lib, xb)
    y = lib.gemm_w4a4(upload_oracle_weight(lib, wq), got)
    torch.cuda.synchronize()
    exact, _, absy = A.w4a4_gemm(*wq, ref)
    check_bound(bf16_to_f64(y), exact, absy, True, f"w4a4 gemm m={m} n={n} k={k}")
    assert lib.device_error() == 0


@pytest.mark.parametrize("n", [4096, 14336])
@pytest.mark.parametrize("m", [1, 15])
def test_gemm_w4a4_full_size(lib, m, n):
    case = W.DenseCase.sweep(m, n)
    wq = oracle_quantize(case.w())
    xb, _ = case.x()
    got, ref = _quantize_both(lib, xb)
    y = lib.gemm_w4a4(upload_oracle_weight(lib, wq), got)
    torch.cuda.synchronize()
    exact, _, absy = A.w4a4_gemm(*wq, ref)
    check_bound(bf16_to_f64(y), exact, absy, True, f"w4a4 gemm full m={m} n={n}")
    assert lib.device_error() == 0


def _check_argmax(mx, idx, ref, nib, sc, g, xh, what):
    for t in range(len(idx)):
        lg, la = OLM.logits_rows(nib, sc, g, xh[t:t + 1], [idx[t], ref["argmax"][t]])
        tol = 1e-3 * max(la[0, 0], la[0, 1])
        if ref["max"][t] - ref["second"][t] > 2 * tol:
            assert idx[t] == ref["argmax"][t], f"{what}: token {t} argmax {idx[t]} != {ref['argmax'][t]}"
        else:
            assert ref["max"][t] - lg[0, 0] <= 2 * tol, f"{what}: token {t} near-tie row not maximal"
        assert abs(mx[t] - lg[0, 0]) <= tol, f"{what}: token {t} max logit {mx[t]} vs {lg[0, 0]}"


@pytest.mark.parametrize("m", [1, 7, 15, 16])
def test_lm_head_w4a4_small(lib, m):
    vocab, k = 3000, 512
    nib, sc, g = oracle_quantize(W.weight((vocab, k), 8100 + m))
    xb, _ = W.activations((m, k), 8200 + m)
    got, ref = _quantize_both(lib, xb)
    mx, idx = lib.lm_head_argmax_w4a4(upload_oracle_weight(lib, (nib, sc, g)), got)
    torch.cuda.synchronize()
    xh = A.dequantize_activations(*ref)
    r = OLM.lm_head_argmax(nib, sc, g, xh)
    _check_argmax(mx.cpu().numpy(), idx.cpu().numpy(), r, nib, sc, g, xh, f"w4a4 lm_head m={m}")
    assert lib.device_error() == 0


def test_lm_head_w4a4_full_size(lib):
    """The full 262,144 x 2,816 lm_head at M=15 on NVFP4 activations."""
    case = W.LMHeadCase(m=15)
    nib, sc, g = oracle_quantize(case.w_rows(0, case.vocab))
    xb, _ = case.x()
    got, ref = _quantize_both(lib, xb)
    mx, idx = lib.lm_head_argmax_w4a4(upload_oracle_weight(lib, (nib, sc, g)), got)
    torch.cuda.synchronize()
    xh = A.dequantize_activations(*ref)
    r = OLM.lm_head_argmax(nib, sc, g, xh, chunk_rows=16384)
    _check_argmax(mx.cpu().numpy(), idx.cpu().numpy(), r, nib, sc, g, xh, "w4a4 lm_head full")
    assert lib.device_error() == 0


def test_w4a4_rejects_bad_arguments(lib):
    """Host-side checks return before any launch: k % 16, more than 16 tokens."""
    from nvfp4_w4a16_moe_skinny_gb300.binding import NVFP4Error
    xb, _ = W.activations((3, 64), 1)
    with pytest.raises(NVFP4Error):
        lib.quantize_act(upload_bf16(xb)[:, :60].contiguous())
    wt = lib.prepare(torch.randn(64, 64, device=dev()) * 0.02)
    too_many = (torch.zeros((17, 32), dtype=torch.uint8, device=dev()),
                torch.zeros((17, 4), dtype=torch.uint8, device=dev()), torch.ones(17, device=dev()))
    with pytest.raises(NVFP4Error):
        lib.gemm_w4a4(wt, too_many)
    with pytest.raises(NVFP4Error):
        lib.lm_head_argmax_w4a4(wt, too_many)
