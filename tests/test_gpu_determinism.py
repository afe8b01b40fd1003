"""Run-to-run determinism, a stand-in for a race detector (compute-sanitizer is not
available here): every cross-CTA reduction of the library -- the K-split fixup's
ticketed partial sums, the lm_head's packed-key argmax, the MoE grouping and the
fixed-order combine -- must give the same bytes on every repetition, with other
work in between that leaves the workspaces and counters in use."""

import pytest
import torch

from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu

REPS = 12


def _same(outs, what):
    ref = outs[0]
    for i, o in enumerate(outs[1:], 1):
        for a, b in zip(ref, o):
            assert torch.equal(a, b), f"{what}: repetition {i} differs"


@pytest.mark.parametrize("m,n,k", [(1, 4096, 4096), (15, 4096, 4096), (16, 14336, 4096), (3, 136, 32768)])
def test_dense_gemm_repeats_bit_exact(lib, m, n, k):
    g = torch.Generator(device=dev()).manual_seed(m * 7 + n)
    w = lib.prepare(torch.randn(n, k, generator=g, device=dev()) * 0.02)
    x = torch.randn(m, k, generator=g, device=dev()).to(torch.bfloat16)
    outs = []
    for _ in range(REPS):
        outs.append((lib.gemm(w, x).clone(),))
    torch.cuda.synchronize()
    _same(outs, f"gemm m={m} n={n} k={k}")
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [1, 15])
def test_lm_head_repeats_bit_exact(lib, m):
    g = torch.Generator(device=dev()).manual_seed(90 + m)
    w = lib.prepare(torch.randn(65536, 2816, generator=g, device=dev()) * 0.02)
    x = torch.randn(m, 2816, generator=g, device=dev()).to(torch.bfloat16)
    outs = []
    for _ in range(REPS):
        mx, idx = lib.lm_head_argmax(w, x)
        outs.append((mx.clone(), idx.clone()))
    torch.cuda.synchronize()
    _same(outs, f"lm_head m={m}")
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [1, 8, 15, 64])
def test_moe_layer_repeats_bit_exact(lib, m):
    """The layer through moe_forward, decode and prefill (m = 64: 32-pair blocks), with
    a dense GEMM between repetitions sharing the stream."""
    g = torch.Generator(device=dev()).manual_seed(300 + m)
    e, d, inter, k = 64, 1024, 256, 8
    gu = lib.prepare(torch.randn(e, 2 * inter, d, generator=g, device=dev()) * 0.02, gated=True)
    dn = lib.prepare(torch.randn(e, d, inter, generator=g, device=dev()) * 0.02)
    sgu = lib.prepare(torch.randn(2 * inter, d, generator=g, device=dev()) * 0.02, gated=True)
    sdn = lib.prepare(torch.randn(d, inter, generator=g, device=dev()) * 0.02)
    wd = lib.prepare(torch.randn(2048, d, generator=g, device=dev()) * 0.02)
    x = torch.randn(m, d, generator=g, device=dev()).to(torch.bfloat16)
    logits = torch.randn(m, e, generator=g, device=dev())
    outs = []
    for _ in range(REPS):
        y, (ids, probs, offs, pairs) = lib.moe_forward(x, logits, k, gu, dn, sgu, sdn)
        outs.append((y.clone(), ids.clone(), probs.clone(), offs.clone(), pairs.clone()))
        lib.gemm(wd, x[: min(m, 16)])
    torch.cuda.synchronize()
    _same(outs, f"moe m={m}")
    assert lib.device_error() == 0
