"""lm_head_argmax_noalloc: the lm_head entry point for callers that cannot allocate
device memory (it keeps its scratch in a static array of the library's device code).

It is compared, through the C ABI, with lm_head_argmax on the same inputs over two
calls in a row: the argmax indices must be identical and the max logits equal within
the tolerance the other lm_head tests use (they run the same kernel, so in practice
bit-identical).  This file sorts last so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
from oracle import formats as F
from oracle import lm_head as OLM
from tests.gpu_helpers import dev, upload_bf16, upload_f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,vocab,k", [(15, 8192, 2816), (1, 3000, 256), (16, 1037, 512)])
def test_noalloc_matches_lm_head_argmax_twice(lib, m, vocab, k):
    w = W.weight((vocab, k), W.seed_of("noalloc", vocab, k))
    xb, xf = W.activations((m, k), W.seed_of("noalloc-x", m, k))
    wt = lib.prepare(upload_f32(w))
    x = upload_bf16(xb)
    ref_max, ref_idx = lib.lm_head_argmax(wt, x)
    torch.cuda.synchronize()
    # the per-output bound of the lm_head tests: 1e-3 * sum_k |w_hat[n,k] x[m,k]| of the winning row
    nib, sc, g = F.quantize_matrix(w)
    tol = np.array([1e-3 * OLM.logits_rows(nib, sc, g, xf[t:t + 1].astype(np.float64), [int(ref_idx[t])])[1][0, 0]
                    for t in range(m)])
    cw = wt.c()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        mx = torch.full((m,), float("nan"), dtype=torch.float32, device=dev())
        idx = torch.full((m,), -1, dtype=torch.int32, device=dev())
        st = lib.lib.lm_head_argmax_noalloc(ctypes.byref(cw), x.data_ptr(), m, mx.data_ptr(), idx.data_ptr(), stream)
        assert st == 0, lib.lib.nvfp4_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert np.all(np.abs(mx.cpu().numpy().astype(np.float64) - ref_max.cpu().numpy()) <= tol)
    assert lib.device_error() == 0


def test_noalloc_rejects_bad_arguments(lib):
    w = W.weight((64, 64), 3)
    wt = lib.prepare(upload_f32(w))
    cw = wt.c()
    x = upload_bf16(W.activations((1, 64), 4)[0])
    out = torch.empty((17,), dtype=torch.float32, device=dev())
    idx = torch.empty((17,), dtype=torch.int32, device=dev())
    s = torch.cuda.current_stream().cuda_stream
    assert lib.lib.lm_head_argmax_noalloc(ctypes.byref(cw), x.data_ptr(), 17, out.data_ptr(), idx.data_ptr(), s) == 2
    assert lib.lib.lm_head_argmax_noalloc(ctypes.byref(cw), x.data_ptr(), 1, None, idx.data_ptr(), s) == 1
