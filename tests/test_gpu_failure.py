"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up after its limit, records bit 0 of the device error word and
returns; the host reads and clears the word, and the same context then runs a
product that matches the oracle."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as OG
from nvfp4_w4a16_moe_skinny_gb300 import workloads as W
from tests.gpu_helpers import bf16_to_f64, check_bound, upload_bf16, upload_oracle_weight

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit", [200_000, 4_000_000])
def test_bounded_wait_runs_out_reports_and_the_context_survives(lib, limit):
    assert lib.device_error(clear=True) == 0
    lib.selftest_wait_timeout(limit)
    torch.cuda.synchronize()
    assert lib.device_error(clear=False) & 1, "the wait ran out but the device error word shows nothing"
    lib.device_error(clear=True)
    assert lib.device_error() == 0
    # the context is still usable: a ragged GEMM on the oracle's bytes
    m, n, k = 3, 272, 1088
    w = W.weight((n, k), 31337)
    xb, _ = W.activations((m, k), 4711)
    nib, sc, g = F.quantize_matrix(w)
    y = lib.gemm(upload_oracle_weight(lib, (nib, sc, g)), upload_bf16(xb))
    torch.cuda.synchronize()
    exact, _, absy = OG.nvfp4_gemm(nib, sc, g, W.bf16_bits_to_f32(xb).astype(np.float64))
    check_bound(bf16_to_f64(y), exact, absy, True, "gemm after a timed-out wait")
    assert lib.device_error() == 0
