"""C-ABI checks that need no GPU: the library builds, loads, exports every function the
header declares, and its host-side size queries and argument checks behave as documented
(each rejected call returns before any CUDA call)."""

import ctypes
import os
import re

import numpy as np
import pytest

from nvfp4_w4a16_moe_skinny_gb300 import build as B
from oracle import layout as OL

HEADER = os.path.join(B.INCLUDE, "nvfp4_skinny.h")


@pytest.fixture(scope="module")
def so():
    B.build()
    from nvfp4_w4a16_moe_skinny_gb300 import binding
    lib = ctypes.CDLL(B.LIB)
    binding._sig(lib)
    return lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("nvfp4_gemm", "moe_route_topk", "moe_ffn_grouped", "lm_head_argmax", "nvfp4_repack", "nvfp4_quantize"):
        assert n in names


def test_library_exports_every_declared_function(so):
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing
    from nvfp4_w4a16_moe_skinny_gb300 import binding
    assert set(binding.EXPORTS) == set(declared_functions())


def test_status_strings_and_version(so):
    assert so.nvfp4_layout_version() == 2
    for code, text in [(0, b"ok"), (1, b"null pointer"), (2, b"bad shape"), (4, b"workspace missing or too small")]:
        assert so.nvfp4_status_string(code) == text


@pytest.mark.parametrize("n,k,e", [(16, 64, 1), (40, 80, 2), (262144, 2816, 1), (1408, 2816, 128), (1, 16, 1),
                                   (2816, 704, 128), (200, 320, 3)])
def test_repacked_bytes_matches_layout_spec(so, n, k, e):
    assert so.nvfp4_repacked_bytes(n, k, e) == OL.repacked_bytes(n, k, e)


def test_sizes_reject_bad_shapes(so):
    assert so.nvfp4_repacked_bytes(16, 24, 1) == 0          # k % 16
    assert so.nvfp4_repacked_bytes(0, 64, 1) == 0
    assert so.nvfp4_gemm_workspace_bytes(17, 64, 64) == 0   # m > 16
    assert so.lm_head_workspace_bytes(0, 100) == 0
    assert so.moe_ffn_workspace_bytes(4097, 1, 128, 2816, 704) == 0      # m > 4096
    assert so.moe_ffn_workspace_bytes(2049, 8, 128, 2816, 704) == 0      # m * top_k > 16384
    # a prefill chunk (m > 16) is planned like decode, one 16-token block per segment
    assert so.moe_ffn_workspace_bytes(512, 8, 128, 2816, 704) >= (512 * 8 + 512) * (704 * 2 + 2816 * 4)
    # h (bf16) and the per-(token, slot) down outputs (fp32) are always part of it
    assert so.moe_ffn_workspace_bytes(15, 8, 128, 2816, 704) >= (15 * 8 + 15) * (704 * 2 + 2816 * 4)
    # the fixed 512 KiB counter area leads every MoE workspace, whatever the split
    assert so.moe_ffn_workspace_bytes(1, 1, 8, 64, 64) >= 512 * 1024 + 2 * (64 * 2 + 64 * 4)


def _weight(data=1 << 20, gs=1 << 20, n=64, k=64, e=1, flags=0, version=2):
    from nvfp4_w4a16_moe_skinny_gb300.binding import CWeight
    return CWeight(data, gs, n, k, e, flags, version)


def test_gemm_argument_errors_return_before_any_launch(so):
    ws = ctypes.c_void_p(1 << 20)
    x, y = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 20)
    assert so.nvfp4_gemm(None, x, 1, y, ws, 1 << 20, None) == 1
    w = _weight(data=0)
    assert so.nvfp4_gemm(ctypes.byref(w), x, 1, y, ws, 1 << 20, None) == 1
    w = _weight(version=1)                            # weights repacked in the old tile order
    assert so.nvfp4_gemm(ctypes.byref(w), x, 1, y, ws, 1 << 20, None) == 5
    w = _weight(flags=1)
    assert so.nvfp4_gemm(ctypes.byref(w), x, 1, y, ws, 1 << 20, None) == 5
    w = _weight(k=72)
    assert so.nvfp4_gemm(ctypes.byref(w), x, 1, y, ws, 1 << 20, None) == 2
    w = _weight()
    assert so.nvfp4_gemm(ctypes.byref(w), x, 0, y, ws, 1 << 20, None) == 2
    assert so.nvfp4_gemm(ctypes.byref(w), x, 17, y, ws, 1 << 20, None) == 2
    assert so.nvfp4_gemm(ctypes.byref(w), ctypes.c_void_p((1 << 20) + 8), 1, y, ws, 1 << 20, None) == 3
    assert so.nvfp4_gemm(ctypes.byref(w), x, 1, y, None, 1 << 20, None) == 4
    big = _weight(n=4096, k=4096)                     # small N splits K: the fixup area is needed
    need = so.nvfp4_gemm_workspace_bytes(16, 4096, 4096)
    assert need > 256 * 1024                          # the fixed counter area and the partials
    assert so.nvfp4_gemm(ctypes.byref(big), x, 16, y, ws, need - 1, None) == 4
    w = _weight(data=(1 << 20) + 4)
    assert so.nvfp4_gemm(ctypes.byref(w), x, 1, y, ws, 1 << 20, None) == 3


def test_lm_head_and_moe_argument_errors(so):
    p = ctypes.c_void_p(1 << 20)
    w = _weight()
    assert so.lm_head_argmax(ctypes.byref(w), p, 1, None, p, p, 1 << 20, None) == 1
    assert so.lm_head_argmax(ctypes.byref(w), p, 17, p, p, p, 1 << 20, None) == 2
    assert so.lm_head_argmax(ctypes.byref(w), p, 1, p, p, p, 8, None) == 4
    # the sampling lm_head: the same checks, and the temperature must be finite and >= 0
    assert so.lm_head_sample(ctypes.byref(w), p, 1, 1.0, 7, None, p, p, 1 << 20, None) == 1
    assert so.lm_head_sample(ctypes.byref(w), p, 17, 1.0, 7, p, p, p, 1 << 20, None) == 2
    assert so.lm_head_sample(ctypes.byref(w), p, 1, -0.5, 7, p, p, p, 1 << 20, None) == 2
    assert so.lm_head_sample(ctypes.byref(w), p, 1, float("nan"), 7, p, p, p, 1 << 20, None) == 2
    assert so.lm_head_sample(ctypes.byref(w), p, 1, float("inf"), 7, p, p, p, 1 << 20, None) == 2
    assert so.lm_head_sample(ctypes.byref(w), p, 1, 1.0, 7, p, p, p, 8, None) == 4
    # the softcapped sampling lm_head: the cap must be finite and >= 0
    assert so.lm_head_sample_ex(ctypes.byref(w), p, 1, -1.0, 1.0, 7, p, p, p, 1 << 20, None) == 2
    assert so.lm_head_sample_ex(ctypes.byref(w), p, 1, float("inf"), 1.0, 7, p, p, p, 1 << 20, None) == 2
    assert so.lm_head_sample_ex(ctypes.byref(w), p, 1, 30.0, 1.0, 7, None, p, p, 1 << 20, None) == 1
    # the router logits: m <= 16, eps >= 0, the GEMM's workspace
    assert so.moe_router_logits(ctypes.byref(w), p, 17, None, 1e-6, p, p, 1 << 20, None) == 2
    assert so.moe_router_logits(ctypes.byref(w), p, 1, None, -1.0, p, p, 1 << 20, None) == 2
    assert so.moe_router_logits(ctypes.byref(w), None, 1, None, 1e-6, p, p, 1 << 20, None) == 1
    assert so.moe_router_logits(ctypes.byref(w), p, 1, None, 1e-6, p, p, 8, None) == 4
    assert so.moe_route_topk(p, 15, 128, 0, p, p, p, p, None) == 2           # top_k < 1
    assert so.moe_route_topk(p, 15, 4, 8, p, p, p, p, None) == 2             # top_k > n_experts
    assert so.moe_route_topk(p, 15, 2048, 8, p, p, p, p, None) == 2          # n_experts > 1024
    assert so.moe_route_topk(None, 15, 128, 8, p, p, p, p, None) == 1
    gu = _weight(n=1408, k=2816, e=128, flags=1)
    dn = _weight(n=2816, k=704, e=128)
    args = [p, 15, 8, p, p, p, ctypes.byref(gu), ctypes.byref(dn), None, None, p, p, 1 << 30, None]
    bad = list(args)
    bad[7] = ctypes.byref(_weight(n=2816, k=704, e=64))                    # expert count mismatch
    assert so.moe_ffn_grouped(*bad) == 2
    bad = list(args)
    bad[6] = ctypes.byref(_weight(n=1408, k=2816, e=128, flags=0))         # gate_up must be gated
    assert so.moe_ffn_grouped(*bad) == 5
    bad = list(args)
    bad[8] = ctypes.byref(_weight(n=1408, k=2816, flags=1))                # shared gate_up without down
    assert so.moe_ffn_grouped(*bad) == 1
    bad = list(args)
    bad[12] = 1024                                                          # workspace too small
    assert so.moe_ffn_grouped(*bad) == 4
    bad = list(args)                                                        # d and I must be multiples of 64
    bad[6], bad[7] = ctypes.byref(_weight(n=192, k=208, e=128, flags=1)), ctypes.byref(_weight(n=208, k=96, e=128))
    assert so.moe_ffn_grouped(*bad) == 2


def test_binding_refuses_to_run_without_the_library(tmp_path):
    from nvfp4_w4a16_moe_skinny_gb300 import binding
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.Library(str(tmp_path / "missing.so"))


def _host_repack(so, nib, sc, gated):
    e, n, kh = nib.shape
    k = 2 * kh
    out = (ctypes.c_uint8 * OL.repacked_bytes(n, k, e))()
    nib = np.ascontiguousarray(nib)
    sc = np.ascontiguousarray(sc)
    st = so.nvfp4_repack_host(nib.ctypes.data, sc.ctypes.data, e, n, k, 1 if gated else 0, out, len(out))
    assert st == 0
    return np.frombuffer(out, dtype=np.uint8)


@pytest.mark.parametrize("e,n,k,gated", [(1, 16, 64, False), (2, 40, 80, False), (1, 1000, 320, False),
                                         (3, 64, 128, True), (2, 128, 16, True), (1, 192, 704, True)])
def test_host_repack_matches_the_layout_definition(so, e, n, k, gated):
    """The host repack (host bytes in, host bytes out) against the oracle's index
    function of the layout, byte for byte, including the zero padding."""
    rng = np.random.default_rng(n * 5 + k)
    nib = rng.integers(0, 256, (e, n, k // 2), dtype=np.uint8)
    sc = rng.integers(0, 127, (e, n, k // 16), dtype=np.uint8)
    assert np.array_equal(_host_repack(so, nib, sc, gated), OL.repack(nib, sc, gated))


def test_host_repack_folds_negative_scales(so):
    """A scale byte with bit 7 set is stored positive and its 16 codes change sign:
    the dequantized matrix is unchanged."""
    from oracle import formats as F
    rng = np.random.default_rng(6)
    n, k = 48, 128
    nib = rng.integers(0, 256, (1, n, k // 2), dtype=np.uint8)
    sc = rng.integers(1, 127, (1, n, k // 16), dtype=np.uint8)
    sc[0, ::3, 1] |= 0x80
    nib2, sc2 = OL.unrepack(_host_repack(so, nib, sc, False), n, k)
    assert not (sc2 & 0x80).any()
    assert np.array_equal(F.dequantize_matrix(nib2[0], sc2[0], 1.0), F.dequantize_matrix(nib[0], sc[0], 1.0))


def test_host_repack_rejects_bad_arguments(so):
    buf = (ctypes.c_uint8 * 64)()
    small = (ctypes.c_uint8 * 16)()
    assert so.nvfp4_repack_host(None, buf, 1, 16, 64, 0, buf, 64) == 1                    # null
    assert so.nvfp4_repack_host(buf, buf, 1, 16, 60, 0, buf, 64) != 0                     # k % 16
    assert so.nvfp4_repack_host(buf, buf, 1, 40, 64, 1, buf, 64) != 0                     # gated n % 64
    assert so.nvfp4_repack_host(buf, buf, 1, 16, 64, 4, buf, 64) != 0                     # unknown flag
    assert so.nvfp4_repack_host(buf, buf, 1, 16, 64, 0, small, 16) != 0                   # out too small


def test_w4a4_calls_reject_bad_arguments_before_launch(so):
    buf = (ctypes.c_uint8 * 256)()
    ws = (ctypes.c_uint8 * 256)()
    assert so.nvfp4_quantize_act(None, 2, 64, buf, buf, buf, ws, 256, None) == 1           # null x
    assert so.nvfp4_quantize_act(buf, 2, 60, buf, buf, buf, ws, 256, None) != 0            # k % 16
    assert so.nvfp4_quantize_act(buf, 5000, 64, buf, buf, buf, ws, 256, None) != 0         # m > 4096
    assert so.nvfp4_quantize_act(buf, 2, 64, buf, buf, buf, ws, 0, None) != 0              # workspace


def test_moe_forward_checks_both_steps_before_launch(so):
    """moe_forward returns the router's and the FFN's argument errors before its first
    launch: a null logits or ids pointer, an FFN shape error, a bad top_k, a small
    workspace."""
    p = ctypes.c_void_p(1 << 20)
    gu = _weight(n=1408, k=2816, e=128, flags=1)
    dn = _weight(n=2816, k=704, e=128)
    # x, logits, m, top_k, flags, scale, ids, probs, offsets, pairs, gate_up, down, sh_gu, sh_dn, out, ws, bytes, stream
    args = [p, p, 15, 8, 0, None, p, p, p, p, ctypes.byref(gu), ctypes.byref(dn), None, None, p, p, 1 << 30, None]

    def call(i, v):
        bad = list(args)
        bad[i] = v
        return so.moe_forward(*bad)
    assert call(1, None) == 1                                                  # null logits
    assert call(6, None) == 1                                                  # null ids
    assert call(0, None) == 1                                                  # null x
    assert call(11, ctypes.byref(_weight(n=2816, k=704, e=64))) == 2          # expert count mismatch
    assert call(3, 0) == 2                                                     # top_k < 1
    assert call(3, 33) == 2                                                    # top_k > 32
    assert call(16, 1024) == 4                                                 # workspace too small


def test_selftest_rejects_a_limit_out_of_range_before_launch(so):
    assert so.nvfp4_selftest_wait_timeout(0, None) == 2
    assert so.nvfp4_selftest_wait_timeout(-5, None) == 2
    assert so.nvfp4_selftest_wait_timeout((1 << 31) + 1, None) == 2
