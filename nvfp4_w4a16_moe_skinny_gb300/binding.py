"""Thin Python binding over the C ABI of ``libnvfp4skinny.so`` (ctypes).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  There is
no fallback: if the shared library is missing, ``load()`` raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

from .build import LIB

NVFP4_GATED = 1
NVFP4_ROUTE_SOFTMAX_ALL = 1
LAYOUT_VERSION = 2

STATUS = {0: "ok", 1: "null pointer", 2: "bad shape", 3: "misaligned pointer",
          4: "workspace missing or too small", 5: "weight layout version or flags mismatch", 6: "CUDA error"}

EXPORTS = (
    "nvfp4_status_string", "nvfp4_layout_version", "nvfp4_device_error", "nvfp4_repacked_bytes",
    "nvfp4_quantize_workspace_bytes", "nvfp4_quantize", "nvfp4_repack", "nvfp4_gemm_workspace_bytes",
    "nvfp4_gemm", "moe_route_topk", "moe_ffn_workspace_bytes", "moe_ffn_grouped",
    "lm_head_workspace_bytes", "lm_head_argmax", "lm_head_argmax_noalloc", "nvfp4_plan_info",
    "lm_head_sample", "moe_route_topk_ex", "lm_head_sample_ex", "nvfp4_plan_check", "moe_router_logits",
    "nvfp4_repack_host", "nvfp4_quantize_act", "nvfp4_gemm_w4a4", "lm_head_argmax_w4a4", "moe_forward", "nvfp4_selftest_wait_timeout",
)


class NVFP4Error(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} failed: {STATUS.get(status, status)} ({status})")
        self.status = status


class CWeight(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("global_scale", ctypes.c_void_p), ("n", ctypes.c_int32),
                ("k", ctypes.c_int32), ("num_matrices", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("layout_version", ctypes.c_uint32)]


@dataclass
class Weight:
    """A repacked NVFP4 weight living on the GPU (owns its tensors)."""
    data: torch.Tensor          # uint8, repacked tiles
    global_scale: torch.Tensor  # float32 [num_matrices]
    n: int
    k: int
    num_matrices: int = 1
    flags: int = 0

    def c(self) -> CWeight:
        return CWeight(self.data.data_ptr(), self.global_scale.data_ptr(), self.n, self.k,
                       self.num_matrices, self.flags, LAYOUT_VERSION)

    @property
    def nbytes_algorithmic(self) -> int:
        """Bytes the method must read: n*k/2 nibbles + n*k/16 scales per matrix."""
        return self.num_matrices * (self.n * self.k // 2 + self.n * self.k // 16)


_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t


def _sig(lib):
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    lib.nvfp4_status_string.argtypes = [ctypes.c_int]
    lib.nvfp4_layout_version.restype = ctypes.c_uint32
    lib.nvfp4_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), _I]
    lib.nvfp4_repacked_bytes.restype = _SZ
    lib.nvfp4_repacked_bytes.argtypes = [_I, _I, _I]
    lib.nvfp4_quantize_workspace_bytes.restype = _SZ
    lib.nvfp4_quantize_workspace_bytes.argtypes = [_I]
    lib.nvfp4_quantize.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]
    lib.nvfp4_repack.argtypes = [_P, _P, _I, _I, _I, ctypes.c_uint32, _P, _P]
    lib.nvfp4_gemm_workspace_bytes.restype = _SZ
    lib.nvfp4_gemm_workspace_bytes.argtypes = [_I, _I, _I]
    lib.nvfp4_gemm.argtypes = [ctypes.POINTER(CWeight), _P, _I, _P, _P, _SZ, _P]
    lib.moe_route_topk.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P]
    lib.moe_route_topk_ex.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
    lib.moe_route_topk_ex.restype = ctypes.c_int
    lib.moe_ffn_workspace_bytes.restype = _SZ
    lib.moe_ffn_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
    lib.moe_ffn_grouped.argtypes = [_P, _I, _I, _P, _P, _P, ctypes.POINTER(CWeight), ctypes.POINTER(CWeight),
                                    ctypes.POINTER(CWeight), ctypes.POINTER(CWeight), _P, _P, _SZ, _P]
    lib.lm_head_workspace_bytes.restype = _SZ
    lib.lm_head_workspace_bytes.argtypes = [_I, _I]
    lib.lm_head_argmax.argtypes = [ctypes.POINTER(CWeight), _P, _I, _P, _P, _P, _SZ, _P]
    lib.lm_head_argmax_noalloc.argtypes = [ctypes.POINTER(CWeight), _P, _I, _P, _P, _P]
    lib.lm_head_sample.argtypes = [ctypes.POINTER(CWeight), _P, _I, ctypes.c_float, ctypes.c_uint64, _P, _P, _P, _SZ,
                                   _P]
    lib.lm_head_sample.restype = ctypes.c_int
    lib.nvfp4_plan_info.argtypes = [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int32), _I]
    lib.nvfp4_plan_info.restype = ctypes.c_int
    lib.nvfp4_plan_check.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int32), _I]
    lib.nvfp4_plan_check.restype = ctypes.c_int
    lib.lm_head_sample_ex.argtypes = [ctypes.POINTER(CWeight), _P, _I, ctypes.c_float, ctypes.c_float, ctypes.c_uint64,
                                      _P, _P, _P, _SZ, _P]
    lib.lm_head_sample_ex.restype = ctypes.c_int
    lib.moe_router_logits.argtypes = [ctypes.POINTER(CWeight), _P, _I, _P, ctypes.c_float, _P, _P, _SZ, _P]
    lib.moe_router_logits.restype = ctypes.c_int
    lib.moe_forward.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, ctypes.POINTER(CWeight),
                                ctypes.POINTER(CWeight), ctypes.POINTER(CWeight), ctypes.POINTER(CWeight), _P, _P, _SZ,
                                _P]
    lib.moe_forward.restype = ctypes.c_int
    lib.nvfp4_selftest_wait_timeout.argtypes = [ctypes.c_int64, _P]
    lib.nvfp4_selftest_wait_timeout.restype = ctypes.c_int
    lib.nvfp4_quantize_act.argtypes = [_P, _I, _I, _P, _P, _P, _P, _SZ, _P]
    lib.nvfp4_quantize_act.restype = ctypes.c_int
    lib.nvfp4_gemm_w4a4.argtypes = [ctypes.POINTER(CWeight), _P, _P, _P, _I, _P, _P, _SZ, _P]
    lib.nvfp4_gemm_w4a4.restype = ctypes.c_int
    lib.lm_head_argmax_w4a4.argtypes = [ctypes.POINTER(CWeight), _P, _P, _P, _I, _P, _P, _P, _SZ, _P]
    lib.lm_head_argmax_w4a4.restype = ctypes.c_int
    lib.nvfp4_repack_host.argtypes = [_P, _P, _I, _I, _I, ctypes.c_uint32, _P, _SZ]
    lib.nvfp4_repack_host.restype = ctypes.c_int
    for name in ("nvfp4_quantize", "nvfp4_repack", "nvfp4_gemm", "moe_route_topk", "moe_ffn_grouped",
                 "lm_head_argmax", "lm_head_argmax_noalloc", "nvfp4_device_error"):
        getattr(lib, name).restype = ctypes.c_int


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


class Library:
    """The loaded C ABI; methods take CUDA tensors and enqueue on the current stream."""

    def __init__(self, path: str = LIB):
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m nvfp4_w4a16_moe_skinny_gb300.build` "
                               "(there is no CPU fallback)")
        self.path = path
        self.lib = ctypes.CDLL(path)
        _sig(self.lib)
        self._ws = {}

    # -------------------------------------------------------------- plumbing
    def _check(self, call, st):
        if st != 0:
            raise NVFP4Error(call, st)

    def workspace(self, key, nbytes: int, device) -> torch.Tensor:
        """A per-(call kind, device) workspace, zero-filled once at allocation."""
        cur = self._ws.get((key, device))
        if cur is None or cur.numel() < nbytes:
            cur = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)
            self._ws[(key, device)] = cur
        return cur

    def device_error(self, clear: bool = True) -> int:
        v = ctypes.c_uint32(0)
        self._check("nvfp4_device_error", self.lib.nvfp4_device_error(ctypes.byref(v), int(clear)))
        return v.value

    def selftest_wait_timeout(self, limit_cycles: int, stream=None):
        """Run the bounded-wait self-test (a wait that runs out after limit_cycles)."""
        self._check("nvfp4_selftest_wait_timeout", self.lib.nvfp4_selftest_wait_timeout(int(limit_cycles),
                                                                                        _stream(stream)))

    def repacked_bytes(self, n, k, num_matrices=1) -> int:
        return self.lib.nvfp4_repacked_bytes(n, k, num_matrices)

    # -------------------------------------------------------------- offline
    def quantize(self, w: torch.Tensor, stream=None):
        """fp32 [E, n, k] or [n, k] on the GPU -> canonical (nibbles, scales, global_scale)."""
        squeeze = w.dim() == 2
        w3 = w.unsqueeze(0) if squeeze else w
        w3 = w3.contiguous()
        e, n, k = w3.shape
        nib = torch.empty((e, n, k // 2), dtype=torch.uint8, device=w.device)
        sc = torch.empty((e, n, k // 16), dtype=torch.uint8, device=w.device)
        g = torch.empty((e,), dtype=torch.float32, device=w.device)
        ws = torch.empty((max(1, self.lib.nvfp4_quantize_workspace_bytes(e)),), dtype=torch.uint8, device=w.device)
        self._check("nvfp4_quantize", self.lib.nvfp4_quantize(
            w3.data_ptr(), e, n, k, nib.data_ptr(), sc.data_ptr(), g.data_ptr(), ws.data_ptr(), ws.numel(),
            _stream(stream)))
        if squeeze:
            return nib[0], sc[0], g
        return nib, sc, g

    def repack(self, nib: torch.Tensor, sc: torch.Tensor, gscale: torch.Tensor, gated: bool = False,
               stream=None) -> Weight:
        nib3 = nib.unsqueeze(0) if nib.dim() == 2 else nib
        sc3 = sc.unsqueeze(0) if sc.dim() == 2 else sc
        e, n, kh = nib3.shape
        k = 2 * kh
        out = torch.empty((self.repacked_bytes(n, k, e),), dtype=torch.uint8, device=nib.device)
        flags = NVFP4_GATED if gated else 0
        self._check("nvfp4_repack", self.lib.nvfp4_repack(
            nib3.contiguous().data_ptr(), sc3.contiguous().data_ptr(), e, n, k, flags, out.data_ptr(),
            _stream(stream)))
        return Weight(out, gscale.reshape(-1).contiguous().float(), n, k, e, flags)

    def repack_host(self, nib: np.ndarray, sc: np.ndarray, gated: bool = False) -> np.ndarray:
        """The host-memory repack: canonical u8 [E, n, k/2] / [E, n, k/16] (or 2-D) numpy
        arrays -> the repacked bytes (u8 numpy)."""
        nib3 = np.ascontiguousarray(nib.reshape((-1,) + nib.shape[-2:]), np.uint8)
        sc3 = np.ascontiguousarray(sc.reshape((-1,) + sc.shape[-2:]), np.uint8)
        e, n, kh = nib3.shape
        k = 2 * kh
        out = np.empty((self.repacked_bytes(n, k, e),), dtype=np.uint8)
        self._check("nvfp4_repack_host", self.lib.nvfp4_repack_host(
            nib3.ctypes.data, sc3.ctypes.data, e, n, k, NVFP4_GATED if gated else 0, out.ctypes.data, out.nbytes))
        return out

    def prepare(self, w: torch.Tensor, gated: bool = False, stream=None) -> Weight:
        """quantize + repack of fp32 weights already on the GPU."""
        nib, sc, g = self.quantize(w, stream)
        return self.repack(nib, sc, g, gated, stream)

    # -------------------------------------------------------------- hot path
    def gemm(self, w: Weight, x: torch.Tensor, y: torch.Tensor = None, stream=None) -> torch.Tensor:
        m = x.shape[0]
        if y is None:
            y = torch.empty((m, w.n), dtype=torch.bfloat16, device=x.device)
        nbytes = self.lib.nvfp4_gemm_workspace_bytes(m, w.n, w.k)
        ws = self.workspace("gemm", nbytes, x.device)
        cw = w.c()
        self._check("nvfp4_gemm", self.lib.nvfp4_gemm(
            ctypes.byref(cw), x.data_ptr(), m, y.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
        return y

    def lm_head_argmax(self, w: Weight, x: torch.Tensor, out=None, stream=None):
        m = x.shape[0]
        if out is None:
            out = (torch.empty((m,), dtype=torch.float32, device=x.device),
                   torch.empty((m,), dtype=torch.int32, device=x.device))
        nbytes = self.lib.lm_head_workspace_bytes(m, w.n)
        ws = self.workspace("lm_head", nbytes, x.device)
        cw = w.c()
        self._check("lm_head_argmax", self.lib.lm_head_argmax(
            ctypes.byref(cw), x.data_ptr(), m, out[0].data_ptr(), out[1].data_ptr(), ws.data_ptr(), ws.numel(),
            _stream(stream)))
        return out

    # -------------------------------------------------------------- W4A4
    def quantize_act(self, x: torch.Tensor, out=None, stream=None):
        """bf16 activations [m, k] -> NVFP4 per token row: (codes u8 [m, k/2], scales u8
        [m, k/16], global scales fp32 [m])."""
        m, k = x.shape
        if out is None:
            out = (torch.empty((m, k // 2), dtype=torch.uint8, device=x.device),
                   torch.empty((m, k // 16), dtype=torch.uint8, device=x.device),
                   torch.empty((m,), dtype=torch.float32, device=x.device))
        ws = self.workspace("quantize_act", max(16, self.lib.nvfp4_quantize_workspace_bytes(m)), x.device)
        self._check("nvfp4_quantize_act", self.lib.nvfp4_quantize_act(
            x.data_ptr(), m, k, out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), ws.data_ptr(), ws.numel(),
            _stream(stream)))
        return out

    def gemm_w4a4(self, w: Weight, xq, y: torch.Tensor = None, stream=None) -> torch.Tensor:
        codes, scales, g = xq
        m = codes.shape[0]
        if y is None:
            y = torch.empty((m, w.n), dtype=torch.bfloat16, device=codes.device)
        ws = self.workspace("gemm", self.lib.nvfp4_gemm_workspace_bytes(m, w.n, w.k), codes.device)
        cw = w.c()
        self._check("nvfp4_gemm_w4a4", self.lib.nvfp4_gemm_w4a4(
            ctypes.byref(cw), codes.data_ptr(), scales.data_ptr(), g.data_ptr(), m, y.data_ptr(), ws.data_ptr(),
            ws.numel(), _stream(stream)))
        return y

    def lm_head_argmax_w4a4(self, w: Weight, xq, out=None, stream=None):
        codes, scales, g = xq
        m = codes.shape[0]
        if out is None:
            out = (torch.empty((m,), dtype=torch.float32, device=codes.device),
                   torch.empty((m,), dtype=torch.int32, device=codes.device))
        ws = self.workspace("lm_head", self.lib.lm_head_workspace_bytes(m, w.n), codes.device)
        cw = w.c()
        self._check("lm_head_argmax_w4a4", self.lib.lm_head_argmax_w4a4(
            ctypes.byref(cw), codes.data_ptr(), scales.data_ptr(), g.data_ptr(), m, out[0].data_ptr(),
            out[1].data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
        return out

    def lm_head_sample(self, w: Weight, x: torch.Tensor, temperature: float, seed: int, out=None, stream=None,
                       softcap: float = 0.0):
        """Gumbel-max sample per token row (temperature 0: greedy): returns (max key, token).
        softcap > 0 applies cap * tanh(logit / cap) to every logit first."""
        m = x.shape[0]
        if out is None:
            out = (torch.empty((m,), dtype=torch.float32, device=x.device),
                   torch.empty((m,), dtype=torch.int32, device=x.device))
        ws = self.workspace("lm_head", self.lib.lm_head_workspace_bytes(m, w.n), x.device)
        cw = w.c()
        if softcap:
            self._check("lm_head_sample_ex", self.lib.lm_head_sample_ex(
                ctypes.byref(cw), x.data_ptr(), m, float(softcap), float(temperature), int(seed) & (2 ** 64 - 1),
                out[0].data_ptr(), out[1].data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
        else:
            self._check("lm_head_sample", self.lib.lm_head_sample(
                ctypes.byref(cw), x.data_ptr(), m, float(temperature), int(seed) & (2 ** 64 - 1), out[0].data_ptr(),
                out[1].data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
        return out

    def plan_lm_head_sample(self, w: Weight, x: torch.Tensor, temperature: float, seed: int, max_key, token,
                            stream=None):
        """lm_head_sample as a zero-argument callable (arguments marshalled once)."""
        m = x.shape[0]
        ws = self.workspace("lm_head", self.lib.lm_head_workspace_bytes(m, w.n), x.device)
        cw = w.c()
        args = (ctypes.byref(cw), x.data_ptr(), m, float(temperature), int(seed) & (2 ** 64 - 1), max_key.data_ptr(),
                token.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
        fn = self.lib.lm_head_sample

        def run():
            st = fn(*args)
            if st:
                raise NVFP4Error("lm_head_sample", st)
        run.keep = (cw, ws)
        return run

    def router_logits(self, w: Weight, x: torch.Tensor, gate_scale: torch.Tensor = None, eps: float = 1e-6,
                      out: torch.Tensor = None, stream=None) -> torch.Tensor:
        """Router logits: the unweighted RMSNorm of W . x times the per-expert scale (fp32 [m, n_experts])."""
        m = x.shape[0]
        if out is None:
            out = torch.empty((m, w.n), dtype=torch.float32, device=x.device)
        ws = self.workspace("gemm", self.lib.nvfp4_gemm_workspace_bytes(m, w.n, w.k), x.device)
        cw = w.c()
        self._check("moe_router_logits", self.lib.moe_router_logits(
            ctypes.byref(cw), x.data_ptr(), m, _ptr(gate_scale), float(eps), out.data_ptr(), ws.data_ptr(), ws.numel(),
            _stream(stream)))
        return out

    def route_topk(self, logits: torch.Tensor, top_k: int, out=None, stream=None, softmax_all: bool = False,
                   expert_scale: torch.Tensor = None):
        m, e = logits.shape
        if out is None:
            dev = logits.device
            out = (torch.empty((m, top_k), dtype=torch.int32, device=dev),
                   torch.empty((m, top_k), dtype=torch.float32, device=dev),
                   torch.empty((e + 1,), dtype=torch.int32, device=dev),
                   torch.empty((m * top_k,), dtype=torch.int32, device=dev))
        ids, probs, offsets, pairs = out
        if not softmax_all and expert_scale is None:
            self._check("moe_route_topk", self.lib.moe_route_topk(
                logits.data_ptr(), m, e, top_k, ids.data_ptr(), probs.data_ptr(), offsets.data_ptr(),
                pairs.data_ptr(), _stream(stream)))
        else:
            self._check("moe_route_topk_ex", self.lib.moe_route_topk_ex(
                logits.data_ptr(), m, e, top_k, NVFP4_ROUTE_SOFTMAX_ALL if softmax_all else 0,
                expert_scale.data_ptr() if expert_scale is not None else None, ids.data_ptr(), probs.data_ptr(),
                offsets.data_ptr(), pairs.data_ptr(), _stream(stream)))
        return out

    def moe_ffn(self, x, top_k, probs, offsets, pairs, gate_up: Weight, down: Weight, shared_gate_up: Weight = None,
                shared_down: Weight = None, out=None, stream=None):
        m, d = x.shape
        inter = down.k
        if out is None:
            out = torch.empty((m, d), dtype=torch.bfloat16, device=x.device)
        nbytes = self.lib.moe_ffn_workspace_bytes(m, top_k, gate_up.num_matrices, d, inter)
        ws = self.workspace("moe", nbytes, x.device)
        cg, cd = gate_up.c(), down.c()
        sg = ctypes.byref(shared_gate_up.c()) if shared_gate_up is not None else None
        sd = ctypes.byref(shared_down.c()) if shared_down is not None else None
        self._check("moe_ffn_grouped", self.lib.moe_ffn_grouped(
            x.data_ptr(), m, top_k, probs.data_ptr(), offsets.data_ptr(), pairs.data_ptr(), ctypes.byref(cg),
            ctypes.byref(cd), sg, sd, out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
        return out

    # -------------------------------------------------------------- call plans
    # Zero-argument callables with every ctypes argument built once, for timed
    # loops where per-call Python marshalling would otherwise show up.
    def plan_gemm(self, w: Weight, x: torch.Tensor, y: torch.Tensor, stream=None):
        m = x.shape[0]
        ws = self.workspace("gemm", self.lib.nvfp4_gemm_workspace_bytes(m, w.n, w.k), x.device)
        cw = w.c()
        args = (ctypes.byref(cw), x.data_ptr(), m, y.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
        fn = self.lib.nvfp4_gemm

        def run():
            st = fn(*args)
            if st:
                raise NVFP4Error("nvfp4_gemm", st)
        run.keep = (cw, ws)
        return run

    def plan_quantize_act(self, x: torch.Tensor, out, stream=None):
        """nvfp4_quantize_act as a zero-argument callable into `out` = (codes, scales, g)."""
        m, k = x.shape
        ws = self.workspace("quantize_act", max(16, self.lib.nvfp4_quantize_workspace_bytes(m)), x.device)
        args = (x.data_ptr(), m, k, out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), ws.data_ptr(),
                ws.numel(), _stream(stream))
        fn = self.lib.nvfp4_quantize_act

        def run():
            st = fn(*args)
            if st:
                raise NVFP4Error("nvfp4_quantize_act", st)
        run.keep = (ws,)
        return run

    def plan_gemm_w4a4(self, w: Weight, xq, y: torch.Tensor, stream=None):
        codes, scales, g = xq
        m = codes.shape[0]
        ws = self.workspace("gemm", self.lib.nvfp4_gemm_workspace_bytes(m, w.n, w.k), codes.device)
        cw = w.c()
        args = (ctypes.byref(cw), codes.data_ptr(), scales.data_ptr(), g.data_ptr(), m, y.data_ptr(), ws.data_ptr(),
                ws.numel(), _stream(stream))
        fn = self.lib.nvfp4_gemm_w4a4

        def run():
            st = fn(*args)
            if st:
                raise NVFP4Error("nvfp4_gemm_w4a4", st)
        run.keep = (cw, ws)
        return run

    def plan_lm_head_w4a4(self, w: Weight, xq, max_logit: torch.Tensor, argmax: torch.Tensor, stream=None):
        codes, scales, g = xq
        m = codes.shape[0]
        ws = self.workspace("lm_head", self.lib.lm_head_workspace_bytes(m, w.n), codes.device)
        cw = w.c()
        args = (ctypes.byref(cw), codes.data_ptr(), scales.data_ptr(), g.data_ptr(), m, max_logit.data_ptr(),
                argmax.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
        fn = self.lib.lm_head_argmax_w4a4

        def run():
            st = fn(*args)
            if st:
                raise NVFP4Error("lm_head_argmax_w4a4", st)
        run.keep = (cw, ws)
        return run

    def plan_lm_head(self, w: Weight, x: torch.Tensor, max_logit: torch.Tensor, argmax: torch.Tensor, stream=None):
        m = x.shape[0]
        ws = self.workspace("lm_head", self.lib.lm_head_workspace_bytes(m, w.n), x.device)
        cw = w.c()
        args = (ctypes.byref(cw), x.data_ptr(), m, max_logit.data_ptr(), argmax.data_ptr(), ws.data_ptr(),
                ws.numel(), _stream(stream))
        fn = self.lib.lm_head_argmax

        def run():
            st = fn(*args)
            if st:
                raise NVFP4Error("lm_head_argmax", st)
        run.keep = (cw, ws)
        return run

    def moe_forward(self, x, logits, top_k, gate_up: Weight, down: Weight, shared_gate_up: Weight = None,
                    shared_down: Weight = None, route_out=None, out=None, stream=None, softmax_all: bool = False,
                    expert_scale: torch.Tensor = None):
        """The MoE layer in one C call (router + grouped FFN): returns (out, (ids, probs, offsets, pairs))."""
        m, d = x.shape
        e = logits.shape[1]
        dev = x.device
        if route_out is None:
            route_out = (torch.empty((m, top_k), dtype=torch.int32, device=dev),
                         torch.empty((m, top_k), dtype=torch.float32, device=dev),
                         torch.empty((e + 1,), dtype=torch.int32, device=dev),
                         torch.empty((m * top_k,), dtype=torch.int32, device=dev))
        if out is None:
            out = torch.empty((m, d), dtype=torch.bfloat16, device=dev)
        ws = self.workspace("moe", self.lib.moe_ffn_workspace_bytes(m, top_k, gate_up.num_matrices, d, down.k), dev)
        cg, cd = gate_up.c(), down.c()
        sg = shared_gate_up.c() if shared_gate_up is not None else None
        sd = shared_down.c() if shared_down is not None else None
        ids, probs, offsets, pairs = route_out
        self._check("moe_forward", self.lib.moe_forward(
            x.data_ptr(), logits.data_ptr(), m, top_k, NVFP4_ROUTE_SOFTMAX_ALL if softmax_all else 0,
            _ptr(expert_scale), ids.data_ptr(), probs.data_ptr(), offsets.data_ptr(), pairs.data_ptr(),
            ctypes.byref(cg), ctypes.byref(cd), ctypes.byref(sg) if sg is not None else None,
            ctypes.byref(sd) if sd is not None else None, out.data_ptr(), ws.data_ptr(), ws.numel(),
            _stream(stream)))
        return out, route_out

    def plan_moe(self, x, logits, top_k, gate_up: Weight, down: Weight, shared_gate_up: Weight, shared_down: Weight,
                 route_out, out, stream=None):
        """The MoE layer (moe_forward: router + grouped FFN in one C call) as a zero-argument callable."""
        m, d = x.shape
        e = logits.shape[1]
        ids, probs, offsets, pairs = route_out
        ws = self.workspace("moe", self.lib.moe_ffn_workspace_bytes(m, top_k, gate_up.num_matrices, d, down.k),
                            x.device)
        cg, cd = gate_up.c(), down.c()
        sg = shared_gate_up.c() if shared_gate_up is not None else None
        sd = shared_down.c() if shared_down is not None else None
        s = _stream(stream)
        args = (x.data_ptr(), logits.data_ptr(), m, top_k, 0, None, ids.data_ptr(), probs.data_ptr(),
                offsets.data_ptr(), pairs.data_ptr(), ctypes.byref(cg), ctypes.byref(cd),
                ctypes.byref(sg) if sg is not None else None, ctypes.byref(sd) if sd is not None else None,
                out.data_ptr(), ws.data_ptr(), ws.numel(), s)
        fn = self.lib.moe_forward

        def run():
            st = fn(*args)
            if st:
                raise NVFP4Error("moe_forward", st)
        run.keep = (cg, cd, sg, sd, ws)
        return run


_LIB = None


def load(path: str = LIB) -> Library:
    global _LIB
    if _LIB is None or _LIB.path != path:
        _LIB = Library(path)
    return _LIB
