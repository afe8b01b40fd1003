"""Seeded synthetic inputs for the five workloads.

This module is the only one that both the CUDA path and the CPU oracle use.
It holds none of the method's arithmetic: it draws random numbers and rounds
activations to bf16 (the input format), nothing else.

Recipes (the pages name no dataset; every input is synthetic):

* weights: fp32 ``0.02 * N(0, 1)`` drawn with numpy's PCG64 ``default_rng`` in
  float32; the tiny 512 x 256 matrix uses seed 0, every other tensor a seed
  derived from its name (``seed_of``).
* activations x: ``N(0, 1)`` drawn in float32, rounded to bf16
  (round-to-nearest-even on the bit pattern).
* router logits: fp32 ``N(0, 1)``.

Shapes (Gemma-4-26B-A4B: hidden 2816, 128 experts, top-8 + 1 shared,
262,144-entry vocabulary; expert intermediate 704; verify block M = 15 =
14 drafted + 1):
"""

from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np

HIDDEN = 2816
N_EXPERTS = 128
TOP_K = 8
INTER = 704
VOCAB = 262144

TINY = dict(m=1, n=512, k=256)
DENSE_K = 4096
DENSE_N = (4096, 14336)
DENSE_M = (1, 4, 15, 16)
DECODE_M = (1, 15)
PREFILL_M = 512


def seed_of(*parts) -> int:
    """Stable 31-bit seed from a name path, e.g. seed_of('moe', 'gate_up', 17)."""
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def normal_f32(shape, seed: int, std: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    return z


def to_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x_f32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(shape, seed: int):
    """(bf16 bits uint16, the same values as float32)."""
    bits = to_bf16_bits(normal_f32(shape, seed))
    return bits, bf16_bits_to_f32(bits)


def weight(shape, seed: int) -> np.ndarray:
    return normal_f32(shape, seed, std=0.02)


@dataclass(frozen=True)
class DenseCase:
    m: int
    n: int
    k: int
    w_seed: int
    x_seed: int

    @staticmethod
    def tiny():
        return DenseCase(TINY["m"], TINY["n"], TINY["k"], 0, seed_of("tiny", "x"))

    @staticmethod
    def sweep(m: int, n: int, k: int = DENSE_K):
        return DenseCase(m, n, k, seed_of("dense", n, k, "w"), seed_of("dense", m, n, k, "x"))

    def w(self):
        return weight((self.n, self.k), self.w_seed)

    def x(self):
        return activations((self.m, self.k), self.x_seed)


@dataclass(frozen=True)
class MoECase:
    m: int
    d: int = HIDDEN
    inter: int = INTER
    n_experts: int = N_EXPERTS
    top_k: int = TOP_K
    tag: str = "moe"

    def gate_up(self, e: int) -> np.ndarray:
        """Expert e's fused [gate || up] weight [2I, d] (e = -1: the shared expert)."""
        return weight((2 * self.inter, self.d), seed_of(self.tag, self.d, self.inter, "gate_up", e))

    def down(self, e: int) -> np.ndarray:
        return weight((self.d, self.inter), seed_of(self.tag, self.d, self.inter, "down", e))

    def x(self):
        return activations((self.m, self.d), seed_of(self.tag, self.m, self.d, "x"))

    def logits(self) -> np.ndarray:
        return normal_f32((self.m, self.n_experts), seed_of(self.tag, self.m, self.n_experts, "logits"))


@dataclass(frozen=True)
class LMHeadCase:
    m: int
    vocab: int = VOCAB
    d: int = HIDDEN

    def w_rows(self, lo: int, hi: int) -> np.ndarray:
        """Rows [lo, hi) of the vocab matrix; drawn in 8192-row chunks so any slice is reproducible."""
        chunk = 8192
        out = np.empty((hi - lo, self.d), np.float32)
        c0 = lo // chunk
        for c in range(c0, -(-hi // chunk)):
            a, b = c * chunk, min(self.vocab, (c + 1) * chunk)
            block = weight((b - a, self.d), seed_of("lm_head", self.vocab, self.d, c))
            s, t = max(a, lo), min(b, hi)
            out[s - lo:t - lo] = block[s - a:t - a]
        return out

    def x(self):
        return activations((self.m, self.d), seed_of("lm_head", self.m, self.d, "x"))
