"""The repacked kernel layout as an index function (oracle; test infrastructure only).

The pages say only that weights are repacked once, offline, "into
mma-fragment order" so kernel loads are 16-byte coalesced
(gemma-cuda-hybrid README, "Everything it has / Inference engine" and
"NVFP4-specific").  The layout itself is this library's; its specification,
for layout version 2, is:

* Rows are padded to a multiple of 64, K to a multiple of 64, with zero bytes.
* A *gated* matrix [gate || up] with N = 2I (I % 32 == 0) first has its rows
  permuted: gate row i goes to row 16*(i//8) + i%8, up row i to
  16*(i//8) + 8 + i%8, so each 16-row block holds 8 gate rows and the 8 up rows
  of the same indices.
* The padded matrix is cut into tiles of 16 rows x 64 columns.  Four
  consecutive 16-row blocks form a 64-row group; tile (group G, chunk kc,
  block r in 0..3) starts at byte 576 * ((G * KC + kc) * 4 + r), KC = K_pad / 64:
  the four tiles of one group and one 64-column chunk are contiguous (2,304 B).
  A stack of E matrices puts matrix e at byte e * (NG * KC * 4 * 576),
  NG = N_pad / 64.
* Tile bytes [0, 512): byte 16*lane + 4*kt + r (lane = 4*g + t, g in 0..7,
  t in 0..3, kt in 0..3, r in 0..3) is the canonical byte holding columns
  (c, c+1) of the tile's row g + 8*(r & 1), with c = 64*kc + 16*kt + 2*t +
  8*(r >> 1); low nibble = column c.
* Tile bytes [512, 576): byte 512 + 8*g + 2*kt + h is the scale of the tile's
  row g + 8*h, group 4*kc + kt.

This module computes the same mapping independently of the CUDA repack kernel:
for every (row, column pair) and (row, group) it places the canonical byte.
"""

from __future__ import annotations

import numpy as np

TILE_ROWS = 16
GROUP_ROWS = 64
TILE_COLS = 64
TILE_BYTES = 576


def padded_dims(n: int, k: int):
    n_pad = -(-n // GROUP_ROWS) * GROUP_ROWS
    k_pad = -(-k // TILE_COLS) * TILE_COLS
    return n_pad, k_pad


def repacked_bytes(n: int, k: int, num_matrices: int = 1) -> int:
    n_pad, k_pad = padded_dims(n, k)
    return num_matrices * (n_pad // TILE_ROWS) * (k_pad // TILE_COLS) * TILE_BYTES


def row_permutation(n: int, gated: bool) -> np.ndarray:
    """dest_row[n] for each original row n."""
    rows = np.arange(n)
    if not gated:
        return rows
    inter = n // 2
    i = np.where(rows < inter, rows, rows - inter)
    half = (rows >= inter).astype(np.int64)
    return 16 * (i // 8) + 8 * half + i % 8


def _tile_start(dest_row, kc, kc_count):
    rb = dest_row // 16
    grp, r = rb // 4, rb % 4
    return TILE_BYTES * ((grp * kc_count + kc) * 4 + r)


def nibble_byte_offset(dest_row, col_pair, kc_count):
    """Byte offset (within one matrix) of the canonical byte (dest_row, column pair col_pair)."""
    dest_row = np.asarray(dest_row, np.int64)
    c = 2 * np.asarray(col_pair, np.int64)
    rr = dest_row % 16
    kc, cc = c // 64, c % 64
    g, hrow = rr % 8, rr // 8
    kt, c16 = cc // 16, cc % 16
    hcol, t2 = c16 // 8, c16 % 8
    t = t2 // 2
    r = hrow + 2 * hcol
    lane = 4 * g + t
    return _tile_start(dest_row, kc, kc_count) + 16 * lane + 4 * kt + r


def scale_byte_offset(dest_row, group, kc_count):
    dest_row = np.asarray(dest_row, np.int64)
    grp = np.asarray(group, np.int64)
    rr = dest_row % 16
    kc, kt = grp // 4, grp % 4
    g, h = rr % 8, rr // 8
    return _tile_start(dest_row, kc, kc_count) + 512 + 8 * g + 2 * kt + h


def repack(nib: np.ndarray, scales: np.ndarray, gated: bool = False) -> np.ndarray:
    """Canonical [E, N, K/2] + [E, N, K/16] (or 2-D) -> repacked uint8 buffer."""
    if nib.ndim == 2:
        nib, scales = nib[None], scales[None]
    e_count, n, kh = nib.shape
    k = 2 * kh
    n_pad, k_pad = padded_dims(n, k)
    kc_count = k_pad // 64
    per = repacked_bytes(n, k, 1)
    out = np.zeros(e_count * per, dtype=np.uint8)
    dest = row_permutation(n, gated)
    rows = np.repeat(dest, kh)
    pairs = np.tile(np.arange(kh), n)
    noff = nibble_byte_offset(rows, pairs, kc_count)
    srows = np.repeat(dest, k // 16)
    groups = np.tile(np.arange(k // 16), n)
    soff = scale_byte_offset(srows, groups, kc_count)
    for e in range(e_count):
        out[e * per + noff] = nib[e].reshape(-1)
        out[e * per + soff] = scales[e].reshape(-1)
    return out


def unrepack(buf: np.ndarray, n: int, k: int, num_matrices: int = 1, gated: bool = False):
    """Inverse of ``repack``: returns canonical (nib [E, N, K/2], scales [E, N, K/16])."""
    n_pad, k_pad = padded_dims(n, k)
    kc_count = k_pad // 64
    per = repacked_bytes(n, k, 1)
    kh = k // 2
    dest = row_permutation(n, gated)
    noff = nibble_byte_offset(np.repeat(dest, kh), np.tile(np.arange(kh), n), kc_count)
    soff = scale_byte_offset(np.repeat(dest, k // 16), np.tile(np.arange(k // 16), n), kc_count)
    nib = np.stack([buf[e * per + noff].reshape(n, kh) for e in range(num_matrices)])
    sc = np.stack([buf[e * per + soff].reshape(n, k // 16) for e in range(num_matrices)])
    return nib, sc
