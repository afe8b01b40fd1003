"""The library's launch plans checked against the streaming kernels' work
decomposition on the CPU (no GPU).

nvfp4_plan_check walks a product's whole launch -- every CTA, run, warp and
piece -- with the kernels' own decomposition code (the DecodeDeal and
PrefillDeal structs that the decode and prefill kernels call), for a given
number of segments, and reports whether every (segment, 64-row group, 16-row
tile, K slice) is computed exactly once, every piece lies in its CTA's staged
columns and segments (a prefill piece in its run's block), and every K-split
counter in its fixed area; and the largest staged span and segment count
against the planned capacities.  The plans come from the library's planner (the
one the products call), so a planner or decomposition change that breaks
coverage or capacity fails here before any kernel runs.  Segment counts come
from uniform, concentrated and block-boundary routings."""

import ctypes
import random

import pytest

from nvfp4_w4a16_moe_skinny_gb300 import build as B

MAX_SMEM = 227 * 1024


def cdiv(a, b):
    return -(-a // b)


@pytest.fixture(scope="module")
def so():
    B.build()
    from nvfp4_w4a16_moe_skinny_gb300 import binding
    lib = ctypes.CDLL(B.LIB)
    binding._sig(lib)
    return lib


def plan_of(so, product, m, n, k, top_k=0, n_experts=0, sms=152):
    out = (ctypes.c_int32 * 11)()
    st = so.nvfp4_plan_info(product, m, n, k, top_k, n_experts, sms, out, 11)
    assert st == 0, (product, m, n, k, top_k, n_experts, sms, st)
    keys = ("S", "L", "ns", "xs_chunks", "xs_rows", "max_cta_segs", "grid", "max_segs", "per_run", "smem",
            "slice_ctas")
    return dict(zip(keys, list(out)))


def check(so, product, m, n, k, n_seg, top_k=0, n_experts=0, sms=152):
    out = (ctypes.c_int32 * 8)()
    st = so.nvfp4_plan_check(product, m, n, k, top_k, n_experts, sms, n_seg, out, 8)
    assert st == 0, (product, m, n, k, n_seg, sms, st)
    r = dict(zip(("ok", "max_span", "xs_chunks", "max_segs", "cta_segs", "tiles", "pieces", "smem"), list(out)))
    pl = plan_of(so, product, m, n, k, top_k, n_experts, sms)
    what = f"product {product} m={m} n={n} k={k} n_seg={n_seg} sms={sms}: {r} {pl}"
    assert r["ok"] == 1, what
    assert r["max_span"] <= r["xs_chunks"], what
    assert r["max_segs"] <= max(r["cta_segs"], 1), what
    assert r["smem"] <= MAX_SMEM, what
    assert r["tiles"] == n_seg * cdiv(n, 64) * 4 * pl["S"], what
    if not pl["per_run"]:
        # staged rows: a CTA's segments x at most 16 rows each (the down product), or the m tokens
        rows = r["max_segs"] * min(m, 16) if product == 3 else m
        assert rows <= pl["xs_rows"] <= 128, what
    return r, pl


def routings(m, top_k, n_experts, seed):
    """Per-expert pair counts: uniform random, every token on the same experts, and
    as many experts as possible just past a block boundary."""
    rng = random.Random(seed)
    out = []
    c = [0] * n_experts
    for _ in range(m):
        for e in rng.sample(range(n_experts), top_k):
            c[e] += 1
    out.append(c)
    c = [0] * n_experts
    for e in range(top_k):
        c[e] = m
    out.append(c)
    c, left = [0] * n_experts, m * top_k
    for e in range(n_experts):
        take = min(left, m, 33 if m > 16 else 1)
        c[e], left = take, left - take
    for e in range(n_experts):
        add = min(left, m - c[e])
        c[e], left = c[e] + add, left - add
    assert sum(c) == m * top_k and max(c) <= m
    out.append(c)
    return out


def segments(counts, m, shared=True):
    """Segments the kernels build from per-expert pair counts: one per active expert
    (decode), or one per block of 32 pairs (prefill), plus the shared expert's."""
    blk = 32 if m > 16 else 10 ** 9
    return sum(cdiv(c, blk) if m > 16 else 1 for c in counts if c > 0) + (cdiv(m, 32) if m > 16 else 1) * shared


@pytest.mark.parametrize("sms", [152, 148, 16])
@pytest.mark.parametrize("n,k", [(4096, 4096), (14336, 4096), (512, 256), (1000, 320), (40, 80), (64, 1024),
                                 (512, 16384), (136, 32768), (1000, 12288)])
def test_dense_plans_cover_every_tile_once(so, sms, n, k):
    for m in (1, 2, 4, 7, 8, 15, 16):
        check(so, 0, m, n, k, 1, sms=sms)


def test_split_dense_ctas_stay_in_one_slice(so):
    """A dense GEMM split along K on a grid the split divides stages one slice per CTA."""
    for n in (4096, 14336):
        for m in (1, 15):
            r, pl = check(so, 0, m, n, 4096, 1)
            if pl["S"] > 1 and 152 % pl["S"] == 0:
                assert pl["slice_ctas"] == 1 and r["max_span"] <= pl["L"] == pl["xs_chunks"], (r, pl)


@pytest.mark.parametrize("m", [1, 15])
def test_lm_head_plan_covers_every_tile_once(so, m):
    _, pl = check(so, 1, m, 262144, 2816, 1)
    assert pl["S"] == 1  # the lm_head never splits K


def test_busiest_warp_report(so):
    """The walk reports the busiest warp's (tile x chunk) steps against the mean: the
    lm_head's 26-27 whole 64-row groups per CTA over 16 warps give warps one or two
    groups (2 x 4 tiles x 44 chunks = 352 against a mean of ~297)."""
    out = (ctypes.c_int32 * 10)()
    assert so.nvfp4_plan_check(1, 15, 262144, 2816, 0, 0, 152, 1, out, 10) == 0
    assert out[0] == 1 and out[8] == 2 * 4 * 44
    assert out[9] == -(-262144 // 64 * 4 * 44 // (152 * 16))


@pytest.mark.parametrize("m,top_k,n_exp,d,inter", [
    (1, 8, 128, 2816, 704), (15, 8, 128, 2816, 704), (16, 8, 128, 2816, 704), (512, 8, 128, 2816, 704),
    (2, 3, 8, 128, 64), (16, 2, 6, 192, 128), (40, 3, 8, 128, 64), (100, 1, 40, 192, 128), (17, 2, 6, 192, 128),
    (16, 32, 1024, 128, 64), (1, 32, 1024, 256, 128), (16, 16, 512, 128, 64), (16, 3, 8, 320, 192),
    (2048, 8, 128, 128, 64), (4096, 4, 16, 128, 64)])
@pytest.mark.parametrize("sms", [152, 148, 16])
def test_moe_plans_cover_every_tile_once(so, m, top_k, n_exp, d, inter, sms):
    for i, counts in enumerate(routings(m, top_k, n_exp, 7 * m + top_k)):
        n_seg = segments(counts, m)
        for product, n, k in ((2, 2 * inter, d), (3, d, inter)):
            pl = plan_of(so, product, m, n, k, top_k, n_exp, sms)
            assert n_seg <= pl["max_segs"], (counts, n_seg, pl)
            check(so, product, m, n, k, n_seg, top_k, n_exp, sms)


def test_plan_query_rejects_bad_shapes(so):
    out = (ctypes.c_int32 * 10)()
    assert so.nvfp4_plan_info(0, 17, 64, 64, 0, 0, 152, out, 10) != 0     # dense m > 16
    assert so.nvfp4_plan_info(9, 1, 64, 64, 0, 0, 152, out, 10) != 0      # unknown product
    assert so.nvfp4_plan_info(0, 1, 64, 60, 0, 0, 152, out, 10) != 0      # k % 16
    assert so.nvfp4_plan_info(0, 1, 64, 64, 0, 0, 0, out, 10) != 0        # no SMs
    out8 = (ctypes.c_int32 * 8)()
    assert so.nvfp4_plan_check(2, 15, 1408, 2816, 8, 128, 152, 10 ** 6, out8, 8) != 0   # more segments than planned


def test_random_shapes_always_get_a_valid_plan(so):
    """Seeded random shapes the ABI accepts all get plans that pass the walk."""
    rng = random.Random(12)
    for _ in range(60):
        product = rng.choice([0, 1, 2, 3])
        sms = rng.choice([152, 148, 132, 16, 7])
        if product in (0, 1):
            m = rng.randint(1, 16)
            n, k = rng.randint(1, 3000), 16 * rng.randint(1, 300)
            check(so, product, m, n, k, 1, sms=sms)
        else:
            m = rng.choice([1, 3, 15, 16, 17, 40, 200])
            n_exp = rng.choice([4, 8, 40, 128])
            top_k = rng.randint(1, min(8, n_exp))
            d, inter = 64 * rng.randint(1, 40), 64 * rng.randint(1, 12)
            n, k = (2 * inter, d) if product == 2 else (d, inter)
            pl = plan_of(so, product, m, n, k, top_k, n_exp, sms)
            check(so, product, m, n, k, rng.randint(1, pl["max_segs"]), top_k, n_exp, sms)
