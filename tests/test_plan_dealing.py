"""The launch plans of the library's planner, checked against the kernels' work
decomposition on the CPU (no GPU): for every CTA and warp of a grid, the pieces the
streaming kernels would take are enumerated with the kernels' own dealing rules
(restated here in Python), and the checks are that every (segment, 64-row group,
16-row tile, K slice) is computed exactly once, that no copy starts outside its
matrix, that every CTA's staged rows and columns fit the planned capacity, and
that K-split arrival counters stay inside their fixed area.

The plans come from the library itself (nvfp4_plan_info), so a planner change that
breaks the decomposition fails here before any kernel runs.  The dealing rules are
those of the decode kernel (kernel.cuh: units of four tiles, whole or split
dealing, one staging per CTA) and of the prefill kernel (prefill.cuh: units of two
tiles, one run per (segment, K slice))."""

import ctypes
import random

import pytest

from nvfp4_w4a16_moe_skinny_gb300 import build as B

WARPS = 16
TILE_BYTES = 576
STAGE_BYTES = 4 * TILE_BYTES
X_CHUNK = 128
MAX_STAGED_ROWS = 128
COUNTER_CELLS = 512 * 1024 // 4
MAX_SMEM = 227 * 1024
SHARED = -1


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
    out = (ctypes.c_int32 * 10)()
    st = so.nvfp4_plan_info(product, m, n, k, top_k, n_experts, sms, out, 10)
    assert st == 0, (product, m, n, k, top_k, n_experts, sms, st)
    keys = ("S", "L", "ns", "xs_chunks", "xs_rows", "max_cta_segs", "grid", "max_segs", "per_run", "smem")
    return dict(zip(keys, list(out)))


def whole_dealing(nu, tiles_per_unit):
    return cdiv(nu, WARPS) * tiles_per_unit * 100 <= cdiv(tiles_per_unit * nu, WARPS) * 115


def pieces(lo, nu, tiles_per_unit, warp):
    """(unit, first tile within the unit, tiles) of warp `warp` over units [lo, lo+nu)."""
    tpu = tiles_per_unit
    if whole_dealing(nu, tpu):
        return [(lo + k * WARPS + warp, 0, tpu) for k in range((nu - warp + WARPS - 1) // WARPS)]
    t0, t1 = (tpu * nu * warp) // WARPS, (tpu * nu * (warp + 1)) // WARPS
    out = []
    if t1 > t0:
        for k in range((t1 - 1) // tpu - t0 // tpu + 1):
            start = t0 if k == 0 else (t0 // tpu + k) * tpu
            end = min(t1, (t0 // tpu + k + 1) * tpu)
            out.append((lo + start // tpu, start % tpu, end - start))
    return out


def check_decode(plan, m, ng, kc, segs, x_by_pair):
    """segs: staged rows of each segment (dense: [m]).  Mirrors stream_kernel."""
    S, L, grid = plan["S"], plan["L"], plan["grid"]
    per_seg = S * ng
    n_units = len(segs) * per_seg
    mat_bytes = ng * kc * STAGE_BYTES
    seen = set()
    assert plan["smem"] <= MAX_SMEM
    for b in range(grid):
        u0, u1 = n_units * b // grid, n_units * (b + 1) // grid
        nu = u1 - u0
        if nu == 0:
            continue
        cseg0 = u0 // per_seg
        nsc = (u1 - 1) // per_seg - cseg0 + 1
        c_lo, c_hi = 0, kc
        if nsc == 1:
            c_lo = ((u0 - cseg0 * per_seg) // ng) * L
            c_hi = min(kc, ((u1 - 1 - cseg0 * per_seg) // ng + 1) * L)
        assert nsc <= plan["max_cta_segs"] and c_hi - c_lo <= plan["xs_chunks"], (b, nsc, c_lo, c_hi, plan)
        rows = sum(min(m, segs[cseg0 + i]) for i in range(nsc)) if x_by_pair else m
        assert rows <= plan["xs_rows"] <= MAX_STAGED_ROWS, (b, rows, plan)
        for w in range(WARPS):
            for unit, t0, tn in pieces(u0, nu, 4, w):
                assert u0 <= unit < u1 and 1 <= tn and t0 + tn <= 4
                seg, r = divmod(unit, per_seg)
                s, grp = divmod(r, ng)
                kc0, nch = s * L, min(kc, (s + 1) * L) - s * L
                assert nch >= 1 and c_lo <= kc0 and kc0 + nch <= c_hi
                if tn == 4:  # bulk copies of whole chunks
                    assert (grp * kc + kc0 + nch) * STAGE_BYTES <= mat_bytes
                else:  # tensor boxes start inside the matrix (they may run past K: zero fill)
                    assert grp < ng and kc0 < kc
                for t in range(t0, t0 + tn):
                    key = (seg, grp, t, s)
                    assert key not in seen, key
                    seen.add(key)
                if S > 1:
                    assert (seg * ng + grp) * 4 + t0 + tn <= COUNTER_CELLS
    assert len(seen) == len(segs) * ng * 4 * S


def check_prefill(plan, ng, kc, segs):
    """segs: valid slots of each segment (<= 32).  Mirrors prefill_kernel."""
    S, L, grid = plan["S"], plan["L"], plan["grid"]
    assert plan["per_run"] == 1 and L <= plan["xs_chunks"] and plan["smem"] <= MAX_SMEM
    assert len(segs) <= plan["max_segs"]
    upg = 2 * ng
    per_seg = S * upg
    n_units = len(segs) * per_seg
    seen = set()
    for b in range(grid):
        u0, u1 = n_units * b // grid, n_units * (b + 1) // grid
        if u1 == u0:
            continue
        b0 = u0 // upg
        for r in range((u1 - 1) // upg - b0 + 1):
            lo, hi = max(u0, (b0 + r) * upg), min(u1, (b0 + r + 1) * upg)
            seg_r, slice_r = divmod(b0 + r, S)
            assert 1 <= segs[seg_r] <= 32
            for w in range(WARPS):
                for unit, t0, tn in pieces(lo, hi - lo, 2, w):
                    assert lo <= unit < hi and 1 <= tn and t0 + tn <= 2
                    seg, rr = divmod(unit, per_seg)
                    s, q = divmod(rr, upg)
                    grp, tile0 = q >> 1, 2 * (q & 1) + t0
                    assert seg == seg_r and s == slice_r and grp < ng and s * L < kc
                    for t in range(tile0, tile0 + tn):
                        key = (seg, grp, t, s)
                        assert key not in seen, key
                        seen.add(key)
                    if S > 1:
                        assert (seg * ng + grp) * 4 + tile0 + tn <= COUNTER_CELLS
    assert len(seen) == len(segs) * ng * 4 * S


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


@pytest.mark.parametrize("sms", [152, 148, 16])
@pytest.mark.parametrize("n,k", [(4096, 4096), (14336, 4096), (512, 256), (1000, 320), (40, 80), (64, 1024)])
def test_dense_plans_cover_every_tile_once(so, sms, n, k):
    for m in (1, 2, 4, 7, 8, 15, 16):
        plan = plan_of(so, 0, m, n, k, sms=sms)
        check_decode(plan, m, cdiv(n, 64), cdiv(k, 64), [m], False)


@pytest.mark.parametrize("m", [1, 15])
def test_lm_head_plan_covers_every_tile_once(so, m):
    plan = plan_of(so, 1, m, 262144, 2816)
    assert plan["S"] == 1  # the lm_head never splits K
    check_decode(plan, m, 4096, 44, [m], False)


@pytest.mark.parametrize("m,top_k,n_exp,d,inter", [
    (1, 8, 128, 2816, 704), (15, 8, 128, 2816, 704), (16, 3, 8, 128, 64), (5, 2, 6, 192, 128),
    (17, 3, 8, 128, 64), (40, 2, 6, 192, 128), (100, 3, 8, 128, 64), (512, 8, 128, 2816, 704)])
@pytest.mark.parametrize("sms", [152, 16])
def test_moe_plans_cover_every_tile_once(so, m, top_k, n_exp, d, inter, sms):
    blk = 32 if m > 16 else 16
    for counts in routings(m, top_k, n_exp, seed=m * 131 + n_exp):
        rows = [c for c in counts if c > 0]          # decode: one segment per active expert
        blocks = []                                   # prefill: blocks of 32 pairs
        for c in counts:
            blocks += [min(blk, c - blk * b) for b in range(cdiv(c, blk))]
        shared_blocks = [min(blk, m - blk * b) for b in range(cdiv(m, blk))]
        for product, n, k in ((2, 2 * inter, d), (3, d, inter)):
            plan = plan_of(so, product, m, n, k, top_k, n_exp, sms)
            if m > 16:
                check_prefill(plan, cdiv(n, 64), cdiv(k, 64), blocks + shared_blocks)
            else:
                assert plan["per_run"] == 0
                check_decode(plan, m, cdiv(n, 64), cdiv(k, 64), rows + [m], product == 3)


def test_plan_query_rejects_bad_shapes(so):
    out = (ctypes.c_int32 * 10)()
    assert so.nvfp4_plan_info(0, 17, 64, 64, 0, 0, 152, out, 10) == 2   # dense m > 16
    assert so.nvfp4_plan_info(4, 1, 64, 64, 0, 0, 152, out, 10) == 2    # unknown product
    assert so.nvfp4_plan_info(2, 1, 128, 64, 9, 8, 152, out, 10) == 2   # top_k > n_experts
    assert so.nvfp4_plan_info(0, 1, 64, 64, 0, 0, 152, None, 10) == 1


def test_random_shapes_always_get_a_valid_plan(so):
    """Shapes the ABI accepts, drawn at random (seeded): the planner returns a plan for
    each, and the plan passes the decomposition checks under a random routing."""
    rng = random.Random(2026)
    for _ in range(40):
        m = rng.randint(1, 16)
        n = rng.randint(1, 300) * rng.choice([1, 16, 64])
        k = 16 * rng.randint(1, 400)
        sms = rng.choice([152, 148, 132, 16])
        check_decode(plan_of(so, 0, m, n, k, sms=sms), m, cdiv(n, 64), cdiv(k, 64), [m], False)
    for _ in range(25):
        m = rng.choice([1, 2, 7, 15, 16, 17, 31, 33, 64, 200, 512])
        n_exp = rng.choice([2, 8, 40, 128, 256])
        top_k = rng.randint(1, min(8, n_exp))
        d, inter = 64 * rng.randint(1, 48), 64 * rng.randint(1, 16)
        sms = rng.choice([152, 16])
        counts = routings(m, top_k, n_exp, seed=rng.randint(0, 10 ** 6))[0]
        blk = 32 if m > 16 else 16
        blocks = [min(blk, c - blk * b) for c in counts for b in range(cdiv(c, blk))]
        for product, nn, kk in ((2, 2 * inter, d), (3, d, inter)):
            plan = plan_of(so, product, m, nn, kk, top_k, n_exp, sms)
            if m > 16:
                check_prefill(plan, cdiv(nn, 64), cdiv(kk, 64), blocks + [min(blk, m - blk * b) for b in range(cdiv(m, blk))])
            else:
                check_decode(plan, m, cdiv(nn, 64), cdiv(kk, 64), [c for c in counts if c > 0] + [m], product == 3)
