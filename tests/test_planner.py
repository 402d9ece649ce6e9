"""Host split planner: exact partition of every sequence, no empty split, the
unit numbering the kernels assume (checked by brute force on the CPU)."""
import itertools
import random

import numpy as np

import pytest

from mla_attention_decode_gb300 import binding


def n_splits(plan, L):
    if L <= 0:
        return 1
    return max(1, min(plan.max_splits, -(-L // plan.chunk_tokens), -(-L // plan.tile_tokens)))


class Partition:
    """Schedule 1's CTA ranges (mla_decode.h): CTA c owns [lo(c), lo(c + 1)),
    the last L CTAs D positions fewer; written from the rule, and cta(x) found
    by search rather than by the closed form the library uses."""

    def __init__(self, plan, C):
        G, D = plan.grid, plan.late_tiles
        L = min(G, max(0, G + plan.batch - plan.num_sms)) if D > 0 else 0
        Cp = C + L * D
        self.G = G
        self.b = [k * Cp // G - D * max(0, k - (G - L)) for k in range(G + 1)]
        assert self.b[0] == 0 and self.b[G] == C

    def lo(self, c):
        return self.b[c]

    def cta(self, x):
        c = max(k for k in range(self.G) if self.b[k] <= x)
        assert x < self.b[c + 1]
        return c


def positions(plan, lens):
    """Schedule 1 (mla_decode.h): tiles per sequence, first-tile positions, the partition."""
    R, U = plan.tile_tokens, plan.unit_cost
    w = [max(1, -(-L // R)) for L in lens]
    T = sum(w)
    assert plan.total_tiles == T
    X = [sum(w[:b]) + U * b for b in range(len(w))]
    return w, X, Partition(plan, T + U * max(0, len(w) - 1))


def contiguous_units(plan, lens):
    """Schedule 1 (mla_decode.h): per sequence its splits, each (start, end)."""
    R = plan.tile_tokens
    w, X, part = positions(plan, lens)
    out, start = [], 0
    for L, wb, x in zip(lens, w, X):
        cf, cl = part.cta(x), part.cta(x + wb - 1)
        for c in range(cf, cl + 1):
            lo, hi = part.lo(c), part.lo(c + 1)
            a, e = max(lo, x) - x, min(hi, x + wb) - x
            out.append((start + R * a, min(start + L, start + R * e)) if L > 0 else (start, start))
        start += max(L, 0)
    return out


def units_of(plan, lens):
    """The split ranges the plan defines (the rule stated in mla_decode.h)."""
    if plan.schedule == 1:
        return contiguous_units(plan, lens)
    out = []
    start = 0
    for L in lens:
        s = n_splits(plan, L)
        R = plan.tile_tokens
        t = -(-max(L, 0) // R)
        for i in range(s):
            out.append((start + R * (i * t // s), start + min(L, R * ((i + 1) * t // s)) if L > 0 else start))
        start += max(L, 0)
    return out


def check_contiguous(plan, lens):
    """Schedule 1: every CTA's range is within one position of its share
    (C' / G, less D for the late CTAs), no CTA is left without tiles, and the
    unit count per CTA matches the plan."""
    G, D = plan.grid, plan.late_tiles
    w, X, part = positions(plan, lens)
    L = min(G, max(0, G + plan.batch - plan.num_sms)) if D > 0 else 0
    C = part.lo(G)
    Cp = C + L * D
    for c in range(G):
        n = part.lo(c + 1) - part.lo(c) + (D if c >= G - L else 0)
        assert n in (Cp // G, -(-Cp // G)), (c, n)
    per_cta, tiles = [0] * G, [0] * G
    for wb, x in zip(w, X):
        for c in range(part.cta(x), part.cta(x + wb - 1) + 1):
            per_cta[c] += 1
            tiles[c] += min(part.lo(c + 1), x + wb) - max(part.lo(c), x)
    assert max(per_cta) == plan.units_per_cta
    assert min(tiles) >= 1, "a CTA without tiles"
    assert sum(tiles) == sum(w)


def n_splits_of(plan, lens):
    if plan.schedule == 0:
        return [n_splits(plan, L) for L in lens]
    w, X, part = positions(plan, lens)
    return [part.cta(x + wb - 1) - part.cta(x) + 1 for wb, x in zip(w, X)]


def first_rows_of(plan, lens, ind):
    """Per CTA, the first row of its first non-empty unit (mla_plan.first_row)."""
    G, R = plan.grid, plan.tile_tokens
    first = [-1] * 256
    us = units_of(plan, lens)
    if plan.schedule == 1:
        w, X, part = positions(plan, lens)
        owner = []
        for wb, x in zip(w, X):
            owner += list(range(part.cta(x), part.cta(x + wb - 1) + 1))
    else:
        owner = [u % G for u in range(len(us))]
    for (a, b), c in zip(us, owner):
        if b > a and c < 256 and first[c] < 0:
            first[c] = a + ind[0]
    return first


def check_plan(lens, dtype="fp8", num_sms=152, num_splits=0):
    ind = [0] + list(itertools.accumulate(lens))
    plan = binding.mla_decode_plan(ind, dtype, num_sms=num_sms, num_splits=num_splits)
    assert list(plan.first_row) == first_rows_of(plan, lens, ind)
    us = units_of(plan, lens)
    assert plan.num_work == len(us)
    assert plan.batch == len(lens) and plan.total_kv == ind[-1]
    if plan.schedule == 0:
        assert plan.grid == min(plan.num_work, num_sms)
        assert plan.units_per_cta == -(-plan.num_work // plan.grid)
    else:
        assert num_splits == 0 and plan.grid == min(plan.total_tiles, num_sms)
        check_contiguous(plan, lens)
    splits = n_splits_of(plan, lens)
    # contiguous, ordered, exact cover of each sequence; no empty split of a non-empty sequence
    pos = 0
    k = 0
    smax = 0
    for L, b0, s in zip(lens, ind, splits):
        smax = max(smax, s)
        assert s >= 1
        if L > 0:
            assert s <= -(-L // plan.tile_tokens)
        cur = b0
        for i in range(s):
            a, b = us[k]
            assert a == cur and b >= a
            if L > 0:
                assert b > a, "empty split"
                assert (a - b0) % plan.tile_tokens == 0, "split does not start on a tile boundary"
            cur = b
            k += 1
        assert cur == b0 + max(L, 0)
    assert plan.splits_max == smax
    return plan


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "mxfp4"])
def test_benchmark_shapes(dtype):
    for b, L in [(4, 1024), (32, 1024), (4, 8192), (64, 8192), (32, 8192), (256, 1024), (256, 8192)]:
        plan = check_plan([L] * b, dtype)
        assert plan.grid <= 152
        assert plan.tile_tokens == (64 if dtype == "bf16" else 128)


def test_forced_splits():
    for s in (1, 2, 3, 7, 64):
        plan = check_plan([1, 5, 64, 1000, 0], num_splits=s)
        assert plan.max_splits == s and plan.chunk_tokens == 1


def test_random_ragged_sweep():
    rng = random.Random(0)
    for _ in range(300):
        b = rng.randint(1, 80)
        lens = [rng.choice([0, 1, 2, rng.randint(1, 300), rng.randint(1, 20000)]) for _ in range(b)]
        sms = rng.choice([1, 7, 148, 152])
        dtype, ns = rng.choice(["bf16", "fp8", "mxfp4"]), rng.choice([0, 0, 1, 2, 5])
        if dtype == "mxfp4":
            # an MXFP4 CTA holds at most 64 units: layouts that need more are refused
            tile = 128
            need = b if ns == 0 else sum(max(1, min(ns, -(-L // tile))) if L > 0 else 1 for L in lens)
            if need > 64 * sms:
                with pytest.raises(binding.MLAError) as e:
                    binding.mla_decode_plan(np.cumsum([0] + lens).astype(np.int32), dtype, num_sms=sms,
                                            num_splits=ns)
                assert e.value.status == binding.MLA_ERR_UNSUPPORTED
                continue
        check_plan(lens, dtype, num_sms=sms, num_splits=ns)


def test_auto_plan_balances_benchmark_shapes():
    # every configuration of the benchmark fills the 152 SMs with a balanced split
    for b, L in [(32, 1024), (4, 8192), (64, 8192), (32, 8192)]:
        plan = check_plan([L] * b, "fp8")
        assert plan.grid == 152 or plan.num_work >= 128, plan.as_dict()


def test_rejects_bad_layouts():
    with pytest.raises(binding.MLAError):
        binding.mla_decode_plan([0, 5, 3], "fp8", num_sms=152)  # decreasing
    with pytest.raises(binding.MLAError):
        binding.mla_decode_plan([-1, 5], "fp8", num_sms=152)
    with pytest.raises(binding.MLAError):
        binding.mla_decode_plan([0, 5], 7, num_sms=152)


def test_paged_plan_matches_lengths():
    """A paged layout plans like the contiguous layout of the same lengths; its
    row space starts each sequence at page_indptr[b] * page_size."""
    rng = random.Random(5)
    for _ in range(60):
        b = rng.randint(1, 40)
        P = rng.choice([1, 2, 8, 16, 32, 64, 128, 256, 1024])
        npages = [rng.choice([0, 1, 2, rng.randint(1, 40)]) for _ in range(b)]
        last = [rng.randint(1, P) if n else 0 for n in npages]
        lens = [(n - 1) * P + l if n else 0 for n, l in zip(npages, last)]
        pind = [0] + list(itertools.accumulate(npages))
        dtype = rng.choice(["bf16", "fp8", "mxfp4"])
        sms = rng.choice([7, 152])
        plan = binding.mla_decode_plan_paged(pind, last, P, pind[-1] + 2, dtype, num_sms=sms)
        ref = binding.mla_decode_plan(np.cumsum([0] + lens).astype(np.int32), dtype, num_sms=sms)
        d, r = plan.as_dict(), ref.as_dict()
        assert d.pop("total_kv") == pind[-1] * P and d.pop("page_size") == P and d.pop("num_pages") == pind[-1] + 2
        r.pop("total_kv"), r.pop("page_size"), r.pop("num_pages")
        assert d == r


def test_paged_plan_rules():
    for P in (0, 3, 24, 96):  # not a power of two
        with pytest.raises(binding.MLAError) as e:
            binding.mla_decode_plan_paged([0, 1], [1], P, 1, "fp8", num_sms=152)
        assert e.value.status == binding.MLA_ERR_UNSUPPORTED
    for P in (1, 2, 4, 8, 16, 32):  # small pages: a tile's rows come from many pages
        plan = binding.mla_decode_plan_paged([0, 3], [1], P, 3, "fp8", num_sms=152)
        assert plan.page_size == P and plan.total_kv == 3 * P
    for pind, last in (([0, 2], [65]), ([0, 2], [0]), ([1, 0], [1])):  # last page length, order
        with pytest.raises(binding.MLAError) as e:
            binding.mla_decode_plan_paged(pind, last, 64, 4, "fp8", num_sms=152)
        assert e.value.status == binding.MLA_ERR_INVALID_ARG
    plan = binding.mla_decode_plan_paged([0, 0, 3], [0, 7], 64, 3, "fp8", num_sms=152)
    assert plan.total_kv == 192 and plan.page_size == 64


def test_multi_token_plan_matches_token_lengths():
    """q_len tokens per sequence plan like the batch of the tokens' visible
    lengths L_b - (q_len - 1 - i), one output row per token."""
    rng = random.Random(11)
    for _ in range(60):
        b = rng.randint(1, 30)
        q_len = rng.choice([2, 3, 4, 8])
        lens = [rng.choice([0, 1, 2, rng.randint(1, 300), rng.randint(1, 9000)]) for _ in range(b)]
        dtype = rng.choice(["bf16", "fp8", "mxfp4"])
        sms = rng.choice([7, 152])
        ind = np.cumsum([0] + lens).astype(np.int32)
        plan = binding.mla_decode_plan_multi(ind, q_len, dtype, num_sms=sms)
        if q_len == 2 and dtype == "fp8":
            continue  # the fused form (test below)
        tok = [max(0, L - (q_len - 1 - i)) for L in lens for i in range(q_len)]
        ref = binding.mla_decode_plan(np.cumsum([0] + tok).astype(np.int32), dtype, num_sms=sms)
        d, r = plan.as_dict(), ref.as_dict()
        assert d.pop("q_len") == q_len and r.pop("q_len") == 0
        assert d.pop("total_kv") == ind[-1]
        r.pop("total_kv")
        assert d.pop("tokens_fused") == 0 and r.pop("tokens_fused") == 0
        assert d == r and plan.batch == b * q_len


def test_two_token_e4m3_plan_is_fused():
    """e4m3 with two tokens per sequence: the unit list is the one-token plan
    of the sequences' full lengths, each unit serving both tokens (two output
    rows and two partial slots per unit)."""
    rng = random.Random(12)
    for _ in range(60):
        b = rng.randint(1, 40)
        lens = [rng.choice([0, 1, 2, 129, rng.randint(1, 300), rng.randint(1, 9000)]) for _ in range(b)]
        sms = rng.choice([3, 7, 152])
        splits = rng.choice([0, 0, 1, 3, 17])
        ind = np.cumsum([0] + lens).astype(np.int32)
        plan = binding.mla_decode_plan_multi(ind, 2, "fp8", num_sms=sms, num_splits=splits)
        ref = binding.mla_decode_plan(ind, "fp8", num_sms=sms, num_splits=splits)
        d, r = plan.as_dict(), ref.as_dict()
        assert (d.pop("q_len"), d.pop("tokens_fused"), d.pop("batch")) == (2, 2, 2 * b)
        for k in ("q_len", "tokens_fused", "batch"):
            r.pop(k)
        if plan.late_tiles == 0 and ref.late_tiles == 0:
            assert d.pop("num_work") == 2 * r.pop("num_work")
            assert d == r
        else:
            # the late CTAs' share follows the two output rows per sequence of
            # the query preparation: the same tiles, cut by that partition
            for k in ("num_work", "late_tiles", "units_per_cta", "splits_max"):
                d.pop(k)
                r.pop(k)
            assert d == r
            us = units_of(plan, lens)
            assert plan.num_work == 2 * len(us)
            check_contiguous(plan, lens)
            assert plan.splits_max == max(n_splits_of(plan, lens))
        assert binding.mla_decode_workspace_bytes(plan) > binding.mla_decode_workspace_bytes(ref)
    for dtype in ("bf16", "mxfp4"):
        assert binding.mla_decode_plan_multi([0, 300], 2, dtype, num_sms=152).tokens_fused == 0
    assert binding.mla_decode_plan_multi([0, 300], 3, "fp8", num_sms=152).tokens_fused == 0


def test_multi_token_plan_rules():
    for q_len in (0, 17):
        with pytest.raises(binding.MLAError) as e:
            binding.mla_decode_plan_multi([0, 10], q_len, "fp8", num_sms=152)
        assert e.value.status == binding.MLA_ERR_UNSUPPORTED


def test_two_token_slots_partition_the_workspace():
    """Two-token plans (mla_decode.h): token i of unit s of sequence b writes
    partial slot 2 ub + i S_b + s (ub = the sequence's first unit).  Over a
    batch the slots are a partition of [0, num_work), each token's slots are
    contiguous (what the combine kernel reads), and a token's last unit is
    the unit that holds its sequence's last row."""
    rng = random.Random(13)
    for _ in range(40):
        b = rng.randint(1, 50)
        lens = [rng.choice([0, 1, 2, 129, rng.randint(1, 4000), rng.randint(1, 20000)]) for _ in range(b)]
        sms = rng.choice([4, 9, 152])
        splits = rng.choice([0, 0, 3, 17])
        ind = np.cumsum([0] + lens).astype(np.int32)
        plan = binding.mla_decode_plan_multi(ind, 2, "fp8", num_sms=sms, num_splits=splits)
        one = binding.mla_decode_plan(ind, "fp8", num_sms=sms, num_splits=splits)
        S = n_splits_of(one, lens)
        assert sum(S) * 2 == plan.num_work
        seen = []
        ub = 0
        for Sb in S:
            for i in range(2):
                slots = [2 * ub + i * Sb + s for s in range(Sb)]
                assert slots == list(range(slots[0], slots[0] + Sb))
                seen += slots
            ub += Sb
        assert sorted(seen) == list(range(plan.num_work))
        units = units_of(one, lens)
        u = 0
        for bi, (L, Sb) in enumerate(zip(lens, S)):
            # the sequence's units tile its rows in order; the last one ends at its
            # last row, the only row token 0 does not see
            mine = units[u:u + Sb]
            assert mine[0][0] == ind[bi] and mine[-1][1] == ind[bi + 1]
            assert all(x[1] == y[0] for x, y in zip(mine, mine[1:]))
            assert all(x[1] > x[0] for x in mine) or L == 0
            u += Sb


def test_first_rows_follow_the_units():
    """mla_plan.first_row: per CTA, the first row of its first non-empty unit
    (rows of the device kv_indptr, which may start above 0); -1 for CTAs
    without one and for paged and multi-token plans."""
    rng = random.Random(17)
    for _ in range(60):
        lens = [rng.choice([0, 1, 130, rng.randint(1, 5000), rng.randint(1, 40000)]) for _ in range(rng.randint(1, 70))]
        base = rng.choice([0, 0, 7, 1000])
        ind = [base] + [base + x for x in itertools.accumulate(lens)]
        for dtype in ("bf16", "fp8", "mxfp4"):
            plan = binding.mla_decode_plan(ind, dtype, num_sms=rng.choice([5, 152]),
                                           num_splits=rng.choice([0, 0, 3]))
            assert list(plan.first_row) == first_rows_of(plan, lens, ind)
    m = binding.mla_decode_plan_multi([0, 300, 700], 2, "fp8", num_sms=152)
    assert set(m.first_row) == {-1}
    pg = binding.mla_decode_plan_paged([0, 2, 5], [7, 3], 8, 8, "fp8", num_sms=152)
    assert set(pg.first_row) == {-1}


@pytest.mark.parametrize("dtype,lens,late", [
    ("fp8", [8192] * 64, True), ("mxfp4", [8192] * 32, True), ("bf16", [8192] * 64, False),
    ("fp8", [1024] * 32, False),
])
def test_late_ctas_own_fewer_positions(dtype, lens, late):
    """The CTAs that start behind the query-preparation grid (the last
    G + batch - num_sms) own late_tiles positions fewer than the others; bf16
    (no query preparation) and plans too small to share have none."""
    ind = [0] + list(itertools.accumulate(lens))
    plan = binding.mla_decode_plan(ind, dtype, num_sms=152)
    assert (plan.late_tiles > 0) == late
    if plan.schedule == 0:
        return
    w, X, part = positions(plan, lens)
    sizes = [part.lo(c + 1) - part.lo(c) for c in range(plan.grid)]
    if late:
        L = plan.grid + plan.batch - plan.num_sms
        early, tail = sizes[:plan.grid - L], sizes[plan.grid - L:]
        assert min(early) - max(tail) >= plan.late_tiles - 1 and max(early) - min(tail) <= plan.late_tiles + 1
    check_plan(lens, dtype)
