"""The tensor-core cache kernel's split plan (spec_split_plan, host logic, no GPU).

The plan decides which KV tiles each CTA covers and which partial slot each (CTA, unit) pair
writes; the merge finds the partials of a unit from the same plan. These checks hold for every
shape: the ranges tile [0, total) in order, empty ranges come only at the end, every (CTA, unit)
pair has its own slot inside the workspace's slot count, row groups get blocks of CTAs with the
same cut, dense plans are balanced against the cost of entering a unit, sparse plans without row
groups are an even cut, and a dense and a sparse call of one shape take the same CTA count (one
workspace size serves both).
"""

from __future__ import annotations

import itertools
import math

import pytest

from speculative_decoding_verification_77_gb300 import ops

TILE = 128
UNIT_SWITCH_TILES = 4  # the balanced plan's charge for entering a unit after the first


def shape_grid():
    heads = [(32, 8), (64, 8), (8, 2), (12, 4), (4, 1), (16, 2)]
    for (B, N, (Hq, Hkv), L, sms) in itertools.product([1, 3, 16], [1, 8, 17, 64, 130, 256], heads,
                                                       [1, 90, 2048, 16384, 131072], [152, 148, 7]):
        yield B, N, Hq, Hkv, L, sms


def ranges(plan):
    s = plan["starts"]
    return [(s[c], s[c + 1]) for c in range(plan["ctas"])]


def units_of(lo, hi, tpu):
    return range(lo // tpu, (hi - 1) // tpu + 1) if hi > lo else range(0)


def cost(lo, hi, tpu):
    """Tiles plus the charge for every unit entered after the first."""
    return (hi - lo) + UNIT_SWITCH_TILES * max(0, len(units_of(lo, hi, tpu)) - 1)


def check(B, N, Hq, Hkv, L, sms, sparse):
    p = ops.split_plan(B, N, Hq, Hkv, L, sms=sms, sparse=sparse)
    G = Hq // Hkv
    M = G * N
    BM = 256 if M > 128 else 128
    rg = math.ceil(M / BM)
    tpu = max(1, math.ceil(L / TILE))
    units = B * Hkv * rg
    total = units * tpu
    assert (p["BM"], p["row_groups"], p["units"], p["tiles_per_unit"]) == (BM, rg, units, tpu)
    assert p["split_tiles"] == (1 if M <= 128 else 0) and p["pipes"] == 2
    ctas = p["ctas"]
    assert 1 <= ctas <= min(sms, total, 512)
    s = p["starts"]
    assert s[0] == 0 and s[ctas] == total
    assert all(a <= b for a, b in zip(s, s[1:]))
    rs = ranges(p)
    sizes = [hi - lo for lo, hi in rs]
    first_empty = next((c for c, n in enumerate(sizes) if n == 0), ctas)
    assert all(n == 0 for n in sizes[first_empty:]), "empty ranges only at the end"
    # every (CTA, unit) pair writes partial slot c + u: distinct, inside the workspace's slots
    pairs = [(c, u) for c, (lo, hi) in enumerate(rs) for u in units_of(lo, hi, tpu)]
    slots = [c + u for c, u in pairs]
    assert len(set(slots)) == len(slots)
    assert max(slots) < ctas + units - 1 or (ctas == 1 and units == 1)
    assert p["slots"] == (ctas + units - 1) * p["pipes"]
    # every unit is covered, each of its tiles by exactly one CTA (the ranges tile [0, total))
    assert sorted({u for _, u in pairs}) == list(range(units))
    if rg > 1 and min(sms, total, 512) >= rg:
        # one block of CTAs per row group, the same even cut in each
        assert ctas % rg == 0 and p["uniform"] == 0
        per, blk = ctas // rg, total // rg
        cut0 = [s[i] for i in range(per + 1)]
        for r in range(rg):
            assert [s[r * per + i] - r * blk for i in range(per + 1)] == cut0
        assert max(sizes) - min(sizes) <= 1
    elif sparse:
        assert p["uniform"] == 1 and max(sizes) - min(sizes) <= 1
        assert sizes == sorted(sizes, reverse=True)  # the first `rem` CTAs take one tile more
    else:
        # balanced: no CTA costs more than in the even cut with the same CTA count
        q, rem = divmod(total, ctas)
        even = [(c * q + min(c, rem), (c + 1) * q + min(c + 1, rem)) for c in range(ctas)]
        assert max(cost(lo, hi, tpu) for lo, hi in rs) <= max(cost(lo, hi, tpu) for lo, hi in even)
    return p


@pytest.mark.parametrize("sparse", [False, True])
def test_split_plan_invariants(sparse):
    n = 0
    for B, N, Hq, Hkv, L, sms in shape_grid():
        check(B, N, Hq, Hkv, L, sms, sparse)
        n += 1
    assert n > 1000


def test_dense_and_sparse_take_one_cta_count():
    for B, N, Hq, Hkv, L, sms in shape_grid():
        d = ops.split_plan(B, N, Hq, Hkv, L, sms=sms)
        s = ops.split_plan(B, N, Hq, Hkv, L, sms=sms, sparse=True)
        assert (d["ctas"], d["slots"]) == (s["ctas"], s["slots"]), (B, N, Hq, Hkv, L, sms)


def test_bench_workload_plans():
    """The plans behind the measured numbers: the headline's balanced cut over 32 units, the sparse
    workload's even cut, and four 38-CTA row-group blocks at N = 256."""
    head = check(4, 64, 32, 8, 32768, 152, False)
    assert head["ctas"] == 152 and head["units"] == 32 and head["uniform"] == 0
    sp = check(16, 8, 32, 8, 2048, 152, True)
    assert sp["ctas"] == 152 and sp["uniform"] == 1 and sp["split_tiles"] == 1
    n256 = check(8, 256, 32, 8, 16384, 152, False)
    assert n256["row_groups"] == 4 and n256["ctas"] == 152
    assert n256["starts"][38] == 8 * 8 * 128  # the second row group's block starts on its first tile


def test_rejections():
    with pytest.raises(ops.SpecError):
        ops.split_plan(1, 1, 3, 2, 100, sms=152)  # Hq not a multiple of Hkv
    with pytest.raises(ops.SpecError):
        ops.split_plan(1, 1, 4, 1, 100, sms=0)
    with pytest.raises(ops.SpecError):
        ops.split_plan(1 << 20, 256, 64, 8, 1 << 20, sms=152)  # beyond the 32-bit tile numbering


def _align(n, a=256):
    return (n + a - 1) // a * a


def test_workspace_holds_the_plans_partials():
    """spec_verify_workspace_size covers the header, the plan's fp32 partial rows (o and lse, one
    slot of 128 rows per (CTA, unit, pipe)) and the paged index scratch, for the SM count it sizes
    for (the current device's, 160 on a machine without one), dense and sparse alike."""
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 160
    lib = ops.load_library()
    d = 128
    for B, N, Hq, Hkv, L, _ in shape_grid():
        ws = lib.spec_verify_workspace_size(B, N, Hq, Hkv, d, L)
        for sparse in (False, True):
            p = ops.split_plan(B, N, Hq, Hkv, L, sms=sms, sparse=sparse)
            rows = p["slots"] * 128
            need = 256 + _align(rows * d * 4) + _align(rows * 4) + _align(B * L * 4)
            assert ws >= need, (B, N, Hq, Hkv, L, sparse, ws, need)
