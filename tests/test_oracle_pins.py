"""Pins of the CPU oracle against what the pages and the mathematics fix.

The oracle is only trusted because of these checks. Each one is chosen so that
a plausible slip in the oracle (dropped term, wrong sign or index, transposed
operand, off-by-one in the mask or the tiers) fails at least one of them; the
mutation tests in test_oracle_mutants.py plant such slips and check that.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_77_gb300 import workloads as W
from tests import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def tiny_problem(seed, B=2, N=5, Hq=4, Hkv=2, d=8, L=11, parents=None):
    g = torch.Generator().manual_seed(seed)
    q = _bf16((B, N, Hq, d), g)
    kc = _bf16((B, Hkv, L, d), g)
    vc = _bf16((B, Hkv, L, d), g)
    kd = _bf16((B, N, Hkv, d), g)
    vd = _bf16((B, N, Hkv, d), g)
    if parents is None:
        parents = [W.random_parents(N, 3, g) for _ in range(B)]
    par = torch.tensor(parents, dtype=torch.int32)
    return q, kc, vc, kd, vd, par


def _lists(t):
    return t.float().tolist()


# ---------------------------------------------------------------------------
# attention


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_attention_matches_bruteforce(seed):
    """Brute force with fsum and recursive ancestor sets, tiny sizes, random trees."""
    q, kc, vc, kd, vd, par = tiny_problem(seed)
    scale = 0.37
    out, lse, st = oracle.attend(q, kc, vc, kd, vd, par, scale=scale)
    assert st == 0
    bo, bl = bf.attention(_lists(q), _lists(kc), _lists(vc), _lists(kd), _lists(vd),
                          par.tolist(), scale)
    B, N, Hq, d = q.shape
    np.testing.assert_allclose(out.reshape(B, N, Hq, d), np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(B, N, Hq), np.array(bl), rtol=0, atol=1e-12)


def test_attention_bruteforce_ragged_and_sparse():
    """Ragged contexts, a sparse index set with padding, a forest."""
    parents = [[-1, -1, 0, 2, 1], [-1, 0, 0, -1, 3]]
    q, kc, vc, kd, vd, par = tiny_problem(7, parents=parents)
    ctx = torch.tensor([11, 6], dtype=torch.int32)
    idx = torch.tensor([[0, 2, 3, 7, 10, -1], [1, 4, 5, -1, -1, -1]], dtype=torch.int32)
    for ix in (None, idx):
        out, lse, st = oracle.attend(q, kc, vc, kd, vd, par, scale=0.5, ctx_lens=ctx, idx=ix)
        assert st == 0
        bo, bl = bf.attention(_lists(q), _lists(kc), _lists(vc), _lists(kd), _lists(vd), parents,
                              0.5, ctx_lens=ctx.tolist(), idx=None if ix is None else ix.tolist())
        np.testing.assert_allclose(out.reshape(q.shape), np.array(bo), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse.reshape(q.shape[:3]), np.array(bl), rtol=0, atol=1e-12)


def test_closed_form_golden():
    """Logits 0, 1, 2 give weights 1 : e : e^2 (hand-derived fixture)."""
    with open(os.path.join(GOLDEN, "attention_closed_form.json")) as f:
        c = json.load(f)
    bt = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)
    q = bt([[[c["q"]]]])  # [1,1,1,2]
    kc = bt([[c["k_cache"]]])  # [1,1,2,2]
    vc = bt([[c["v_cache"]]])
    kd = bt([[c["k_draft"]]]).reshape(1, 1, 1, 2)
    vd = bt([[c["v_draft"]]]).reshape(1, 1, 1, 2)
    par = torch.tensor([c["parent"]], dtype=torch.int32)
    out, lse, st = oracle.attend(q, kc, vc, kd, vd, par, scale=c["scale"])
    assert st == 0
    np.testing.assert_allclose(out[0], c["expected_out"], rtol=0, atol=1e-14)
    assert abs(lse[0] - c["expected_lse"]) < 1e-14


def _merge64(parts):
    """fp64 log-sum-exp merge of normalised parts [(o, lse), ...]."""
    lses = np.stack([p[1] for p in parts])  # [P, rows]
    m = np.max(lses, axis=0)
    tot = m + np.log(np.sum(np.exp(lses - m), axis=0))
    o = sum(np.exp(p[1] - tot)[:, None] * p[0] for p in parts)
    return o, tot


@pytest.mark.parametrize("splits", [[0, 11], [0, 4, 11], [0, 1, 5, 6, 11]])
def test_lse_merge_of_parts_equals_monolithic(splits):
    """LongSpec section 2.C: cache part (no mask) and tree part merged by LSE = one softmax.

    Also for any split of the cache into ranges (the split-KV reduction).
    """
    q, kc, vc, kd, vd, par = tiny_problem(11)
    full_o, full_l, _ = oracle.attend(q, kc, vc, kd, vd, par, scale=0.3)
    parts = []
    for t0, t1 in zip(splits[:-1], splits[1:]):
        o, l_, _ = oracle.attend(q, kc, vc, None, None, par, scale=0.3, cache_range=(t0, t1))
        parts.append((o, l_))
    # tree part alone: empty cache range
    o, l_, _ = oracle.attend(q, kc, vc, kd, vd, par, scale=0.3, cache_range=(0, 0))
    parts.append((o, l_))
    mo, ml = _merge64(parts)
    np.testing.assert_allclose(mo, full_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, full_l, rtol=0, atol=1e-12)


def test_oracle_lse_merge_function():
    """The fp64 merge routine on fp32 parts: identity with monolithic to fp32 rounding,
    an empty part (lse=-inf) is neutral, two equal parts add log 2 to lse."""
    q, kc, vc, kd, vd, par = tiny_problem(12)
    full_o, full_l, _ = oracle.attend(q, kc, vc, kd, vd, par, scale=0.3)
    ca, la, _ = oracle.attend(q, kc, vc, None, None, par, scale=0.3)
    cb, lb, _ = oracle.attend(q, kc, vc, kd, vd, par, scale=0.3, cache_range=(0, 0))
    mo, ml = oracle.lse_merge(ca.astype(np.float32), la.astype(np.float32),
                              cb.astype(np.float32), lb.astype(np.float32))
    np.testing.assert_allclose(mo, full_o, rtol=0, atol=1e-6)
    np.testing.assert_allclose(ml, full_l, rtol=0, atol=1e-5)
    # merge order does not matter
    mo2, ml2 = oracle.lse_merge(cb.astype(np.float32), lb.astype(np.float32),
                                ca.astype(np.float32), la.astype(np.float32))
    np.testing.assert_allclose(mo2, mo, rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml2, ml, rtol=0, atol=1e-15)
    # empty part
    rows, d = ca.shape
    empty_o = np.zeros((rows, d), np.float32)
    empty_l = np.full((rows,), -np.inf, np.float32)
    eo, el = oracle.lse_merge(ca.astype(np.float32), la.astype(np.float32), empty_o, empty_l)
    np.testing.assert_array_equal(eo, ca.astype(np.float32).astype(np.float64))
    np.testing.assert_array_equal(el, la.astype(np.float32).astype(np.float64))
    eo, el = oracle.lse_merge(empty_o, empty_l, empty_o, empty_l)
    assert np.all(el == -np.inf) and np.all(eo == 0)
    # equal parts
    so, sl = oracle.lse_merge(ca.astype(np.float32), la.astype(np.float32),
                              ca.astype(np.float32), la.astype(np.float32))
    np.testing.assert_allclose(so, ca.astype(np.float32), rtol=0, atol=1e-7)
    np.testing.assert_allclose(sl, la.astype(np.float32).astype(np.float64) + math.log(2), atol=1e-12)


@pytest.mark.parametrize("L", [0, 9])
def test_chain_equals_causal_attention(L):
    """A chain tree is causal attention over [cache ; draft] (library SDPA, fp64, explicit mask)."""
    B, N, Hq, Hkv, d = 2, 6, 4, 2, 16
    q, kc, vc, kd, vd, par = tiny_problem(21, B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, L=max(L, 1),
                                         parents=[W.chain_parents(N)] * B)
    kc, vc = kc[:, :, :L], vc[:, :, :L]
    scale = 1.0 / math.sqrt(d)
    out, lse, st = oracle.attend(q, kc, vc, kd, vd, par, scale=scale)
    assert st == 0
    G = Hq // Hkv
    qq = q.double().permute(0, 2, 1, 3)  # [B,Hq,N,d]
    kk = torch.cat([kc.double(), kd.double().permute(0, 2, 1, 3)], dim=2).repeat_interleave(G, dim=1)
    vv = torch.cat([vc.double(), vd.double().permute(0, 2, 1, 3)], dim=2).repeat_interleave(G, dim=1)
    mask = torch.ones(N, L + N, dtype=torch.bool)
    mask[:, L:] = torch.tril(torch.ones(N, N, dtype=torch.bool))
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
    ref = ref.permute(0, 2, 1, 3).reshape(-1, d).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # lse against torch.logsumexp of the masked logits
    logits = torch.einsum("bhnd,bhtd->bhnt", qq, kk) * scale
    logits = logits.masked_fill(~mask, -math.inf)
    ref_l = torch.logsumexp(logits, dim=-1).permute(0, 2, 1).reshape(-1).numpy()
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_budget_covering_context_equals_dense():
    """Dustin: a budget that covers the context is full verification (bit-for-bit in the oracle)."""
    q, kc, vc, kd, vd, par = tiny_problem(31)
    B, L = q.shape[0], kc.shape[2]
    idx = torch.tensor([list(range(L)) + [-1, -1]] * B, dtype=torch.int32)
    do, dl, _ = oracle.attend(q, kc, vc, kd, vd, par, scale=0.4)
    so, sl, st = oracle.attend(q, kc, vc, kd, vd, par, scale=0.4, idx=idx)
    assert st == 0
    np.testing.assert_array_equal(so, do)
    np.testing.assert_array_equal(sl, dl)


def test_closed_forms():
    """Constant V; identical keys; no cache (N=1); star tree = node alone with the cache."""
    B, N, Hq, Hkv, d, L = 1, 4, 2, 1, 8, 7
    q, kc, vc, kd, vd, par = tiny_problem(41, B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, L=L)
    # constant V -> o = c
    c = 0.75
    out, _, _ = oracle.attend(q, kc, torch.full_like(vc, c), kd, torch.full_like(vd, c), par, scale=0.5)
    np.testing.assert_allclose(out, c, rtol=0, atol=1e-15)
    # identical keys (cache and draft) -> uniform weights over visible keys
    kone = kc[:, :, :1].expand_as(kc).contiguous()
    kdone = kc[:, :, 0].reshape(B, 1, Hkv, d).expand(B, N, Hkv, d).contiguous()
    parents = [[-1, 0, 1, 0]]
    par = torch.tensor(parents, dtype=torch.int32)
    out, lse, _ = oracle.attend(q, kone, vc, kdone, vd, par, scale=0.5)
    for i in range(N):
        anc = bf.ancestor_set(parents[0], i)
        vis_v = [vc[0, 0, t].double() for t in range(L)] + [vd[0, j, 0].double() for j in sorted(anc)]
        mean = torch.stack(vis_v).mean(0).numpy()
        for h in range(Hq):
            r = i * Hq + h
            s = 0.5 * float((q[0, i, h].double() * kc[0, 0, 0].double()).sum())
            np.testing.assert_allclose(out[r], mean, rtol=0, atol=1e-13)
            assert abs(lse[r] - (s + math.log(L + len(anc)))) < 1e-12
    # no cache, single node: o = v_draft, lse = own logit
    kc0, vc0 = kc[:, :, :0], vc[:, :, :0]
    par1 = torch.tensor([[-1]], dtype=torch.int32)
    out, lse, _ = oracle.attend(q[:, :1], kc0, vc0, kd[:, :1], vd[:, :1], par1, scale=0.5)
    for h in range(Hq):
        np.testing.assert_array_equal(out[h], vd[0, 0, 0].double().numpy())
        s = 0.5 * float((q[0, 0, h].double() * kd[0, 0, 0].double()).sum())
        assert abs(lse[h] - s) < 1e-13
    # star tree: node i sees the cache and itself = a one-node problem for node i
    star = torch.full((1, N), -1, dtype=torch.int32)
    out, lse, _ = oracle.attend(q, kc, vc, kd, vd, star, scale=0.5)
    for i in range(N):
        o1, l1, _ = oracle.attend(q[:, i:i + 1], kc, vc, kd[:, i:i + 1], vd[:, i:i + 1], par1, scale=0.5)
        np.testing.assert_array_equal(out[i * Hq:(i + 1) * Hq], o1)
        np.testing.assert_array_equal(lse[i * Hq:(i + 1) * Hq], l1)


@pytest.mark.parametrize("pos", [0, 63, 64, 127, 128, 1000, 2047])
def test_needle(pos):
    """One key with logit +30 at a chosen position: o is that key's value."""
    B, N, Hq, Hkv, d, L = 1, 2, 4, 2, 128, 2048
    g = torch.Generator().manual_seed(pos)
    q = _bf16((B, N, Hq, d), g)
    kc = _bf16((B, Hkv, L, d), g, 0.05)
    vc = _bf16((B, Hkv, L, d), g)
    kd = _bf16((B, N, Hkv, d), g, 0.05)
    vd = _bf16((B, N, Hkv, d), g)
    par = torch.tensor([[-1, 0]], dtype=torch.int32)
    scale = 1.0 / math.sqrt(d)
    # needle for kv head 1, query head 2 (G=2 -> head 2 maps to kv head 1), node 0
    qv = q[0, 0, 2].double()
    kn = (qv * (30.0 / (scale * float(qv.dot(qv))))).to(torch.bfloat16)
    kc[0, 1, pos] = kn
    out, lse, _ = oracle.attend(q, kc, vc, kd, vd, par, scale=scale, rows=[2])
    np.testing.assert_allclose(out[0], vc[0, 1, pos].double().numpy(), rtol=0, atol=1e-6)
    assert abs(lse[0] - scale * float(qv.dot(kn.double()))) < 1e-6
    # the needle is invisible through a sparse set that skips it
    idx = torch.tensor([[t for t in range(0, L, 2) if t != pos]], dtype=torch.int32)
    out2, _, _ = oracle.attend(q, kc, vc, kd, vd, par, scale=scale, rows=[2], idx=idx)
    assert np.abs(out2[0] - vc[0, 1, pos].double().numpy()).max() > 0.1


def test_bad_inputs_are_reported():
    """Parent outside [-1, i) and non-ascending / out-of-range indices: masked, status 5."""
    q, kc, vc, kd, vd, par = tiny_problem(51, parents=[[-1, 0, 1, 2, 3], [-1, 0, 1, 2, 3]])
    bad = par.clone()
    bad[0, 3] = 3  # self-parent
    _, _, st = oracle.attend(q, kc, vc, kd, vd, bad, scale=0.5)
    assert st == 5
    idx = torch.tensor([[0, 5, 5, 2, 20, -1], [1, 2, 3, -1, -1, -1]], dtype=torch.int32)
    o_bad, l_bad, st = oracle.attend(q, kc, vc, kd, vd, par, scale=0.5, idx=idx)
    assert st == 5
    # the bad entries are skipped: same as the clean set {0, 5} for sequence 0
    clean = torch.tensor([[0, 5, -1, -1, -1, -1], [1, 2, 3, -1, -1, -1]], dtype=torch.int32)
    o_ok, l_ok, st = oracle.attend(q, kc, vc, kd, vd, par, scale=0.5, idx=clean)
    assert st == 0
    np.testing.assert_array_equal(o_bad, o_ok)
    np.testing.assert_array_equal(l_bad, l_ok)


# ---------------------------------------------------------------------------
# selection


def _parse(vals):
    return np.array([float(v) for v in vals], dtype=np.float32)


def test_selection_golden():
    with open(os.path.join(GOLDEN, "select_hand.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        ds = _parse(c["draft"])[None]
        ts = _parse(c["target"])[None]
        idx, cnt, st = oracle.select(ds, ts, sink=c["sink"], window=c["window"], top_m=c["top_m"],
                                     budget=c["budget"], ctx_lens=np.array([c["ctx_len"]], np.int32))
        assert st == 0
        exp = c["expected"] + [-1] * (c["budget"] - len(c["expected"]))
        assert idx[0].tolist() == exp, c["name"]
        assert cnt[0] == min(c["budget"], c["ctx_len"])


@pytest.mark.parametrize("seed", range(6))
def test_selection_matches_bruteforce(seed):
    """Enumeration of all tier subsets (dominance), tiny L, with ties, NaN and +-0."""
    rng = np.random.default_rng(seed)
    L = 12
    B = 4
    vals = np.array([0.0, -0.0, 1.0, 2.0, -1.0, np.nan, np.inf, -np.inf, 0.5], np.float32)
    ds = rng.choice(vals, size=(B, L)).astype(np.float32)
    ts = rng.choice(vals, size=(B, L)).astype(np.float32)
    ctx = np.array([12, 11, 9, 5], np.int32)
    for sink, window, top_m, budget in [(1, 2, 2, 7), (0, 0, 3, 5), (2, 1, 0, 6), (1, 1, 9, 8), (3, 3, 1, 6)]:
        idx, cnt, st = oracle.select(ds, ts, sink=sink, window=window, top_m=top_m, budget=budget,
                                     ctx_lens=ctx)
        assert st == 0
        for b in range(B):
            exp = bf.select_row(ds[b].tolist(), ts[b].tolist(), int(ctx[b]), sink, window, top_m, budget)
            assert idx[b].tolist() == exp, (b, sink, window, top_m, budget)


def test_selection_invariants_large():
    """Config-3 shaped rows: sink and window kept, |I| = budget, ascending unique,
    tier D = the m largest draft scores outside sink/window (library lexsort), and
    every unselected candidate has target score <= every fill token's."""
    B, L, S, Wn, m, k = 3, 32768, 4, 64, 512, 2048
    ds, ts = W.random_scores(B, L, seed=9)
    ds, ts = ds.numpy(), ts.numpy()
    idx, cnt, st = oracle.select(ds, ts, sink=S, window=Wn, top_m=m, budget=k)
    assert st == 0
    for b in range(B):
        I = idx[b]
        assert cnt[b] == k and np.all(I >= 0)
        assert np.all(np.diff(I) > 0)
        Is = set(I.tolist())
        assert set(range(S)) <= Is and set(range(L - Wn, L)) <= Is
        R = np.arange(S, L - Wn)
        order = np.lexsort((R, -ds[b, R]))  # by score desc, then index asc
        D = set(R[order[:m]].tolist())
        assert D <= Is
        F = Is - D - set(range(S)) - set(range(L - Wn, L))
        assert len(F) == k - S - Wn - m
        rest = np.array(sorted(set(R.tolist()) - Is))
        fmin = min(ts[b, list(F)])
        assert ts[b, rest].max() <= fmin


def test_selection_all_equal_scores():
    """All-equal scores: every tier takes the lowest indices available to it."""
    L, k = 100, 30
    ds = np.full((1, L), 0.25, np.float32)
    ts = np.full((1, L), 0.25, np.float32)
    idx, _, _ = oracle.select(ds, ts, sink=4, window=6, top_m=10, budget=k)
    exp = list(range(4)) + list(range(4, 24)) + list(range(94, 100))
    assert idx[0].tolist() == exp


# ---------------------------------------------------------------------------
# workload generator (input side)


def test_workloads_are_deterministic():
    w = W.workload(1)
    a = W.make_inputs(w)
    b = W.make_inputs(w)
    for key in ("q", "k_cache", "v_cache", "k_draft", "v_draft", "parent"):
        assert torch.equal(a[key], b[key])
    c = W.make_inputs(w, seed=77)
    assert not torch.equal(a["q"], c["q"])


def test_random_tree_shape():
    g = torch.Generator().manual_seed(5)
    for depth_max in (1, 3, 8):
        p = W.random_parents(64, depth_max, g)
        depth = []
        for i, pi in enumerate(p):
            assert -1 <= pi < i
            depth.append(1 if pi == -1 else depth[pi] + 1)
        assert max(depth) <= depth_max


def test_best_first_golden():
    with open(os.path.join(GOLDEN, "best_first_hand.json")) as f:
        c = json.load(f)
    t = W.best_first_tree(np.array(c["marginals"]), c["N"])
    assert t.parents == c["expected_parents"]
    assert t.depth == c["expected_depth"]
    np.testing.assert_allclose(t.rho, c["expected_rho"], rtol=1e-12)
    assert abs(sum(t.rho) - c["expected_surrogate"]) < 1e-12


def _all_prefix_closed_best(marginals, N):
    """Brute force: max of sum(rho) over prefix-closed subtrees with N nodes."""
    import itertools

    block, nc = marginals.shape
    nodes = []  # (path tuple)
    for dpt in range(1, block + 1):
        nodes += list(itertools.product(range(nc), repeat=dpt))
    rho = {p: float(np.prod([marginals[k, c] for k, c in enumerate(p)])) for p in nodes}
    best = -1.0
    for S in itertools.combinations(nodes, N):
        s = set(S)
        if all(len(p) == 1 or p[:-1] in s for p in S):
            best = max(best, sum(rho[p] for p in S))
    return best


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_best_first_is_optimal_and_concave(seed):
    """BASTION section 2: best-first maximises sum(rho) at every budget; gains shrink."""
    rng = np.random.default_rng(seed)
    marg = W.dirichlet_marginals(rng, 3, 2, 0.3)
    full = W.best_first_tree(marg, 14)
    # popped path scores are non-increasing, the tree is prefix-closed
    assert all(a >= b for a, b in zip(full.rho, full.rho[1:]))
    for i, p in enumerate(full.parents):
        assert -1 <= p < i
        if p >= 0:
            assert full.depth[i] == full.depth[p] + 1
    for n in range(1, 8):
        t = W.best_first_tree(marg, n)
        assert abs(sum(t.rho) - _all_prefix_closed_best(marg, n)) < 1e-12
    gains = full.rho  # marginal gain of node n is its rho: non-increasing = concave surrogate
    assert all(g1 >= g2 for g1, g2 in zip(gains, gains[1:]))


# ---------------------------------------------------------------------------
# paged cache (the same cache in fixed-size blocks of a pool, through a block table)


def to_pool(kc, vc, bs, gen, extra=3):
    """Scatter the caches [B, Hkv, L, d] into a pool of blocks of bs rows, in a random block
    order with `extra` unused blocks of noise and one guard block past the end (never named by
    a valid entry). Returns (k_pool, v_pool, table [B, nb + 2], num_blocks): table slots past a
    sequence's blocks hold -7."""
    B, Hkv, L, d = kc.shape
    nb = (L + bs - 1) // bs
    total = B * nb + extra
    perm = torch.randperm(total, generator=gen)
    kp = _bf16((total + 1, Hkv, bs, d), gen)
    vp = _bf16((total + 1, Hkv, bs, d), gen)
    table = torch.full((B, nb + 2), -7, dtype=torch.int32)
    for b in range(B):
        for j in range(nb):
            blk = int(perm[b * nb + j])
            table[b, j] = blk
            t0, t1 = j * bs, min(L, (j + 1) * bs)
            kp[blk, :, : t1 - t0] = kc[b, :, t0:t1]
            vp[blk, :, : t1 - t0] = vc[b, :, t0:t1]
    return kp, vp, table, total


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_paged_equals_contiguous(bs):
    """Paged = contiguous, bit for bit: dense and sparse, full and ragged contexts."""
    q, kc, vc, kd, vd, par = tiny_problem(40 + bs, L=37)
    g = torch.Generator().manual_seed(bs)
    kp, vp, table, nblk = to_pool(kc, vc, bs, g)
    cl = torch.tensor([37, 20], dtype=torch.int32)
    idx = torch.tensor([[0, 3, 4, 9, 17, 30, 36, -1], [1, 2, 5, 8, 13, 19, -1, -1]], dtype=torch.int32)
    for kw in (dict(), dict(ctx_lens=cl), dict(idx=idx), dict(idx=idx, ctx_lens=cl)):
        ro, rl, rs = oracle.attend(q, kc, vc, kd, vd, par, scale=0.3, **kw)
        po, pl, ps = oracle.attend_paged(q, kp, vp, kd, vd, par, table, L=37, scale=0.3, num_blocks=nblk, **kw)
        assert rs == ps == 0
        assert np.array_equal(ro, po) and np.array_equal(rl, pl)


@pytest.mark.parametrize("bad", [-1, "pool_size"])
def test_paged_bad_block_entry(bad):
    """A block entry outside the pool hides its tokens and is reported: the result equals the
    contiguous sparse attention over the other tokens."""
    q, kc, vc, kd, vd, par = tiny_problem(50, L=37)
    bs = 4
    g = torch.Generator().manual_seed(5)
    kp, vp, table, nblk = to_pool(kc, vc, bs, g)
    table[1, 2] = -1 if bad == -1 else nblk
    po, pl, ps = oracle.attend_paged(q, kp, vp, kd, vd, par, table, L=37, scale=0.3, num_blocks=nblk)
    assert ps == 5
    keep = [t for t in range(37) if not 8 <= t < 12]
    idx = torch.tensor([list(range(37)), keep + [-1] * 4], dtype=torch.int32)
    ro, rl, rs = oracle.attend(q, kc, vc, kd, vd, par, scale=0.3, idx=idx)
    assert rs == 0
    assert np.array_equal(ro, po) and np.array_equal(rl, pl)


def test_paged_entries_past_the_context_are_not_read():
    q, kc, vc, kd, vd, par = tiny_problem(51, L=37)
    bs = 4
    g = torch.Generator().manual_seed(6)
    kp, vp, table, nblk = to_pool(kc, vc, bs, g)
    cl = torch.tensor([37, 9], dtype=torch.int32)
    table[1, 3:] = -5  # blocks 3.. of sequence 1 lie past its 9 tokens
    po, pl, ps = oracle.attend_paged(q, kp, vp, kd, vd, par, table, L=37, scale=0.3, ctx_lens=cl, num_blocks=nblk)
    ro, rl, rs = oracle.attend(q, kc, vc, kd, vd, par, scale=0.3, ctx_lens=cl)
    assert ps == rs == 0
    assert np.array_equal(ro, po) and np.array_equal(rl, pl)


# ---------------------------------------------------------------------------
# fp8 cache (E4M3 codes, value = the code's number times a scale per sequence and KV head)


def test_e4m3_decoding_table():
    """Every code against torch's own float8_e4m3fn conversion (an independent implementation of
    the OCP E4M3 format), and the format's landmarks by hand: subnormals m * 2^-9, bias 7, the
    largest number 448, no infinities, S.1111.111 = NaN."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for c in range(256):
        got, want = oracle.e4m3_value(c), float(ref[c])
        assert (math.isnan(got) and math.isnan(want)) or got == want, (c, got, want)
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
            0x77: 240.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    for c, v in hand.items():
        assert oracle.e4m3_value(c) == v, hex(c)
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    assert math.copysign(1.0, oracle.e4m3_value(0x80)) == -1.0


def fp8_codes(shape, gen):
    """E4M3 codes with a random sign, exponent field 0..8 (subnormals included) and mantissa:
    numbers of magnitude below 4, so that scores stay moderate."""
    sign = torch.randint(0, 2, shape, generator=gen) << 7
    exp_ = torch.randint(0, 9, shape, generator=gen) << 3
    man = torch.randint(0, 8, shape, generator=gen)
    return (sign | exp_ | man).to(torch.uint8)


def fp8_problem(seed, B=2, N=5, Hq=8, Hkv=2, L=150, d=128):
    """A bf16 problem (queries, draft block, tree) with an E4M3 cache and power-of-two scales per
    (sequence, KV head); also the bf16 cache holding exactly the numbers the codes stand for."""
    g = torch.Generator().manual_seed(seed)
    x = W.make_inputs(W.Workload("fp8", B=B, L=L, Hq=Hq, Hkv=Hkv, N=N, tree="random", depth_max=3, seed=seed))
    kc, vc = fp8_codes((B, Hkv, L, d), g), fp8_codes((B, Hkv, L, d), g)
    ks = 2.0 ** torch.randint(-3, 3, (B, Hkv), generator=g).to(torch.float32)
    vs = 2.0 ** torch.randint(-3, 3, (B, Hkv), generator=g).to(torch.float32)

    def values(codes, sc):  # exact: a 4-bit mantissa times a power of two fits bf16
        v = codes.view(torch.float8_e4m3fn).to(torch.float32) * sc[:, :, None, None]
        return v.to(torch.bfloat16)

    return x, kc, vc, ks, vs, values(kc, ks), values(vc, vs)


@pytest.mark.parametrize("mode", ["dense", "sparse", "ragged"])
def test_fp8_equals_bf16_on_the_numbers_it_stands_for(mode):
    x, kc, vc, ks, vs, kb, vb = fp8_problem(11 if mode == "dense" else 12)
    B, L = kc.shape[0], kc.shape[2]
    kw = {}
    if mode == "sparse":
        ds, ts = W.random_scores(B, L, seed=5)
        idx = torch.from_numpy(oracle.select(ds, ts, sink=4, window=16, top_m=20, budget=64)[0])
        kw["idx"] = idx
    if mode == "ragged":
        kw["ctx_lens"] = torch.tensor([L, 37], dtype=torch.int32)
    o8, l8, s8 = oracle.attend_fp8(x["q"], kc, vc, ks, vs, x["k_draft"], x["v_draft"], x["parent"],
                                   scale=x["scale"], **kw)
    ob, lb, sb = oracle.attend(x["q"], kb, vb, x["k_draft"], x["v_draft"], x["parent"], scale=x["scale"], **kw)
    assert s8 == sb == 0
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_fp8_v_scale_scales_the_cache_output_only():
    """No draft block: doubling every V scale doubles out exactly and leaves lse alone; doubling
    every K scale while halving the softmax scale changes nothing."""
    x, kc, vc, ks, vs, _, _ = fp8_problem(13)
    args = (x["q"], kc, vc)
    o1, l1, _ = oracle.attend_fp8(*args, ks, vs, None, None, None, scale=x["scale"])
    o2, l2, _ = oracle.attend_fp8(*args, ks, 2 * vs, None, None, None, scale=x["scale"])
    o3, l3, _ = oracle.attend_fp8(*args, 2 * ks, vs, None, None, None, scale=x["scale"] / 2)
    assert np.array_equal(o2, 2 * o1) and np.array_equal(l2, l1)
    assert np.array_equal(o3, o1) and np.array_equal(l3, l1)
