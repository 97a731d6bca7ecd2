"""Pure-Python brute force for tiny cases (independent of the C oracle).

These restate the definitions a second way, for pinning the oracle:

* attention: visibility of draft node j from node i is taken from the
  ancestor *set* built recursively (anc(i) = {i} | anc(parent(i))), not from
  a parent walk; sums use math.fsum; the softmax is exp(s - max) / fsum.
* selection: a tier of size m is the unique subset X of the candidates such
  that every member of X ranks before every non-member (dominance), found by
  enumerating all subsets of size m, not by sorting.
"""

from __future__ import annotations

import itertools
import math

import numpy as np


def rank_key(score: float, index: int):
    """Sort key for 'ranks first': larger score first, NaN last, ties to lower index."""
    if math.isnan(score):
        return (1, 0.0, index)
    return (0, -score, index)  # -0.0 and +0.0 compare equal as floats


def ancestor_set(parents: list[int], i: int) -> set[int]:
    if parents[i] == -1:
        return {i}
    return {i} | ancestor_set(parents, parents[i])


def attention_row(qv, cache_k, cache_v, draft_k, draft_v, visible_draft, scale):
    """One row: qv [d]; cache_k/v lists of [d]; draft_k/v lists indexed by node; visible_draft set."""
    keys = list(cache_k) + [draft_k[j] for j in sorted(visible_draft)]
    vals = list(cache_v) + [draft_v[j] for j in sorted(visible_draft)]
    if not keys:
        return [0.0] * len(qv), -math.inf
    s = [scale * math.fsum(a * b for a, b in zip(qv, k)) for k in keys]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = math.fsum(e)
    lse = m + math.log(z)
    d = len(qv)
    o = [math.fsum(e[j] * vals[j][c] for j in range(len(keys))) / z for c in range(d)]
    return o, lse


def attention(q, k_cache, v_cache, k_draft, v_draft, parents, scale, ctx_lens=None, idx=None):
    """All rows of a tiny problem as nested lists. Tensors are plain nested Python lists.

    q [B][N][Hq][d]; k_cache [B][Hkv][L][d]; k_draft [B][N][Hkv][d] or None;
    parents [B][N]; idx [B][k] or None. Returns (out[B][N][Hq][d], lse[B][N][Hq]).
    """
    scale = float(np.float32(scale))  # the scale argument is an fp32 value
    B, N, Hq = len(q), len(q[0]), len(q[0][0])
    Hkv = len(k_cache[0])
    L = len(k_cache[0][0])
    G = Hq // Hkv
    out, lse = [], []
    for b in range(B):
        n = L if ctx_lens is None else ctx_lens[b]
        if idx is None:
            toks = list(range(n))
        else:
            toks = []
            for j, t in enumerate(idx[b]):
                if 0 <= t < n and (j == 0 or t > idx[b][j - 1]):
                    toks.append(t)
        ob, lb = [], []
        for i in range(N):
            vis = ancestor_set(parents[b], i) if k_draft is not None else set()
            oi, li = [], []
            for h in range(Hq):
                hk = h // G
                ck = [k_cache[b][hk][t] for t in toks]
                cv = [v_cache[b][hk][t] for t in toks]
                dk = [k_draft[b][j][hk] for j in range(N)] if k_draft is not None else []
                dv = [v_draft[b][j][hk] for j in range(N)] if k_draft is not None else []
                o, l_ = attention_row(q[b][i][h], ck, cv, dk, dv, vis, scale)
                oi.append(o)
                li.append(l_)
            ob.append(oi)
            lb.append(li)
        out.append(ob)
        lse.append(lb)
    return out, lse


def _dominant_subset(cands: list[int], scores, m: int) -> list[int]:
    """The unique size-m subset whose members all rank before all non-members."""
    found = []
    for X in itertools.combinations(cands, m):
        xs = set(X)
        rest = [t for t in cands if t not in xs]
        if all(rank_key(scores[a], a) < rank_key(scores[b], b) for a in X for b in rest):
            found.append(sorted(X))
    assert len(found) == 1, found
    return found[0]


def select_row(draft, target, n, sink, window, top_m, budget):
    """Selection for one row by enumeration (tiny n only)."""
    if budget >= n:
        return list(range(n)) + [-1] * (budget - n)
    s0 = min(sink, n)
    w0 = min(window, n - s0)
    C = set(range(s0)) | set(range(n - w0, n))
    R = [t for t in range(n) if t not in C]
    m = min(top_m, budget - len(C), len(R))
    D = _dominant_subset(R, draft, m)
    R2 = [t for t in R if t not in set(D)]
    f = budget - len(C) - m
    F = _dominant_subset(R2, target, f)
    chosen = sorted(C | set(D) | set(F))
    return chosen + [-1] * (budget - len(chosen))
