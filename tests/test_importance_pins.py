"""Pins of the oracle's target-historical importance scores (Dustin "Metodologia"), no GPU.

The score of a cache token is the sum over the chosen heads and the draft queries
of the final attention probability on it. Pins: probability mass adds up to one
per row (closed form), an explicit softmax over [cache ; tree] written out entry by
entry, context lengths, repeated heads, and planted mistakes that must fail them.
"""

from __future__ import annotations

import inspect
import textwrap

import numpy as np
import pytest
import torch

import oracle


def case(seed, B=2, N=3, Hq=4, Hkv=2, L=40, d=8):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, N, Hq, d))
    kc = rng.standard_normal((B, Hkv, L, d))
    kd = rng.standard_normal((B, N, Hkv, d))
    return q, kc, kd


def explicit(q, kc, kd, parent, heads, scale, ctx):
    """Softmax over [cache tokens < ctx ; the node itself and its ancestors], written out."""
    B, N, Hq, d = q.shape
    Hkv, L = kc.shape[1], kc.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, L))
    lse = np.zeros((B, N, Hq))
    for b in range(B):
        for i in range(N):
            anc = []
            j = i
            while j >= 0:
                anc.append(j)
                j = parent[b][j]
            for h in range(Hq):
                logits = [scale * float(q[b, i, h] @ kc[b, h // G, t]) for t in range(ctx[b])]
                logits += [scale * float(q[b, i, h] @ kd[b, j, h // G]) for j in anc]
                m = max(logits)
                z = sum(np.exp(x - m) for x in logits)
                lse[b, i, h] = m + np.log(z)
                if h in heads:
                    for t in range(ctx[b]):
                        out[b, t] += heads.count(h) * np.exp(logits[t] - m) / z
    return out, lse


def run_pins(fn):
    q, kc, kd = case(1)
    B, N, Hq = q.shape[:3]
    parent = [[-1, 0, 1], [-1, -1, 0]]
    ctx = [40, 23]
    heads = [1, 3, 3]  # head 3 listed twice counts twice; head 1 uses KV head 0 (1 // G), not 1
    scale = 0.3
    want, lse = explicit(q, kc, kd, parent, heads, scale, ctx)
    got = fn(q, kc, lse, heads, scale=scale, ctx_lens=ctx)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)
    assert np.all(got[1, 23:] == 0.0)
    # cache-only rows (lse over the cache alone): every row's mass on the cache is exactly one
    lse_cache = np.zeros((B, N, Hq))
    for b in range(B):
        for i in range(N):
            for h in range(Hq):
                s = scale * (kc[b, h // 2, : ctx[b]] @ q[b, i, h])
                lse_cache[b, i, h] = np.logaddexp.reduce(s)
    got = fn(q, kc, lse_cache, heads, scale=scale, ctx_lens=ctx)
    assert np.allclose(got.sum(axis=1), len(heads) * N, rtol=1e-12)
    # a row with lse = -inf (it attends nothing) scores nothing
    lse2 = lse_cache.copy()
    lse2[0, :, 0] = -np.inf
    got2 = fn(q, kc, lse2, [0], scale=scale, ctx_lens=ctx)
    assert np.all(got2[0] == 0.0)


def test_pins_hold_for_the_oracle():
    run_pins(oracle.importance_scores)


def test_matches_the_attention_oracle_lse():
    """The lse the attention oracle returns gives the cache's share of each row's mass: the scores
    plus the tree's share add up to one per (row, head)."""
    x_q, x_kc, x_kd = case(5, B=1, N=4, Hq=4, Hkv=2, L=30, d=128)
    parent = np.array([[-1, 0, 0, 2]], np.int32)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    q, kc, kd = t(x_q), t(x_kc), t(x_kd)
    vd = torch.zeros_like(kd)
    scale = 0.125  # exact in fp32, the precision the attention oracle takes it in
    _, lse, st = oracle.attend(q, kc, torch.zeros_like(kc), kd, vd, torch.from_numpy(parent), scale=scale)
    assert st == 0
    lse = lse.reshape(1, 4, 4)
    qf, kf, kdf = q.double().numpy(), kc.double().numpy(), kd.double().numpy()
    got = oracle.importance_scores(qf, kf, lse, [1], scale=scale)
    tree = 0.0
    for i, anc in enumerate([[0], [1, 0], [2, 0], [3, 2, 0]]):
        for j in anc:
            tree += np.exp(scale * float(qf[0, i, 1] @ kdf[0, j, 0]) - lse[0, i, 1])
    assert abs(got.sum() + tree - 4.0) < 1e-9


MUTANTS = {
    "KV head by modulo": ("kc[b, h // G, :n, :]", "kc[b, h % Hkv, :n, :]"),
    "scale dropped": ("s = scale * (qn", "s = 1.0 * (qn"),
    "row max instead of lse": ("np.exp(s - np.where(np.isfinite(row), row, 0.0))",
                               "np.exp(s - s.max(axis=1, keepdims=True))"),
    "context length ignored": ("n = int(min(max(ctx[b], 0), L))", "n = L"),
    "repeated heads counted once": ("for h in heads:", "for h in sorted(set(heads)):"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_fail_a_pin(name):
    src = textwrap.dedent(inspect.getsource(oracle.importance_scores))
    old, new = MUTANTS[name]
    assert old in src, name
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    with pytest.raises((AssertionError, ValueError, IndexError)):
        run_pins(ns["importance_scores"])
