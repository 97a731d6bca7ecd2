"""Pins of the oracle's greedy acceptance and cache commit (no GPU).

The rule (a reading of Dustin "Workflow di Verifica", steps 4-5, under the
greedy decoding of BASTION "Risultati Sperimentali"): from the root, accept the
lowest-index child whose draft token equals the target's greedy token after the
current node; stop when none does; the bonus token is the target's token after
the last accepted node; the accepted draft K/V rows go to the cache at
[ctx, ctx + accepted). The pins below are hand-worked trees, a brute-force
characterisation over random trees, and planted mistakes that must fail them.
"""

from __future__ import annotations

import inspect
import textwrap

import numpy as np
import pytest

import oracle

# Hand-worked tree (node: parent, token):
#   0: root, 10    1: 0, 20    2: 0, 21    3: 1, 30    4: 2, 31    5: root, 11
# target_next (column 0 = after the last committed token, 1 + i = after node i):
#   [10, 21, 99, 31, 0, 0, 0]
# root wants 10 -> node 0 (node 5 has 11); after 0 wants 21 -> node 2 (not 1);
# after 2 wants target_next[3] = 31 -> node 4; after 4 wants target_next[5] = 0,
# node 4 has no child -> stop. Path [0, 2, 4], bonus target_next[5] = 0.
HAND_TOK = [[10, 20, 21, 30, 31, 11]]
HAND_PAR = [[-1, 0, 0, 1, 2, -1]]
HAND_TN = [[10, 21, 99, 31, 0, 0, 0]]


def run_pins(fn):
    """Every pin against an implementation `fn` with the oracle's signature."""
    path, n, bonus, *_ = fn(HAND_TOK, HAND_PAR, HAND_TN)
    assert list(path[0]) == [0, 2, 4, -1, -1, -1] and n[0] == 3 and bonus[0] == 0

    # the root's children all mismatch: nothing accepted, bonus = target_next[0]
    path, n, bonus, *_ = fn([[5, 6]], [[-1, 0]], [[7, 5, 6]])
    assert n[0] == 0 and bonus[0] == 7 and list(path[0]) == [-1, -1]

    # a chain that matches throughout: all N accepted, bonus = target_next[N]
    N = 5
    tok = [[100 + i for i in range(N)]]
    par = [[i - 1 for i in range(N)]]
    tn = [[100 + i for i in range(N)] + [777]]
    path, n, bonus, *_ = fn(tok, par, tn)
    assert n[0] == N and bonus[0] == 777 and list(path[0]) == list(range(N))

    # two root children carry the same token: the lower index is taken even though the
    # other one's subtree would match longer
    tok = [[1, 1, 2, 3]]
    par = [[-1, -1, 1, 2]]
    tn = [[1, 9, 2, 3, 4]]
    path, n, bonus, *_ = fn(tok, par, tn)
    assert n[0] == 1 and path[0][0] == 0 and bonus[0] == 9

    # cache commit: rows of the path in order at [ctx, ctx + n), nothing else touched
    rng = np.random.default_rng(3)
    B, Hkv, L, d = 1, 2, 12, 4
    kc = rng.standard_normal((B, Hkv, L, d))
    vc = rng.standard_normal((B, Hkv, L, d))
    kd = rng.standard_normal((B, 6, Hkv, d))
    vd = rng.standard_normal((B, 6, Hkv, d))
    out = fn(HAND_TOK, HAND_PAR, HAND_TN, kc, vc, kd, vd, [4])
    k2, v2, ctx, st = out[3], out[4], out[5], out[6]
    assert st == 0 and ctx[0] == 7
    for j, node in enumerate([0, 2, 4]):
        assert np.array_equal(k2[0, :, 4 + j], kd[0, node]) and np.array_equal(v2[0, :, 4 + j], vd[0, node])
    keep = [t for t in range(L) if not 4 <= t < 7]
    assert np.array_equal(k2[0][:, keep], kc[0][:, keep]) and np.array_equal(v2[0][:, keep], vc[0][:, keep])

    # not enough room: the rows that fit, the length grows by those, status 5
    out = fn(HAND_TOK, HAND_PAR, HAND_TN, kc, vc, kd, vd, [L - 2])
    assert out[6] == 5 and out[5][0] == L and np.array_equal(out[3][0, :, L - 1], kd[0, 2])

    # a context length outside [0, L]: nothing copied, length unchanged, status 5
    out = fn(HAND_TOK, HAND_PAR, HAND_TN, kc, vc, kd, vd, [L + 1])
    assert out[6] == 5 and out[5][0] == L + 1 and np.array_equal(out[3], kc)

    # a parent entry outside [-1, i) never makes a child, and is reported
    path, n, bonus, *rest = fn([[4, 4]], [[-1, 5]], [[4, 4, 9]])
    assert n[0] == 1 and rest[-1] == 5


def deepest_full_match(tok, par, tn):
    """Brute force: the depth of the deepest node whose whole root path matches the
    target (each node's token equals the target's token after its parent)."""
    N = len(tok)
    best = 0
    for i in range(N):
        depth, c, ok = 0, i, True
        while c >= 0:
            if tok[c] != tn[par[c] + 1]:
                ok = False
                break
            depth += 1
            c = par[c]
        if ok:
            best = max(best, depth)
    return best


def test_pins_hold_for_the_oracle():
    run_pins(oracle.accept_commit)


@pytest.mark.parametrize("seed", range(40))
def test_length_equals_deepest_fully_matching_node(seed):
    """With distinct tokens among siblings the greedy walk reaches the deepest node
    whose whole path matches; the path is that node's ancestor chain."""
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 40))
    par = [-1] + [int(rng.integers(-1, i)) for i in range(1, N)]
    tok = [0] * N
    used: dict = {}
    for i in range(N):  # distinct tokens among the children of each node
        s = used.setdefault(par[i], set())
        t = int(rng.integers(0, 6))
        while t in s:
            t += 1
        s.add(t)
        tok[i] = t
    tn = [int(rng.integers(0, 4)) for _ in range(N + 1)]
    if rng.random() < 0.5:  # make a random path match to reach long acceptances
        c = int(rng.integers(0, N))
        while c >= 0:
            tn[par[c] + 1] = tok[c]
            c = par[c]
    path, n, bonus, *_ = oracle.accept_commit([tok], [par], [tn])
    assert n[0] == deepest_full_match(tok, par, tn)
    acc = [int(x) for x in path[0][: n[0]]]
    for j, c in enumerate(acc):  # a root path, each step a matching child
        assert par[c] == (acc[j - 1] if j else -1) and tok[c] == tn[par[c] + 1]
    assert bonus[0] == tn[(acc[-1] if acc else -1) + 1]


MUTANTS = {
    "target token of the node itself": ("want = tn[b, cur + 1]", "want = tn[b, max(cur, 0)]"),
    "highest-index matching sibling": ("                    nxt = c\n                    break",
                                       "                    nxt = c"),
    "bonus after the parent of the last node": ("bonus[b] = tn[b, cur + 1]", "bonus[b] = tn[b, max(cur, 0)]"),
    "context length not advanced": ("ctx[b] = c0 + fit", "ctx[b] = c0"),
    "rows placed from position 0": ("kc[b, :, c0 + j, :]", "kc[b, :, j, :]"),
    "no capacity check": ("fit = min(int(length[b]), L - c0)", "fit = int(length[b])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_fail_a_pin(name):
    src = textwrap.dedent(inspect.getsource(oracle.accept_commit))
    old, new = MUTANTS[name]
    assert old in src, name
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    with pytest.raises((AssertionError, IndexError, ValueError)):
        run_pins(ns["accept_commit"])
