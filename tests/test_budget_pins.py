"""Pins of the oracle's budget controller (BASTION "Metodologia" sections 1-3), no GPU.

Hand-worked trees and stop points, brute-force optimality of the best-first
surrogate over every prefix-closed tree on tiny inputs, exact recovery of the
latency calibration, and planted mistakes that must fail the pins.
"""

from __future__ import annotations

import inspect
import itertools
import json
import os
import textwrap

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HAND_Q = [[0.6, 0.4], [0.7, 0.3], [0.9, 0.1]]
# Linear cost: bandwidth-bound roofline T_roof(N) = N (bytes0 = 0, one byte per node, bw = 1),
# calibration samples on the roofline itself (a = 1, c = 0), t_draft = 1, l_ar = 1:
# C(N) = 1 + N. Path scores in pop order 0.6, 0.42, 0.4, 0.378, 0.28 (the golden tree), so
# A = 0.6, 1.02, 1.42, 1.798, 2.078 and S = A / (1 + N) = 0.3, 0.34, 0.355, 0.3596, 0.34633:
# S first falls at N = 5, the chosen size is 4.
HAND_COST = dict(t_draft=1.0, l_ar=1.0, bytes0=0.0, bytes_per_node=1.0, flops_per_node=0.0, bw=1.0, peak=1.0,
                 cal_n=[1, 2, 4], cal_t=[1.0, 2.0, 4.0])


def run_pins(fn):
    with open(os.path.join(GOLDEN, "best_first_hand.json")) as f:
        g = json.load(f)
    r = fn(g["marginals"], g["N"], **dict(HAND_COST, t_draft=1e9))  # huge draft cost: S never falls
    assert r["parents"] == g["expected_parents"] and r["depth"] == g["expected_depth"]
    assert np.allclose(r["rho"], g["expected_rho"], rtol=0, atol=1e-12)
    assert abs(sum(r["rho"]) - g["expected_surrogate"]) < 1e-12 and r["n"] == g["N"]

    r = fn(HAND_Q, 10, **HAND_COST)
    assert r["n"] == 4 and r["n_eval"] == 5
    assert np.allclose(r["speedup"], [0.3, 0.34, 0.355, 0.3596, 2.078 / 6], rtol=0, atol=1e-12)
    assert abs(r["a"] - 1) < 1e-12 and abs(r["c"]) < 1e-12

    # calibration: samples of T = 2.5 T_roof + 0.75 on a compute-bound roofline are recovered
    cost = dict(HAND_COST, bytes_per_node=0.0, flops_per_node=3.0, peak=2.0,
                cal_n=[1, 3, 8, 20], cal_t=[2.5 * 1.5 * n + 0.75 for n in (1, 3, 8, 20)])
    r = fn(HAND_Q, 3, **cost)
    assert abs(r["a"] - 2.5) < 1e-12 and abs(r["c"] - 0.75) < 1e-12
    # a single distinct roofline value: ratio of the means, no offset
    cost = dict(HAND_COST, bytes0=4.0, bytes_per_node=0.0, cal_n=[1, 2], cal_t=[6.0, 10.0])
    r = fn(HAND_Q, 3, **cost)
    assert abs(r["a"] - 2.0) < 1e-12 and r["c"] == 0.0

    # exact ties (uniform marginals, two positions): the frontier takes candidates in the
    # order they entered it. Root candidates 0, 1 (rho 0.5) enter first; popping node 0
    # pushes its children (0.25, 0.25), popping node 1 pushes its own after them.
    r = fn([[0.5, 0.5], [0.5, 0.5]], 6, **dict(HAND_COST, t_draft=1e9))
    assert r["parents"] == [-1, -1, 0, 0, 1, 1] and r["cand"] == [0, 1, 0, 1, 0, 1]

    # the stop uses the total step cost: with no drafting cost S falls at once
    r = fn(HAND_Q, 10, **dict(HAND_COST, t_draft=0.0))
    assert r["n"] == 1 and r["n_eval"] == 2


def test_pins_hold_for_the_oracle():
    run_pins(oracle.budget_plan)


def prefix_closed_best(q, n):
    """Brute force: the largest sum of path scores over every prefix-closed tree of n nodes."""
    K, C = len(q), len(q[0])
    nodes = []  # (path tuple, rho)
    for d in range(1, K + 1):
        for path in itertools.product(range(C), repeat=d):
            r = 1.0
            for k, c in enumerate(path):
                r *= q[k][c]
            nodes.append((path, r))
    best = -1.0
    for subset in itertools.combinations(range(len(nodes)), n):
        paths = {nodes[i][0] for i in subset}
        if all(len(p) == 1 or p[:-1] in paths for p in paths):
            best = max(best, sum(nodes[i][1] for i in subset))
    return best


@pytest.mark.parametrize("seed", range(6))
def test_best_first_surrogate_is_optimal(seed):
    rng = np.random.default_rng(seed)
    K, C = 3, 2
    q = -np.sort(-rng.dirichlet(np.ones(C), size=K), axis=1)
    r = oracle.budget_plan(q, 8, **dict(HAND_COST, t_draft=1e9))
    rho = r["rho"]
    assert all(rho[i] >= rho[i + 1] for i in range(len(rho) - 1))  # diminishing returns
    for n in range(1, 9):
        assert abs(sum(rho[:n]) - prefix_closed_best(q.tolist(), n)) < 1e-12


MUTANTS = {
    "stop reports the size that fell": ("n_star = n - 1", "n_star = n"),
    "children scored by the parent's position": ("r * float(q[dep, c2])", "r * float(q[dep - 1, c2])"),
    "ties to the later candidate": ("o < frontier[best][1]", "o > frontier[best][1]"),
    "calibration without offset": ("c = float(tm - a * xm)", "c = 0.0"),
    "step cost without drafting": ("cost = t_draft + (a * t_roof(n) + c)", "cost = a * t_roof(n) + c + 1.0"),
    "surrogate of the last node only": ("surrogate += r", "surrogate = r"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_fail_a_pin(name):
    src = textwrap.dedent(inspect.getsource(oracle.budget_plan))
    old, new = MUTANTS[name]
    assert old in src, name
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    with pytest.raises((AssertionError, ValueError, ZeroDivisionError)):
        run_pins(ns["budget_plan"])
