"""BASTION's controller on a recorded GB300 sweep (no GPU).

The calibration samples are the verify-step times the bench measured on the tree-size sweep
(tests/golden/bastion_sweep_gb300.json); the controller's outputs are computed here by the
oracle and by the library's host implementation (spec_budget_plan), which must agree, and
checked against what the controller's definition fixes: (a, c) is the least-squares line of
the measured times on the roofline, and N* is the last size before the speedup first falls.
"""

from __future__ import annotations

import json
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_77_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bastion_sweep_gb300.json")


def problem():
    g = json.load(open(GOLDEN))
    m = g["marginals"]
    q = W.dirichlet_marginals(np.random.default_rng(m["seed"]), m["block"], m["cands"], m["alpha"])
    w = g["workload"]
    B, L, Hq, Hkv, d = w["B"], w["L"], w["Hq"], w["Hkv"], w["d"]
    ns = [float(n) for n in g["cal_n"]]
    ts = [float(t) for t in g["cal_t_us"]]
    l_ar = ts[ns.index(1.0)]
    cost = dict(t_draft=g["controller"]["t_draft_over_l_ar"] * l_ar, l_ar=l_ar,
                bytes0=float(2 * B * Hkv * L * d * 2),
                bytes_per_node=float(B * (Hq * d * 2 + 2 * Hkv * d * 2 + Hq * (d + 1) * 4)),
                flops_per_node=float(4 * B * Hq * L * d),
                bw=g["peaks"]["hbm_gbs"] * 1e3, peak=g["peaks"]["bf16_tflops_sustained"] * 1e6,  # per microsecond
                cal_n=ns, cal_t=ts)
    return g, q, g["controller"]["n_max"], cost


@pytest.fixture(scope="module")
def ops():
    from speculative_decoding_verification_77_gb300 import build, ops as o

    build.build()
    o.load_library()
    return o


def test_calibration_is_the_least_squares_line():
    g, q, n_max, cost = problem()
    want = oracle.budget_plan(q, n_max, **cost)
    n = np.asarray(cost["cal_n"])
    troof = np.maximum((cost["bytes0"] + cost["bytes_per_node"] * n) / cost["bw"], cost["flops_per_node"] * n / cost["peak"])
    a, c = np.polyfit(troof, np.asarray(cost["cal_t"]), 1)
    assert np.isclose(want["a"], a, rtol=1e-9) and np.isclose(want["c"], c, rtol=1e-9, atol=1e-9)
    # the measured times lie above the roofline: the fitted line's slope exceeds 1 here
    assert want["a"] > 1.0


def test_chosen_size_is_where_the_speedup_first_falls():
    g, q, n_max, cost = problem()
    want = oracle.budget_plan(q, n_max, **cost)
    s = np.asarray(want["speedup"])
    n = want["n"]
    assert 1 <= n <= want["n_eval"]
    assert np.all(np.diff(s[:n]) >= 0)  # no fall before N*
    if n < want["n_eval"]:
        assert s[n] < s[n - 1]  # the first fall comes right after N*


def test_library_matches_the_oracle_on_the_recorded_sweep(ops):
    g, q, n_max, cost = problem()
    want = oracle.budget_plan(q, n_max, **cost)
    got = ops.budget_plan(q, n_max, **cost)
    assert got["n"] == want["n"] and got["n_eval"] == want["n_eval"]
    assert got["parents"] == want["parents"] and got["cand"] == want["cand"] and got["rho"] == want["rho"]
    assert np.allclose(got["speedup"], want["speedup"], rtol=1e-12, atol=0)
    assert np.isclose(got["a"], want["a"], rtol=1e-12) and np.isclose(got["c"], want["c"], rtol=1e-9, atol=1e-12)
    # and the run that measured the sweep reported the same controller outputs
    bl = g["bench_line"]
    assert want["n"] == bl["n_chosen"]
    assert abs(want["a"] - bl["a"]) < 1e-6 and abs(want["c"] - bl["c_us"]) < 1e-4
