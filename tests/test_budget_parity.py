"""The library's host budget controller (spec_budget_plan) against the oracle (no GPU).

spec_budget_plan runs on the host, so its parity is checked here: the oracle's
pins run against the product, and random controller problems with GB300-like
roofline numbers compare tree, path scores, calibration, speedup curve and
chosen size.
"""

from __future__ import annotations

import ctypes
import time

import numpy as np
import pytest

import oracle
from tests.test_budget_pins import run_pins


@pytest.fixture(scope="module")
def ops():
    from speculative_decoding_verification_77_gb300 import build, ops as o

    build.build()
    o.load_library()
    return o


def test_product_passes_the_oracle_pins(ops):
    run_pins(ops.budget_plan)


def headline_costs(rng, n_cal=5):
    """Roofline of one verify step at B=4, L=32k, 32/8 heads, d=128 on this GPU's measured peaks
    (6.7 TB/s, 2.2 PFLOP/s), with calibration samples scattered around a corrected roofline."""
    B, Hq, Hkv, L, d = 4, 32, 8, 32768, 128
    cost = dict(t_draft=float(rng.uniform(20e-6, 200e-6)), l_ar=float(rng.uniform(5e-3, 20e-3)),
                bytes0=float(2 * B * Hkv * L * d * 2), bytes_per_node=float(B * (Hq * d * 6 + Hkv * d * 4)),
                flops_per_node=float(4 * B * Hq * L * d), bw=6.7e12, peak=2.2e15)
    n = np.sort(rng.choice(np.arange(1, 300), n_cal, replace=False)).astype(float)
    tr = np.maximum((cost["bytes0"] + cost["bytes_per_node"] * n) / cost["bw"], cost["flops_per_node"] * n / cost["peak"])
    cost["cal_n"] = n
    cost["cal_t"] = tr * rng.uniform(1.1, 1.6) + rng.uniform(0, 10e-6) + rng.normal(0, 1e-6, n_cal)
    return cost


@pytest.mark.parametrize("seed", range(30))
def test_random_problems_match_the_oracle(ops, seed):
    rng = np.random.default_rng(seed)
    K, C = int(rng.integers(1, 17)), int(rng.integers(1, 9))
    q = -np.sort(-rng.dirichlet(np.full(C, float(rng.uniform(0.1, 2.0))), size=K), axis=1)
    n_max = int(rng.integers(1, 300))
    cost = headline_costs(rng)
    want = oracle.budget_plan(q, n_max, **cost)
    got = ops.budget_plan(q, n_max, **cost)
    assert got["n"] == want["n"] and got["n_eval"] == want["n_eval"]
    assert got["parents"] == want["parents"] and got["depth"] == want["depth"] and got["cand"] == want["cand"]
    assert got["rho"] == want["rho"]  # the same products in the same order
    assert np.allclose(got["speedup"], want["speedup"], rtol=1e-12, atol=0)
    assert np.isclose(got["a"], want["a"], rtol=1e-12) and np.isclose(got["c"], want["c"], rtol=1e-9, atol=1e-15)


def test_rejects_bad_arguments(ops):
    from speculative_decoding_verification_77_gb300.ops import SpecError

    good = dict(t_draft=1.0, l_ar=1.0, bytes0=0.0, bytes_per_node=1.0, flops_per_node=0.0, bw=1.0, peak=1.0,
                cal_n=[1, 2], cal_t=[1.0, 2.0])
    for bad in (dict(bw=0.0), dict(peak=-1.0), dict(l_ar=float("nan")), dict(t_draft=-10.0)):
        with pytest.raises(SpecError):
            ops.budget_plan([[0.6, 0.4]], 4, **dict(good, **bad))
    with pytest.raises(SpecError):
        ops.budget_plan([[1.5, 0.4]], 4, **good)  # a probability above 1
    lib = ops.load_library()
    z = ctypes.c_void_p(16)
    assert lib.spec_budget_plan(None, 1, 1, 1, 1.0, 1.0, 0.0, 1.0, 0.0, 1.0, 1.0, z, z, 1, z, z, z, z, z, z, z, z) == 1


def test_host_time_at_the_largest_tree(ops):
    """The controller must cost little next to a verify step (about 0.1 ms): time 256 nodes of
    16 candidates."""
    rng = np.random.default_rng(0)
    q = -np.sort(-rng.dirichlet(np.full(16, 0.3), size=16), axis=1)
    cost = dict(headline_costs(rng), t_draft=1e3)  # S keeps growing: all 256 nodes are built
    ops.budget_plan(q, 256, **cost)
    t0 = time.perf_counter()
    for _ in range(20):
        r = ops.budget_plan(q, 256, **cost)
    per_call = (time.perf_counter() - t0) / 20
    assert r["n_eval"] == 256
    assert per_call < 5e-3, per_call
