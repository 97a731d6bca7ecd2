"""bench.py's roofline arithmetic on the CPU (no GPU): algorithmic bytes and flops per workload,
the bound a kernel is held to, and the fractions it reports."""

from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verification_77_gb300 import workloads as W  # noqa: E402

PEAKS = {"hbm_gbs": 6683.2, "bf16_tflops": 1940.8, "bf16_tflops_sustained": 1728.1}


def test_algorithmic_bytes_and_flops():
    head = W.workload(2)  # B=4, L=32k, 8 KV heads, d=128: K and V in bf16
    assert head.kv_bytes() == 2 * 4 * 8 * 32768 * 128 * 2 == 536_870_912
    assert head.flops() == 4 * 4 * 32 * 64 * 32768 * 128  # QK^T and PV, 2 flops a multiply-add
    sparse = W.workload(3)  # only the 2,048 selected tokens of each sequence
    assert sparse.kv_bytes() == 2 * 16 * 8 * 2048 * 128 * 2 == 134_217_728


@pytest.mark.parametrize("n,bound", [(1, "hbm"), (64, "hbm"), (256, "tensor")])
def test_bound_follows_the_ridge(n, bound):
    """The sweep's intensity grows with N: 4N flops per K/V byte (G*N query rows, 2 flops per
    multiply-add, QK and PV, over 2 bf16 bytes of K and V); the ridge of the measured peaks is
    1,728 TFLOP/s / 6.68 TB/s = 259 flop/B, so N = 64 (256 flop/B) stays HBM-bound and N = 256
    (1,024) is tensor-bound."""
    w = W.workload(5, n)
    assert w.flops() / w.kv_bytes() == 4 * n
    r = bench.roofline_entry(w, 0.1, PEAKS, "measured")
    assert r["bound"] == bound


def test_fractions_at_a_known_time():
    w = W.workload(2)
    ms = 0.11115  # a measured kernel time of the headline
    r = bench.roofline_entry(w, ms, PEAKS, "measured")
    gbs = w.kv_bytes() / (ms * 1e-3) / 1e9
    assert r["achieved_gbs"] == round(gbs, 1) and r["frac_hbm"] == round(gbs / 6683.2, 4)
    assert r["frac_bound"] == r["frac_hbm"] or abs(r["frac_bound"] - r["frac_hbm"]) < 1e-4
    assert 0.72 < r["frac_hbm"] < 0.73 and r["kernel_us"] == 111.15
    n256 = bench.roofline_entry(W.workload(5, 256), 0.3869, PEAKS, "measured")
    assert n256["bound"] == "tensor" and 0.82 < n256["frac_bound"] < 0.83
    assert n256["frac_bound"] == n256["frac_tensor_sustained"] or abs(n256["frac_bound"] - n256["frac_tensor_sustained"]) < 1e-4


def test_traffic_entries_name_known_workloads():
    names = {W.workload(c).name for c in (1, 2, 3, 4)} | {W.workload(5, n).name for n in bench.SWEEP_N}
    hashes = {h for h, _ in bench.NCU_TRAFFIC}
    assert len(hashes) == 1  # one capture set, of one kernel source
    for (_, name), traffic in bench.NCU_TRAFFIC.items():
        assert name in names
        w = next(W.workload(c, n) for c, n in [(1, None), (2, None), (3, None), (4, None)] +
                 [(5, n) for n in bench.SWEEP_N] if W.workload(c, n).name == name)
        assert 1.0 <= traffic / w.kv_bytes() < 1.2  # read about once, plus the partials
