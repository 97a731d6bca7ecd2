"""The allocation-free entry point, spec_verify_attn_noalloc.

It is for callers that cannot allocate device memory when they call (engines
that reserved nearly all of HBM for the KV cache at start-up, or C hosts with
no allocator), so it keeps its scratch in a fixed array inside the library.
Here it is called through the C ABI on two calls in a row and compared with the
CPU oracle and with spec_verify_attn, whose workspace the caller provides: the
second call must not see anything the first one left in the shared scratch.
This file is collected last on purpose, and it also passes when run on its own.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_77_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL_O, RTOL_O, ATOL_L = 1e-2, 2e-2, 1e-3  # the tolerances the parity tests use


def _inputs(seed, B, N, Hq, Hkv, L, depth):
    w = W.Workload("noalloc", B=B, L=L, Hq=Hq, Hkv=Hkv, N=N, tree="random", depth_max=depth, seed=seed)
    x = W.make_inputs(w)
    dev = torch.device("cuda:0")
    return x, {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _noalloc(lib, g, scale, parent=None):
    q = g["q"]
    B, N, Hq, d = q.shape
    _, Hkv, L, _ = g["k_cache"].shape
    out = torch.full((B, N, Hq, d), float("nan"), dtype=torch.float32, device=q.device)
    lse = torch.full((B, N, Hq), float("nan"), dtype=torch.float32, device=q.device)
    status = torch.full((1,), -7, dtype=torch.int32, device=q.device)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    kc = g["k_cache"]
    par = g["parent"] if parent is None else parent
    code = lib.spec_verify_attn_noalloc(
        p(q), p(kc), p(g["v_cache"]), kc.stride(0), kc.stride(1), kc.stride(2), p(g["k_draft"]), p(g["v_draft"]),
        p(par), B, N, Hq, Hkv, d, L, None, ctypes.c_float(scale), p(out), p(lse), p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return code, out, lse, status


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    from speculative_decoding_verification_77_gb300 import ops

    lib = ops.load_library()
    # two different problems back to back: the second is smaller, so stale partials of the
    # first would show if the second read any slot it did not write
    cases = [(_inputs(901, B=2, N=24, Hq=16, Hkv=4, L=5000, depth=5)),
             (_inputs(902, B=1, N=7, Hq=8, Hkv=2, L=1300, depth=3))]
    for x, g in cases:
        code, out, lse, status = _noalloc(lib, g, x["scale"])
        assert code == 0, ops.STATUS_NAMES.get(code, code)
        ref_o, ref_l = ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"],
                                       g["parent"], scale=x["scale"])
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        assert (out - ref_o).abs().max().item() <= ATOL_O
        assert (lse - ref_l).abs().max().item() <= ATOL_L
        # and against the fp64 oracle, every row
        ro, rl, st = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                                   scale=x["scale"])
        assert st == 0
        o = out.cpu().numpy().reshape(ro.shape)
        err = np.abs(o - ro).max()
        assert err <= ATOL_O and err <= RTOL_O * np.abs(ro).max()
        assert np.abs(lse.cpu().numpy().reshape(-1) - rl).max() <= ATOL_L


def test_noalloc_reports_bad_input_and_rejects_oversize():
    from speculative_decoding_verification_77_gb300 import ops

    lib = ops.load_library()
    x, g = _inputs(903, B=1, N=6, Hq=4, Hkv=1, L=700, depth=3)
    bad = g["parent"].clone()
    bad[0, 4] = 5  # parent after the node
    code, out, lse, status = _noalloc(lib, g, x["scale"], parent=bad)
    torch.cuda.synchronize()
    assert code == 0 and int(status.item()) == 5
    code, out, lse, status = _noalloc(lib, g, x["scale"])
    torch.cuda.synchronize()
    assert code == 0 and int(status.item()) == 0
    # a problem whose partials exceed the built-in scratch is refused before any launch; the
    # cache is one real 128-element row read with zero strides, so even a launch would stay
    # inside it
    big_q = torch.zeros((8, 32, 64, 128), dtype=torch.bfloat16, device="cuda:0")
    row = torch.zeros((128,), dtype=torch.bfloat16, device="cuda:0")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    o = torch.empty((8, 32, 64, 128), dtype=torch.float32, device="cuda:0")
    l_ = torch.empty((8, 32, 64), dtype=torch.float32, device="cuda:0")
    code = lib.spec_verify_attn_noalloc(p(big_q), p(row), p(row), 0, 0, 0, None, None, None, 8, 32, 64, 8, 128,
                                        131072, None, ctypes.c_float(0.1), p(o), p(l_), None, None)
    torch.cuda.synchronize()
    assert code == 4  # SPEC_ERR_WORKSPACE
    # a split plan of 2^31 tiles or more is refused (32-bit tile numbering), also before any launch
    q1 = torch.zeros((64, 1, 1, 128), dtype=torch.bfloat16, device="cuda:0")
    o1 = torch.empty((64, 1, 1, 128), dtype=torch.float32, device="cuda:0")
    l1 = torch.empty((64, 1, 1), dtype=torch.float32, device="cuda:0")
    code = lib.spec_verify_attn_noalloc(p(q1), p(row), p(row), 0, 0, 0, None, None, None, 64, 1, 1, 1, 128,
                                        2**31 - 1, None, ctypes.c_float(0.1), p(o1), p(l1), None, None)
    torch.cuda.synchronize()
    assert code == 2  # SPEC_ERR_UNSUPPORTED
