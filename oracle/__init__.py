"""CPU oracle for verification attention (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product library never calls it, and it
shares no code with the CUDA path: the arithmetic lives in ``spec_oracle.c``
(plain C, fp64), and this module only marshals arguments into it.

Functions:
  select(...)      hybrid sink/window/top-m/fill selection (Dustin "Metodologia" section 1)
  attend(...)      monolithic fp64 softmax attention with an explicit mask over
                   [cache ; draft tree] (Dustin "Workflow di Verifica";
                   LongSpec section 2.C tree mask)
  lse_merge(...)   log-sum-exp merge of two normalised parts (LongSpec section 2.C)

Each returns (result..., status) where status 0 = ok, 5 = bad input seen.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from .build import build_oracle, oracle_lib_path

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = oracle_lib_path()
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(
                os.path.join(os.path.dirname(__file__), "spec_oracle.c")):
            build_oracle()
        _lib = load_library(path)
    return _lib


def set_library(lib):
    """Swap the loaded oracle library (used by the mutation tests); returns the old one."""
    global _lib
    old = _lib
    _lib = lib
    return old


def load_library(path: str):
    """Load an oracle shared library built from spec_oracle.c and declare its signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.oracle_select.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
    lib.oracle_select.restype = ctypes.c_int
    lib.oracle_attend.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                  P, P, P, P, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, P, ctypes.c_float,
                                  ctypes.c_int64, ctypes.c_int64, P, ctypes.c_int64, P, P]
    lib.oracle_attend.restype = ctypes.c_int
    lib.oracle_lse_merge.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int, P, P]
    lib.oracle_lse_merge.restype = ctypes.c_int
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _np(t, dtype):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        t = t.numpy()
    return np.ascontiguousarray(t, dtype=dtype)


def select(draft_score, target_score, *, sink: int, window: int, top_m: int, budget: int,
           ctx_lens=None):
    """Sequential selector. Scores fp32 [B, L]. Returns (idx int32 [B, budget], count [B], status)."""
    ds = _np(draft_score, np.float32)
    ts = _np(target_score, np.float32)
    B, L = ds.shape
    cl = _np(ctx_lens, np.int32)
    idx = np.empty((B, budget), dtype=np.int32)
    cnt = np.empty((B,), dtype=np.int32)
    st = _load().oracle_select(_ptr(ds), _ptr(ts), L, B, L, _ptr(cl), sink, window, top_m, budget,
                               _ptr(idx), _ptr(cnt))
    if st == 1:
        raise ValueError("oracle_select: invalid argument")
    return idx, cnt, st


def attend(q, k_cache, v_cache, k_draft, v_draft, parent, *, scale: float, ctx_lens=None,
           idx=None, rows=None, cache_range=None):
    """Monolithic fp64 attention for the given rows.

    q [B, N, Hq, d] bf16; k_cache/v_cache [B, Hkv, L, d] bf16 (contiguous);
    k_draft/v_draft [B, N, Hkv, d] bf16 or None (cache-only); parent int32 [B, N];
    idx int32 [B, budget] or None (dense). rows: flat row ids (b*N + i)*Hq + h,
    default all. cache_range=(t0, t1) keeps only cache tokens t0 <= t < t1.
    Returns (out float64 [n_rows, d], lse float64 [n_rows], status).
    """
    qn = _np(q, np.uint16)
    B, N, Hq, d = qn.shape
    kc = _np(k_cache, np.uint16)
    vc = _np(v_cache, np.uint16)
    _, Hkv, L, _ = kc.shape
    kd = _np(k_draft, np.uint16)
    vd = _np(v_draft, np.uint16)
    par = _np(parent, np.int32)
    ix = _np(idx, np.int32)
    budget = 0 if ix is None else ix.shape[1]
    cl = _np(ctx_lens, np.int32)
    if rows is None:
        rows = np.arange(B * N * Hq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    t0, t1 = (0, L) if cache_range is None else cache_range
    out = np.empty((rows.shape[0], d), dtype=np.float64)
    lse = np.empty((rows.shape[0],), dtype=np.float64)
    st = _load().oracle_attend(_ptr(qn), _ptr(kc), _ptr(vc), Hkv * L * d, L * d, d,
                               _ptr(kd), _ptr(vd), _ptr(par), _ptr(ix), budget,
                               B, N, Hq, Hkv, d, L, _ptr(cl), ctypes.c_float(scale),
                               t0, t1, _ptr(rows), rows.shape[0], _ptr(out), _ptr(lse))
    if st == 1:
        raise ValueError("oracle_attend: invalid argument")
    return out, lse, st


def lse_merge(o_a, lse_a, o_b, lse_b):
    """fp64 merge of two fp32 parts. o [rows, d], lse [rows]. Returns (out, lse)."""
    oa = _np(o_a, np.float32)
    ob = _np(o_b, np.float32)
    la = _np(lse_a, np.float32).reshape(-1)
    lb = _np(lse_b, np.float32).reshape(-1)
    d = oa.shape[-1]
    rows = la.shape[0]
    oa = oa.reshape(rows, d)
    ob = ob.reshape(rows, d)
    out = np.empty((rows, d), dtype=np.float64)
    lo = np.empty((rows,), dtype=np.float64)
    st = _load().oracle_lse_merge(_ptr(oa), _ptr(la), _ptr(ob), _ptr(lb), rows, d, _ptr(out), _ptr(lo))
    if st == 1:
        raise ValueError("oracle_lse_merge: invalid argument")
    return out, lo
