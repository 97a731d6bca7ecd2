"""Thin PyTorch binding of libspecverify.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
only checks tensor dtypes/devices, allocates outputs and workspaces with
torch, and passes raw pointers and the current CUDA stream through ctypes.
It has no fallback: if the library is missing or the device is not sm_103a,
the call raises.

Names mirror the C ABI (include/specverify.h):
  select_topk            -> spec_select_topk
  verify_attn            -> spec_verify_attn
  verify_attn_sparse     -> spec_verify_attn_sparse
  verify_attn_ex         -> spec_verify_attn_ex (paged cache, bf16 output)
  lse_merge              -> spec_lse_merge
  accept_commit          -> spec_accept_commit
  budget_plan            -> spec_budget_plan (host)
  split_plan             -> spec_split_plan (host)
  importance_scores      -> spec_importance_scores
  read_device_status     -> spec_read_device_status
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

SPEC_OK = 0
SPEC_ERR_CUDA = 3
SPEC_ERR_BAD_INPUT = 5
STATUS_NAMES = {0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_UNSUPPORTED", 3: "SPEC_ERR_CUDA",
                4: "SPEC_ERR_WORKSPACE", 5: "SPEC_ERR_BAD_INPUT", 6: "SPEC_ERR_TIMEOUT"}

# (name, restype, argtypes) of every exported entry point
P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "spec_status_string": (ctypes.c_char_p, [I]),
    "spec_select_workspace_size": (SZ, [I, I, I]),
    "spec_select_topk": (I, [P, P, I64, I, I, P, I, I, I, I, P, P, P, SZ, P]),
    "spec_verify_workspace_size": (SZ, [I, I, I, I, I, I]),
    "spec_split_plan": (I, [I, I, I, I, I, I, I, P, I, P]),
    "spec_verify_attn": (I, [P, P, P, I64, I64, I64, P, P, P, I, I, I, I, I, I, P, F, P, P, P, SZ, P]),
    "spec_verify_attn_sparse": (I, [P, P, P, I64, I64, I64, P, P, P, I, I, I, I, I, I, P, F, P, I,
                                    P, P, P, SZ, P]),
    "spec_lse_merge": (I, [P, P, P, P, P, P, I64, I, P]),
    "spec_verify_attn_ex": (I, [P, P, P, I64, I64, I64, P, P, P, I, I, I, I, I, I, P, F, P, I, P, P, P, P, SZ, P]),
    "spec_verify_attn_noalloc": (I, [P, P, P, I64, I64, I64, P, P, P, I, I, I, I, I, I, P, F, P, P, P, P]),
    "spec_read_device_status": (I, [P, P]),
    "spec_accept_commit": (I, [P, P, P, I, I, P, P, P, P, P, I64, I64, I64, P, P, I, I, I, P, P, P]),
    "spec_importance_scores": (I, [P, P, I64, I64, I64, P, P, I, I, I, I, I, I, I, P, F, P, I64, P, P]),
    "spec_budget_plan": (I, [P, I, I, I, ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                             ctypes.c_double, ctypes.c_double, ctypes.c_double, P, P, I, P, P, P, P, P, P, P, P]),
    "spec_profile_events": (None, [P, P]),
    "spec_kernel_launches": (ctypes.c_uint64, []),
    "spec_last_cuda_error": (ctypes.c_char_p, []),
}

_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str = ""):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}" + (f" ({detail})" if detail else ""))
        self.code = code


def load_library(path: str = LIB_PATH):
    """Load the C-ABI library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libspecverify.so not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(fn: str, code: int):
    if code != SPEC_OK:
        detail = _lib.spec_last_cuda_error().decode() if code == SPEC_ERR_CUDA and _lib is not None else ""
        raise SpecError(fn, code, detail)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t, dtype, name, dims=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {tuple(t.shape)}")


_workspaces: dict = {}


def workspace(nbytes: int, device: torch.device, key: str = "default") -> torch.Tensor:
    """A cached uint8 device buffer of at least nbytes (one per device, stream and key)."""
    stream = torch.cuda.current_stream(device).cuda_stream
    k = (device.index, stream, key)
    ws = _workspaces.get(k)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[k] = ws
    return ws


def select_topk(draft_score: torch.Tensor, target_score: torch.Tensor, *, sink: int, window: int,
                top_m: int, budget: int, ctx_lens: torch.Tensor | None = None,
                idx: torch.Tensor | None = None, count: torch.Tensor | None = None,
                ws: torch.Tensor | None = None):
    """Hybrid sink/window/top-m/fill selection. Scores fp32 [B, L] (row stride = stride(0))."""
    lib = load_library()
    _need(draft_score, torch.float32, "draft_score", 2)
    _need(target_score, torch.float32, "target_score", 2)
    _need(ctx_lens, torch.int32, "ctx_lens", 1)
    if draft_score.stride(1) != 1 or target_score.stride(1) != 1 or \
            draft_score.stride(0) != target_score.stride(0):
        raise ValueError("score rows must be contiguous with a common row stride")
    B, L = draft_score.shape
    dev = draft_score.device
    if idx is None:
        idx = torch.empty((B, budget), dtype=torch.int32, device=dev)
    if count is None:
        count = torch.empty((B,), dtype=torch.int32, device=dev)
    nbytes = lib.spec_select_workspace_size(B, L, budget)
    if ws is None:
        ws = workspace(nbytes, dev, "select")
    _check("spec_select_topk", lib.spec_select_topk(
        _ptr(draft_score), _ptr(target_score), draft_score.stride(0), B, L, _ptr(ctx_lens), sink, window,
        top_m, budget, _ptr(idx), _ptr(count), _ptr(ws), ws.numel(), _stream(draft_score)))
    return idx, count


def _verify(q, k_cache, v_cache, k_draft, v_draft, parent, scale, ctx_lens, idx, out, lse, ws):
    lib = load_library()
    _need(q, torch.bfloat16, "q", 4)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(k_draft, torch.bfloat16, "k_draft", 4)
    _need(v_draft, torch.bfloat16, "v_draft", 4)
    _need(parent, torch.int32, "parent", 2)
    _need(ctx_lens, torch.int32, "ctx_lens", 1)
    _need(idx, torch.int32, "idx", 2)
    B, N, Hq, d = q.shape
    _, Hkv, L, _ = k_cache.shape
    if not q.is_contiguous():
        raise ValueError("q must be contiguous [B, N, Hq, d]")
    if k_cache.stride() != v_cache.stride() or k_cache.shape != v_cache.shape or k_cache.stride(3) != 1:
        raise ValueError("k_cache and v_cache must share shape and strides, with d contiguous")
    for t, nm in ((k_draft, "k_draft"), (v_draft, "v_draft")):
        if t is not None and (not t.is_contiguous() or tuple(t.shape) != (B, N, Hkv, d)):
            raise ValueError(f"{nm} must be contiguous [B, N, Hkv, d]")
    if parent is not None and (not parent.is_contiguous() or tuple(parent.shape) != (B, N)):
        raise ValueError("parent must be contiguous int32 [B, N]")
    if idx is not None and (not idx.is_contiguous() or idx.shape[0] != B):
        raise ValueError("idx must be contiguous int32 [B, budget]")
    if scale is None:
        scale = d ** -0.5
    dev = q.device
    if out is None:
        out = torch.empty((B, N, Hq, d), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    L_eff = idx.shape[1] if idx is not None else L
    nbytes = lib.spec_verify_workspace_size(B, N, Hq, Hkv, d, L_eff)
    if ws is None:
        ws = workspace(nbytes, dev, "verify")
    sb, sh, st = k_cache.stride(0), k_cache.stride(1), k_cache.stride(2)
    common = (_ptr(q), _ptr(k_cache), _ptr(v_cache), sb, sh, st, _ptr(k_draft), _ptr(v_draft),
              _ptr(parent), B, N, Hq, Hkv, d, L, _ptr(ctx_lens), ctypes.c_float(scale))
    if idx is None:
        code = lib.spec_verify_attn(*common, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(q))
        _check("spec_verify_attn", code)
    else:
        code = lib.spec_verify_attn_sparse(*common, _ptr(idx), idx.shape[1], _ptr(out), _ptr(lse),
                                           _ptr(ws), ws.numel(), _stream(q))
        _check("spec_verify_attn_sparse", code)
    return out, lse


def verify_attn(q, k_cache, v_cache, k_draft=None, v_draft=None, parent=None, *, scale=None,
                ctx_lens=None, out=None, lse=None, ws=None):
    """Dense verification attention: full cache + tree-masked draft block, LSE-merged.

    q [B,N,Hq,d] bf16; k_cache/v_cache [B,Hkv,L,d] bf16 (any strides with d contiguous);
    k_draft/v_draft [B,N,Hkv,d] bf16 and parent int32 [B,N], or all None (cache-only part).
    Returns (out fp32 [B,N,Hq,d], lse fp32 [B,N,Hq]).
    """
    return _verify(q, k_cache, v_cache, k_draft, v_draft, parent, scale, ctx_lens, None, out, lse, ws)


def verify_attn_sparse(q, k_cache, v_cache, k_draft, v_draft, parent, idx, *, scale=None,
                       ctx_lens=None, out=None, lse=None, ws=None):
    """Sparse verification attention over the cache rows idx[b] (int32 [B, budget])."""
    return _verify(q, k_cache, v_cache, k_draft, v_draft, parent, scale, ctx_lens, idx, out, lse, ws)


class _VerifyExt(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("table_ld", ctypes.c_int64), ("block_size", ctypes.c_int),
                ("num_blocks", ctypes.c_int64), ("out_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


def verify_attn_ex(q, k_cache, v_cache, k_draft=None, v_draft=None, parent=None, *, L: int | None = None, idx=None,
                   block_table=None, out_dtype=torch.float32, scale=None, ctx_lens=None, out=None, lse=None, ws=None,
                   k_scale=None, v_scale=None):
    """Verification attention with the extensions of spec_verify_attn_ex: a paged cache, an fp8
    cache and/or a bf16 output (dense, or sparse with idx [B, budget]).

    fp8 cache: k_cache/v_cache torch.float8_e4m3fn (or uint8 codes) with k_scale, v_scale fp32
    [B, Hkv] (the value of a code is its E4M3 number times the scale of its sequence and head).

    Contiguous: k_cache/v_cache [B, Hkv, L, d]. Paged (block_table int32 [B, max_blocks]):
    k_cache/v_cache are the pools, [num_blocks, Hkv, block_size, d] bf16 views (any strides, d
    contiguous; a token-major pool [num_blocks, block_size, Hkv, d] is passed permuted); token t of
    sequence b is row t % block_size of block block_table[b, t // block_size], and L (the longest
    context) must be given. out_dtype torch.float32 or torch.bfloat16.
    Returns (out [B,N,Hq,d] of out_dtype, lse fp32 [B,N,Hq]).
    """
    lib = load_library()
    fp8 = k_cache.dtype in (torch.float8_e4m3fn, torch.uint8)
    for t, nm in ((q, "q"), (k_draft, "k_draft"), (v_draft, "v_draft")):
        _need(t, torch.bfloat16, nm, 4)
    for t, nm in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, k_cache.dtype if fp8 else torch.bfloat16, nm, 4)
    if fp8:
        if k_scale is None or v_scale is None:
            raise ValueError("an fp8 cache needs k_scale and v_scale [B, Hkv]")
        _need(k_scale, torch.float32, "k_scale", 2)
        _need(v_scale, torch.float32, "v_scale", 2)
        if not (k_scale.is_contiguous() and v_scale.is_contiguous()):
            raise ValueError("k_scale and v_scale must be contiguous [B, Hkv]")
    _need(block_table, torch.int32, "block_table", 2)
    _need(parent, torch.int32, "parent", 2)
    _need(ctx_lens, torch.int32, "ctx_lens", 1)
    _need(idx, torch.int32, "idx", 2)
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    B, N, Hq, d = q.shape
    if block_table is None:
        _, Hkv, Lc, _ = k_cache.shape
        L = Lc if L is None else L
        nblk = bs = 0
    else:
        nblk, Hkv, bs, _ = k_cache.shape
        if L is None:
            raise ValueError("a paged call needs L, the longest context")
        if block_table.stride(1) != 1 or block_table.shape[0] != B:
            raise ValueError("block_table must be [B, max_blocks] with unit column stride")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous [B, N, Hq, d]")
    if k_cache.stride() != v_cache.stride() or k_cache.shape != v_cache.shape or k_cache.stride(3) != 1:
        raise ValueError("k_cache and v_cache must share shape and strides, with d contiguous")
    if idx is not None and (not idx.is_contiguous() or idx.shape[0] != B):
        raise ValueError("idx must be contiguous int32 [B, budget]")
    if scale is None:
        scale = d ** -0.5
    dev = q.device
    if out is None:
        out = torch.empty((B, N, Hq, d), dtype=out_dtype, device=dev)
    _need(out, out_dtype, "out", 4)
    if lse is None:
        lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    L_eff = idx.shape[1] if idx is not None else L
    nbytes = lib.spec_verify_workspace_size(B, N, Hq, Hkv, d, L_eff)
    if ws is None:
        ws = workspace(nbytes, dev, "verify")
    ext = _VerifyExt(None if block_table is None else block_table.data_ptr(),
                     0 if block_table is None else block_table.stride(0), bs, nblk,
                     1 if out_dtype == torch.bfloat16 else 0, 1 if fp8 else 0,
                     k_scale.data_ptr() if fp8 else None, v_scale.data_ptr() if fp8 else None)
    code = lib.spec_verify_attn_ex(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.stride(0), k_cache.stride(1), k_cache.stride(2), _ptr(k_draft),
        _ptr(v_draft), _ptr(parent), B, N, Hq, Hkv, d, L, _ptr(ctx_lens), ctypes.c_float(scale), _ptr(idx),
        0 if idx is None else idx.shape[1], ctypes.byref(ext), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(q))
    _check("spec_verify_attn_ex", code)
    return out, lse


def verify_attn_paged(q, k_pool, v_pool, block_table, k_draft=None, v_draft=None, parent=None, *, L: int, **kw):
    """verify_attn_ex over a paged cache (see there)."""
    return verify_attn_ex(q, k_pool, v_pool, k_draft, v_draft, parent, L=L, block_table=block_table, **kw)


def lse_merge(o_a, lse_a, o_b, lse_b, out=None, lse_out=None):
    """Merge two normalised parts by log-sum-exp. o [..., d] fp32, lse [...] fp32."""
    lib = load_library()
    for t, nm in ((o_a, "o_a"), (lse_a, "lse_a"), (o_b, "o_b"), (lse_b, "lse_b")):
        _need(t, torch.float32, nm)
        if not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    d = o_a.shape[-1]
    rows = lse_a.numel()
    if o_a.numel() != rows * d or o_b.numel() != rows * d or lse_b.numel() != rows:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    _check("spec_lse_merge", lib.spec_lse_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(out),
                                                _ptr(lse_out), rows, d, _stream(o_a)))
    return out, lse_out


def accept_commit(draft_token, parent, target_next, k_cache=None, v_cache=None, k_draft=None, v_draft=None,
                  ctx_lens=None):
    """Greedy acceptance of the draft tree, then (with the caches given) the commit of the
    accepted draft K/V rows at [ctx_lens, ctx_lens + accepted), in place.

    draft_token, parent int32 [B, N]; target_next int32 [B, N + 1]; caches bf16 [B, Hkv, L, d]
    (d contiguous), drafts bf16 [B, N, Hkv, d] contiguous, ctx_lens int32 [B] (updated).
    Returns (path int32 [B, N], length int32 [B], bonus int32 [B], status int32 [1]) on the
    device; status holds SPEC_ERR_BAD_INPUT if a parent, a context length or the cache's
    room was out of range.
    """
    lib = load_library()
    _need(draft_token, torch.int32, "draft_token", 2)
    _need(parent, torch.int32, "parent", 2)
    _need(target_next, torch.int32, "target_next", 2)
    for t, nm in ((draft_token, "draft_token"), (parent, "parent"), (target_next, "target_next")):
        if not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    B, N = draft_token.shape
    if tuple(parent.shape) != (B, N) or tuple(target_next.shape) != (B, N + 1):
        raise ValueError("shape mismatch")
    dev = draft_token.device
    path = torch.empty((B, N), dtype=torch.int32, device=dev)
    length = torch.empty((B,), dtype=torch.int32, device=dev)
    bonus = torch.empty((B,), dtype=torch.int32, device=dev)
    status = torch.empty((1,), dtype=torch.int32, device=dev)
    commit = k_cache is not None
    Hkv = d = L = 0
    sb = sh = st = 0
    if commit:
        _need(k_cache, torch.bfloat16, "k_cache", 4)
        _need(v_cache, torch.bfloat16, "v_cache", 4)
        _need(k_draft, torch.bfloat16, "k_draft", 4)
        _need(v_draft, torch.bfloat16, "v_draft", 4)
        _need(ctx_lens, torch.int32, "ctx_lens", 1)
        if k_cache.stride() != v_cache.stride() or k_cache.shape != v_cache.shape or k_cache.stride(3) != 1:
            raise ValueError("k_cache and v_cache must share shape and strides, with d contiguous")
        if not (k_draft.is_contiguous() and v_draft.is_contiguous() and ctx_lens.is_contiguous()):
            raise ValueError("k_draft, v_draft and ctx_lens must be contiguous")
        _, Hkv, L, d = k_cache.shape
        sb, sh, st = k_cache.stride(0), k_cache.stride(1), k_cache.stride(2)
    _check("spec_accept_commit", lib.spec_accept_commit(
        _ptr(draft_token), _ptr(parent), _ptr(target_next), B, N, _ptr(path), _ptr(length), _ptr(bonus),
        _ptr(k_cache), _ptr(v_cache), sb, sh, st, _ptr(k_draft), _ptr(v_draft), Hkv, d, L, _ptr(ctx_lens),
        _ptr(status), _stream(draft_token)))
    return path, length, bonus, status


def importance_scores(q, k_cache, lse, heads, *, scale=None, ctx_lens=None, out=None, status=None):
    """Target-historical importance of every cache token on the given query heads.

    q [B,N,Hq,d] bf16, k_cache [B,Hkv,L,d] bf16 (d contiguous), lse fp32 [B,N,Hq] (from verify_attn),
    heads int32 [nh] on the device. Returns (score fp32 [B, L], status int32 [1]).
    """
    import math

    lib = load_library()
    _need(q, torch.bfloat16, "q", 4)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(lse, torch.float32, "lse", 3)
    _need(heads, torch.int32, "heads", 1)
    _need(ctx_lens, torch.int32, "ctx_lens", 1)
    if not (q.is_contiguous() and lse.is_contiguous() and heads.is_contiguous()) or k_cache.stride(3) != 1:
        raise ValueError("q, lse and heads must be contiguous and k_cache's d contiguous")
    B, N, Hq, d = q.shape
    _, Hkv, L, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, L), dtype=torch.float32, device=q.device)
    if status is None:
        status = torch.empty((1,), dtype=torch.int32, device=q.device)
    _need(status, torch.int32, "status", 1)
    _check("spec_importance_scores", lib.spec_importance_scores(
        _ptr(q), _ptr(k_cache), k_cache.stride(0), k_cache.stride(1), k_cache.stride(2), _ptr(lse), _ptr(heads),
        heads.numel(), B, N, Hq, Hkv, d, L, _ptr(ctx_lens), float(scale), _ptr(out), out.stride(0), _ptr(status),
        _stream(q)))
    return out, status


def split_plan(B: int, N: int, Hq: int, Hkv: int, L: int, *, sms: int, sparse: bool = False) -> dict:
    """The tensor-core cache kernel's split plan for a call of this shape on `sms` SMs (see
    spec_split_plan; host only). L is the budget for a sparse call. Returns dict(ctas, starts,
    units, tiles_per_unit, row_groups, BM, split_tiles, pipes, slots, uniform)."""
    import numpy as np

    lib = load_library()
    starts = np.zeros(513, np.int32)
    info = np.zeros(8, np.int32)
    p = lambda a: ctypes.c_void_p(a.ctypes.data)
    r = lib.spec_split_plan(B, N, Hq, Hkv, L, sms, 1 if sparse else 0, p(starts), starts.shape[0], p(info))
    if r < 0:
        raise SpecError("spec_split_plan", -r)
    keys = ("units", "tiles_per_unit", "row_groups", "BM", "split_tiles", "pipes", "slots", "uniform")
    return dict(ctas=int(r), starts=starts[:r + 1].tolist(), **{k: int(v) for k, v in zip(keys, info)})


def budget_plan(marginals, n_max: int, *, t_draft: float, l_ar: float, bytes0: float, bytes_per_node: float,
                flops_per_node: float, bw: float, peak: float, cal_n, cal_t) -> dict:
    """BASTION's budget controller on the host (see spec_budget_plan). marginals [K, C] array-like.
    Returns dict(n, n_eval, parents, depth, cand, rho, speedup, a, c)."""
    import numpy as np

    lib = load_library()
    q = np.ascontiguousarray(np.asarray(marginals, dtype=np.float64))
    if q.ndim != 2:
        raise ValueError("marginals must be [K, C]")
    cn = np.ascontiguousarray(np.asarray(cal_n, dtype=np.float64).reshape(-1))
    ct = np.ascontiguousarray(np.asarray(cal_t, dtype=np.float64).reshape(-1))
    if cn.shape != ct.shape:
        raise ValueError("cal_n and cal_t differ in length")
    par = np.zeros(n_max, np.int32)
    dep = np.zeros(n_max, np.int32)
    cnd = np.zeros(n_max, np.int32)
    rho = np.zeros(n_max, np.float64)
    spd = np.zeros(n_max, np.float64)
    cal = np.zeros(2, np.float64)
    nc = np.zeros(1, np.int32)
    ne = np.zeros(1, np.int32)
    p = lambda a: ctypes.c_void_p(a.ctypes.data)
    _check("spec_budget_plan", lib.spec_budget_plan(
        p(q), q.shape[0], q.shape[1], n_max, t_draft, l_ar, bytes0, bytes_per_node, flops_per_node, bw, peak,
        p(cn), p(ct), cn.shape[0], p(par), p(dep), p(cnd), p(rho), p(spd), p(cal), p(nc), p(ne)))
    k = int(ne[0])
    return dict(n=int(nc[0]), n_eval=k, parents=par[:k].tolist(), depth=dep[:k].tolist(), cand=cnd[:k].tolist(),
                rho=rho[:k].tolist(), speedup=spd[:k].tolist(), a=float(cal[0]), c=float(cal[1]))


def read_device_status(ws: torch.Tensor) -> int:
    """Synchronise the current stream and read the status word the last call left in ws."""
    return load_library().spec_read_device_status(_ptr(ws), _stream(ws))


def kernel_launches() -> int:
    return load_library().spec_kernel_launches()


def profile_events(start: torch.cuda.Event | None, stop: torch.cuda.Event | None):
    """Record start/stop around the cache-attention kernel of following verify calls (None: off)."""
    lib = load_library()
    if start is None or stop is None:
        lib.spec_profile_events(None, None)
    else:
        lib.spec_profile_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event))
