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
  attend_paged(...) attend() over a paged cache: the same cache in fixed-size blocks
                   of a pool, found through a per-sequence block table (a layout the
                   pages do not use)
  lse_merge(...)   log-sum-exp merge of two normalised parts (LongSpec section 2.C)
  importance_scores(...) target-historical importance of every cache token: the
                   final attention probabilities of the draft queries on the
                   selected heads, summed (Dustin "Metodologia" sections 1-2).
                   numpy, fp64.
  budget_plan(...) BASTION's hardware-aware budget controller: best-first tree
                   growth from the drafter's marginals, the acceptance surrogate,
                   the calibrated roofline latency and the speedup-based stop
                   (BASTION "Metodologia" sections 1-3). Plain Python, fp64.
  accept_commit(...) greedy acceptance of the draft tree and commit of the accepted
                   draft K/V rows into the cache (Dustin "Workflow di Verifica",
                   step 5; BASTION "Risultati Sperimentali": greedy decoding).
                   Integer bookkeeping and row copies: written here in plain
                   Python loops, for the small cases the tests use.

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
    lib.oracle_attend_paged.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        P, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                        P, P, P, P, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, P, ctypes.c_float,
                                        P, ctypes.c_int64, P, P]
    lib.oracle_attend_paged.restype = ctypes.c_int
    lib.oracle_attend_fp8.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P,
                                      P, P, P, P, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, P, ctypes.c_float,
                                      P, ctypes.c_int64, P, P]
    lib.oracle_attend_fp8.restype = ctypes.c_int
    lib.oracle_e4m3_value.argtypes = [ctypes.c_int]
    lib.oracle_e4m3_value.restype = ctypes.c_double
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
        if t.dtype == torch.float8_e4m3fn:  # the 8-bit codes themselves
            return t.view(torch.uint8).numpy()
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


def attend_paged(q, k_pool, v_pool, k_draft, v_draft, parent, block_table, *, L: int, scale: float,
                 ctx_lens=None, idx=None, rows=None, num_blocks=None):
    """attend() over a paged cache (a layout the pages do not use): the cache of
    sequence b is stored in fixed-size blocks of a pool, token t being row
    t % block_size of pool block block_table[b, t // block_size]. A block entry
    outside [0, num_blocks) hides its tokens and is reported (status 5).

    k_pool/v_pool [num_blocks, Hkv, block_size, d] bf16 (copied contiguous);
    block_table int32 [B, max_blocks] with max_blocks >= ceil(L / block_size); num_blocks
    (default: all the pool's blocks) is how many blocks entries may name.
    Returns (out float64 [n_rows, d], lse float64 [n_rows], status).
    """
    qn = _np(q, np.uint16)
    B, N, Hq, d = qn.shape
    kp = _np(k_pool, np.uint16)
    vp = _np(v_pool, np.uint16)
    nblk, Hkv, bs, _ = kp.shape
    if num_blocks is not None:
        assert 0 <= num_blocks <= nblk
        nblk = num_blocks
    kd = _np(k_draft, np.uint16)
    vd = _np(v_draft, np.uint16)
    par = _np(parent, np.int32)
    tab = _np(block_table, np.int32)
    ix = _np(idx, np.int32)
    budget = 0 if ix is None else ix.shape[1]
    cl = _np(ctx_lens, np.int32)
    if rows is None:
        rows = np.arange(B * N * Hq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.shape[0], d), dtype=np.float64)
    lse = np.empty((rows.shape[0],), dtype=np.float64)
    st = _load().oracle_attend_paged(_ptr(qn), _ptr(kp), _ptr(vp), Hkv * bs * d, bs * d, d, _ptr(tab),
                                     tab.shape[1], bs, nblk, _ptr(kd), _ptr(vd), _ptr(par), _ptr(ix), budget,
                                     B, N, Hq, Hkv, d, L, _ptr(cl), ctypes.c_float(scale), _ptr(rows),
                                     rows.shape[0], _ptr(out), _ptr(lse))
    if st == 1:
        raise ValueError("oracle_attend_paged: invalid argument")
    return out, lse, st


def attend_fp8(q, k_codes, v_codes, k_scale, v_scale, k_draft, v_draft, parent, *, scale: float,
               ctx_lens=None, idx=None, rows=None):
    """attend() over a cache stored as 8-bit floats (a layout the pages do not use): K and V
    [B, Hkv, L, d] E4M3 codes (uint8, or torch float8_e4m3fn), the value of a code being the
    OCP E4M3 number it encodes times k_scale[b, h] (v_scale[b, h]), fp32 [B, Hkv]. Queries and
    the draft block are bf16 as in attend(). Returns (out float64 [n_rows, d], lse, status)."""
    qn = _np(q, np.uint16)
    B, N, Hq, d = qn.shape
    kc = _np(k_codes, np.uint8)
    vc = _np(v_codes, np.uint8)
    _, Hkv, L, _ = kc.shape
    ks = _np(k_scale, np.float32)
    vs = _np(v_scale, np.float32)
    assert ks.shape == (B, Hkv) and vs.shape == (B, Hkv)
    kd = _np(k_draft, np.uint16)
    vd = _np(v_draft, np.uint16)
    par = _np(parent, np.int32)
    ix = _np(idx, np.int32)
    budget = 0 if ix is None else ix.shape[1]
    cl = _np(ctx_lens, np.int32)
    if rows is None:
        rows = np.arange(B * N * Hq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.shape[0], d), dtype=np.float64)
    lse = np.empty((rows.shape[0],), dtype=np.float64)
    st = _load().oracle_attend_fp8(_ptr(qn), _ptr(kc), _ptr(vc), Hkv * L * d, L * d, d, _ptr(ks), _ptr(vs),
                                   _ptr(kd), _ptr(vd), _ptr(par), _ptr(ix), budget, B, N, Hq, Hkv, d, L,
                                   _ptr(cl), ctypes.c_float(scale), _ptr(rows), rows.shape[0], _ptr(out),
                                   _ptr(lse))
    if st == 1:
        raise ValueError("oracle_attend_fp8: invalid argument")
    return out, lse, st


def e4m3_value(code: int) -> float:
    """The number an E4M3 code (0..255) stands for (NaN for the two NaN codes)."""
    return float(_load().oracle_e4m3_value(int(code)))


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


def accept_commit(draft_token, parent, target_next, k_cache=None, v_cache=None, k_draft=None, v_draft=None,
                  ctx_lens=None):
    """Greedy (temperature 0) acceptance of a draft tree, then the cache commit.

    The pages say that the target verifies the draft tokens and that the accepted
    ones are appended to the cache while the rejected ones are dropped (Dustin
    "Workflow di Verifica", steps 4-5), under greedy decoding (BASTION
    "Risultati Sperimentali"). They do not spell the acceptance rule out; the
    plainest reading, taken here:

    * target_next[b, 0] is the target's greedy token after the last committed
      token, target_next[b, 1 + i] its greedy token after draft node i;
    * starting at the root (cur = -1), the next accepted node is the lowest-index
      child c of cur (parent[c] == cur, c > cur) with draft_token[c] ==
      target_next[b, cur + 1]; the walk stops when no child matches;
    * the bonus token is target_next[b, last accepted node + 1];
    * the accepted nodes' draft K/V rows (all KV heads) are copied, in path order,
      to cache positions ctx_lens[b], ctx_lens[b] + 1, ..., and ctx_lens[b]
      grows by the number copied.

    A parent entry outside [-1, i) never makes node i a child (it is reported);
    a context length outside [0, L] commits nothing, and rows past L are not
    copied (both reported).

    draft_token, parent: int [B, N]; target_next: int [B, N + 1]; caches
    [B, Hkv, L, d] and drafts [B, N, Hkv, d] (any dtype, copied as they are);
    ctx_lens int [B]. Returns (path [B, N] with -1 after the accepted nodes,
    length [B], bonus [B], k_cache, v_cache, ctx_lens, status) with new arrays for
    the caches and lengths (None when not given) and status 5 if anything was
    reported, else 0.
    """
    tok = np.asarray(draft_token, dtype=np.int64)
    par = np.asarray(parent, dtype=np.int64)
    tn = np.asarray(target_next, dtype=np.int64)
    B, N = tok.shape
    if par.shape != (B, N) or tn.shape != (B, N + 1):
        raise ValueError("accept_commit: shape mismatch")
    path = np.full((B, N), -1, dtype=np.int64)
    length = np.zeros(B, dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    status = 0
    for b in range(B):
        for i in range(N):
            if not (-1 <= par[b, i] < i):
                status = 5
        cur, n = -1, 0
        while True:
            want = tn[b, cur + 1]
            nxt = -1
            for c in range(cur + 1, N):
                if par[b, c] == cur and tok[b, c] == want:
                    nxt = c
                    break
            if nxt < 0:
                break
            path[b, n] = nxt
            n += 1
            cur = nxt
        length[b] = n
        bonus[b] = tn[b, cur + 1]
    if k_cache is None:
        return path, length, bonus, None, None, None, status
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    kd = np.asarray(k_draft)
    vd = np.asarray(v_draft)
    ctx = np.array(ctx_lens, dtype=np.int64, copy=True)
    L = kc.shape[2]
    for b in range(B):
        c0 = int(ctx[b])
        if not (0 <= c0 <= L):
            status = 5
            continue
        fit = min(int(length[b]), L - c0)
        if fit < length[b]:
            status = 5
        for j in range(fit):
            node = path[b, j]
            kc[b, :, c0 + j, :] = kd[b, node, :, :]
            vc[b, :, c0 + j, :] = vd[b, node, :, :]
        ctx[b] = c0 + fit
    return path, length, bonus, kc, vc, ctx, status


def budget_plan(marginals, n_max, *, t_draft, l_ar, bytes0, bytes_per_node, flops_per_node, bw, peak, cal_n, cal_t):
    """Tree size chosen by BASTION's online budget controller (BASTION "Metodologia").

    Section 1 (path score): node i at depth d reached through candidates
    c_1..c_d has rho(i) = prod_k q_k(c_k), q_k = marginals[k - 1].
    Section 2 (surrogate, best-first expansion): A(T) = sum of rho over the
    tree; the tree grows by repeatedly adding the frontier node with the largest
    rho (a node's children are the candidates of the next position). Ties go to
    the candidate that entered the frontier first (children enter in candidate
    order).
    Section 3 (controller): T_verify(N) comes from a roofline,
    max((bytes0 + bytes_per_node N) / bw, flops_per_node N / peak), corrected as
    a T_roof + c with (a, c) the least-squares fit to the measured samples
    (cal_n, cal_t) (with fewer than two distinct roofline values: a = mean(t) /
    mean(T_roof), c = 0). S(N) = A(T_N) l_ar / C(N) with C(N) = t_draft +
    T_verify(N), the drafting cost being the same for every topology. The tree
    grows one node at a time and the answer is the last N before S first
    decreases (or the last N grown, at n_max or when no candidate is left).

    Returns a dict: n (the chosen size), n_eval (sizes evaluated), parents,
    depth, cand, rho (of the n_eval nodes grown), speedup (S(1..n_eval)), a, c.
    """
    q = np.asarray(marginals, dtype=np.float64)
    K, C = q.shape
    cal_n = np.asarray(cal_n, dtype=np.float64)
    cal_t = np.asarray(cal_t, dtype=np.float64)

    def t_roof(n):
        return max((bytes0 + bytes_per_node * n) / bw, flops_per_node * n / peak)

    x = np.array([t_roof(n) for n in cal_n])
    if len(set(x.tolist())) < 2:
        a, c = float(cal_t.mean() / x.mean()), 0.0
    else:
        xm, tm = x.mean(), cal_t.mean()
        a = float(((x - xm) * (cal_t - tm)).sum() / ((x - xm) ** 2).sum())
        c = float(tm - a * xm)

    # frontier entries: [rho, order, parent, depth, candidate]
    frontier = []
    order = 0
    for cc in range(C):
        frontier.append([float(q[0, cc]), order, -1, 1, cc])
        order += 1
    parents, depth, cand, rho, speedup = [], [], [], [], []
    surrogate = 0.0
    n_star = 0
    while len(parents) < n_max and frontier:
        best = 0
        for j in range(1, len(frontier)):
            r, o = frontier[j][0], frontier[j][1]
            if r > frontier[best][0] or (r == frontier[best][0] and o < frontier[best][1]):
                best = j
        r, _, par, dep, cc = frontier.pop(best)
        node = len(parents)
        parents.append(par)
        depth.append(dep)
        cand.append(cc)
        rho.append(r)
        if dep < K:
            for c2 in range(C):
                frontier.append([r * float(q[dep, c2]), order, node, dep + 1, c2])
                order += 1
        surrogate += r
        n = node + 1
        cost = t_draft + (a * t_roof(n) + c)
        if not cost > 0:
            raise ValueError("budget_plan: non-positive step cost")
        speedup.append(surrogate * l_ar / cost)
        if n >= 2 and speedup[-1] < speedup[-2]:
            n_star = n - 1
            break
        n_star = n
    return dict(n=n_star, n_eval=len(parents), parents=parents, depth=depth, cand=cand, rho=rho,
                speedup=speedup, a=a, c=c)


def importance_scores(q, k_cache, lse, heads, *, scale: float, ctx_lens=None):
    """Target-historical importance of each cache token (Dustin "Metodologia").

    Section 1 fuses target-historical attention (the target's attention scores
    from its forward passes) with the drafter's; section 2 restricts the scoring
    to a few semantic retrieval heads found offline. The pages do not say how the
    scores of several heads and queries combine; the plainest reading, taken
    here: the score of cache token t of sequence b is the sum, over the listed
    query heads h (a head listed twice counts twice) and the N draft queries i,
    of the final attention probability of row (b, i, h) on t,
    exp(scale q[b,i,h] . k[b, h // G, t] - lse[b,i,h]), with lse the row's
    log-sum-exp over everything it attends (as spec_verify_attn returns it).
    Tokens at or past ctx_lens[b] score 0, and so do rows with lse = -inf.

    q [B, N, Hq, d], k_cache [B, Hkv, L, d], lse [B, N, Hq] (natural log),
    heads: query-head indices. Returns fp64 [B, L].
    """
    qn = np.asarray(q, dtype=np.float64)
    kc = np.asarray(k_cache, dtype=np.float64)
    ln = np.asarray(lse, dtype=np.float64)
    B, N, Hq, d = qn.shape
    _, Hkv, L, _ = kc.shape
    G = Hq // Hkv
    ctx = np.full(B, L, dtype=np.int64) if ctx_lens is None else np.asarray(ctx_lens, dtype=np.int64)
    out = np.zeros((B, L), dtype=np.float64)
    for b in range(B):
        n = int(min(max(ctx[b], 0), L))
        for h in heads:
            s = scale * (qn[b, :, h, :] @ kc[b, h // G, :n, :].T)  # [N, n]
            row = ln[b, :, h][:, None]
            p = np.where(np.isfinite(row), np.exp(s - np.where(np.isfinite(row), row, 0.0)), 0.0)
            out[b, :n] += p.sum(axis=0)
    return out
