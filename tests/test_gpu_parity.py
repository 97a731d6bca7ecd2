"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Tolerances (from the arithmetic the path must meet): selection indices
bit-exact; attention outputs within max-abs 1e-2 of the fp64 oracle and,
because |o| is only ~0.01 for flat softmax at long context, also within
2e-2 * max|o_ref| (relative infinity norm); lse within 1e-3 absolute.
Large workloads are checked on sampled rows, which the oracle computes one by
one; needles at tile and split boundaries catch a skipped or doubled tile that
the flat-softmax tolerance could miss.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_77_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL_O, RTOL_O, ATOL_L = 1e-2, 2e-2, 1e-3


@pytest.fixture(scope="module")
def ops():
    from speculative_decoding_verification_77_gb300 import ops as o

    o.load_library()
    return o


def dev():
    return torch.device("cuda:0")


def to_dev(x):
    return {k: (v.to(dev()) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def assert_attn_close(out, lse, ro, rl, rows=None):
    o = out.float().cpu().numpy().reshape(-1, out.shape[-1])
    l_ = lse.float().cpu().numpy().reshape(-1)
    if rows is not None:
        o, l_ = o[rows], l_[rows]
    assert np.all(np.isfinite(o)), "non-finite output"
    err = np.abs(o - ro).max()
    ref = np.abs(ro).max()
    assert err <= ATOL_O, f"max-abs {err}"
    assert err <= RTOL_O * ref + 1e-7, f"relative {err / ref}"
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(l_), fin)
    assert np.abs(l_[fin] - rl[fin]).max(initial=0) <= ATOL_L, f"lse {np.abs(l_[fin] - rl[fin]).max()}"


def sample_rows(B, N, Hq, k, seed=0):
    rng = np.random.default_rng(seed)
    total = B * N * Hq
    rows = set(rng.choice(total, size=min(k, total), replace=False).tolist())
    rows |= {0, total - 1, Hq - 1, (N - 1) * Hq}
    return np.array(sorted(rows), dtype=np.int64)


def run_dense(ops, x, g, rows=None, **kw):
    out, lse = ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], g["parent"],
                               scale=x["scale"], ctx_lens=kw.get("ctx_lens_dev"))
    ro, rl, st = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                               scale=x["scale"], rows=rows, ctx_lens=kw.get("ctx_lens"))
    assert st == 0
    torch.cuda.synchronize()
    assert_attn_close(out, lse, ro, rl, rows)
    return out, lse


# ---------------------------------------------------------------------------
# the five workloads


def test_workload1_tiny_dense_all_rows(ops):
    x = W.make_inputs(W.workload(1))
    run_dense(ops, x, to_dev(x))


def test_workload2_llama_layer_all_rows(ops):
    """The headline, every one of its 8,192 output rows against the oracle."""
    x = W.make_inputs(W.workload(2))
    run_dense(ops, x, to_dev(x))


def test_workload3_sparse_hybrid(ops):
    w = W.workload(3)
    x = W.make_inputs(w)
    g = to_dev(x)
    idx, cnt = ops.select_topk(g["draft_score"], g["target_score"], sink=w.sink, window=w.window,
                               top_m=w.top_m, budget=w.budget)
    ridx, rcnt, st = oracle.select(x["draft_score"], x["target_score"], sink=w.sink, window=w.window,
                                   top_m=w.top_m, budget=w.budget)
    assert st == 0
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)
    out, lse = ops.verify_attn_sparse(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"],
                                      g["parent"], idx, scale=x["scale"])
    rows = sample_rows(w.B, w.N, w.Hq, 512)
    ro, rl, st = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                               scale=x["scale"], idx=torch.from_numpy(ridx), rows=rows)
    assert st == 0
    assert_attn_close(out, lse, ro, rl, rows)


def test_selection_and_sparse_verify_back_to_back(ops):
    """The sparse verify's first kernel may launch while the selection runs (the selection lets
    dependents start, the verify's kernels wait for it before they read the index set). Two
    score sets with different selections alternate with no synchronisation in between: every
    result must equal, bit for bit, the same pair run with a synchronisation after the
    selection."""
    w = W.workload(3)
    x = W.make_inputs(w)
    g = to_dev(x)
    sets = [(g["draft_score"], g["target_score"]), (g["target_score"], g["draft_score"])]

    def pair(s, sync):
        idx, _ = ops.select_topk(sets[s][0], sets[s][1], sink=w.sink, window=w.window, top_m=w.top_m,
                                 budget=w.budget)
        if sync:
            torch.cuda.synchronize()
        out, lse = ops.verify_attn_sparse(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"],
                                          g["parent"], idx, scale=x["scale"])
        return idx, out, lse

    ref = []
    for s in range(2):
        r = pair(s, True)
        torch.cuda.synchronize()
        ref.append(r)
    assert not torch.equal(ref[0][0], ref[1][0])  # the two sets select different tokens
    runs = [(i % 2, pair(i % 2, False)) for i in range(12)]
    torch.cuda.synchronize()
    for s, (idx, out, lse) in runs:
        assert torch.equal(idx, ref[s][0])
        assert torch.equal(out, ref[s][1])
        assert torch.equal(lse, ref[s][2])


def unit_rows(w, per_half, seed):
    """Rows covering every (b, h_kv) unit of a dense workload, per_half rows in each half of the
    unit's rows (query heads of h_kv x draft nodes, node-major): the halves are the two softmax
    pipes of the tensor-core kernel when a unit has more than 128 rows."""
    rng = np.random.default_rng(seed)
    G, half = w.G, max(1, w.N // 2)
    rows = []
    for b in range(w.B):
        for hk in range(w.Hkv):
            for lo, hi in ((0, half), (half, w.N)):
                pick = rng.choice((hi - lo) * G, size=min(per_half, (hi - lo) * G), replace=False)
                i, h = lo + pick // G, hk * G + pick % G
                rows += ((b * w.N + i) * w.Hq + h).tolist()
    return np.array(sorted(set(rows)), dtype=np.int64)


def test_workload4_qwen_layer_every_unit(ops):
    """Qwen2.5-72B-shaped layer (G = 8, L = 128k): 2,048 rows, 32 from every (b, h_kv) unit,
    16 from each half of the unit's rows."""
    x = W.make_inputs(W.workload(4))
    w = x["workload"]
    rows = unit_rows(w, 16, seed=4)
    assert len(rows) == 2048 and len({(r // w.Hq // w.N, (r % w.Hq) // w.G) for r in rows}) == w.B * w.Hkv
    run_dense(ops, x, to_dev(x), rows=rows)


@pytest.mark.parametrize("N", [1, 4, 16, 64, 256])
def test_workload5_tree_sweep_sampled(ops, N):
    x = W.make_inputs(W.workload(5, N))
    w = x["workload"]
    run_dense(ops, x, to_dev(x), rows=sample_rows(w.B, w.N, w.Hq, 160, seed=N))


# ---------------------------------------------------------------------------
# edge cases


def small(seed, B=2, N=5, Hq=8, Hkv=2, L=333, tree="random", depth=3):
    w = W.Workload("edge", B=B, L=L, Hq=Hq, Hkv=Hkv, N=N, tree=tree, depth_max=depth, seed=seed)
    return W.make_inputs(w)


@pytest.mark.parametrize("L", [0, 1, 63, 64, 65, 200, 1000])
def test_ragged_lengths_and_tails(ops, L):
    x = small(L + 1, L=L)
    run_dense(ops, x, to_dev(x))


def test_ragged_ctx_lens(ops):
    x = small(3, B=4, L=777)
    cl = torch.tensor([777, 700, 5, 0], dtype=torch.int32)
    run_dense(ops, x, to_dev(x), ctx_lens=cl, ctx_lens_dev=cl.to(dev()))


@pytest.mark.parametrize("tree", ["chain", "star", "forest"])
def test_tree_shapes(ops, tree):
    x = small(11, N=12, L=300, tree="chain")
    if tree == "star":
        x["parent"] = torch.full((2, 12), -1, dtype=torch.int32)
    elif tree == "forest":
        x["parent"] = torch.tensor([[-1, 0, -1, 2, 1, -1, 5, 6, 3, 8, -1, 10]] * 2, dtype=torch.int32)
    run_dense(ops, x, to_dev(x))


# (130, 8, 2) and (70, 8, 1): three row groups per KV head, so the tensor-core kernel's plan gives
# each row group its own block of CTAs with the same cut (on 152 SMs, 50 CTAs a block and two SMs
# without a CTA; on smaller problems as many CTAs as the tiles allow)
@pytest.mark.parametrize("N,Hq,Hkv", [(300, 4, 1), (17, 16, 2), (1, 1, 1), (33, 12, 4), (130, 8, 2), (70, 8, 1)])
def test_row_groups_and_head_ratios(ops, N, Hq, Hkv):
    x = small(5, B=1, N=N, Hq=Hq, Hkv=Hkv, L=500, depth=6)
    run_dense(ops, x, to_dev(x))


# Up to 256 nodes the speculative part runs as its own small-block grid beside the cache
# kernel (parents held in registers, 32 a register); above that the merge walks the tree
# itself. Chains put the deepest walks on both sides of that bound, with G = 8 (two warps
# of four heads per node in the separate grid) and G = 3 (one head per warp).
@pytest.mark.parametrize("N,Hq,Hkv", [(256, 16, 2), (257, 8, 2), (256, 6, 2), (255, 4, 4)])
def test_deep_chains_both_tree_paths(ops, N, Hq, Hkv):
    x = small(31 + N, B=2, N=N, Hq=Hq, Hkv=Hkv, L=700, tree="chain")
    run_dense(ops, x, to_dev(x))


def test_cache_only_then_merge_equals_full(ops):
    x = small(21, L=900)
    g = to_dev(x)
    full_o, full_l = ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"],
                                     g["parent"], scale=x["scale"])
    co, cl = ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], scale=x["scale"])
    # tree part alone: an empty cache
    e = g["k_cache"][:, :, :0]
    to, tl = ops.verify_attn(g["q"], e, e, g["k_draft"], g["v_draft"], g["parent"], scale=x["scale"])
    mo, ml = ops.lse_merge(co, cl, to, tl)
    torch.cuda.synchronize()
    assert torch.allclose(mo, full_o, atol=1e-5, rtol=0)
    assert torch.allclose(ml, full_l, atol=1e-5, rtol=0)
    # each part against the oracle, and the merge against the oracle's merge
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], None, None, x["parent"], scale=x["scale"])
    assert_attn_close(co, cl, ro, rl)
    mo_ref, ml_ref = oracle.lse_merge(co.cpu(), cl.cpu(), to.cpu(), tl.cpu())
    np.testing.assert_allclose(mo.cpu().numpy().reshape(mo_ref.shape), mo_ref, atol=1e-6, rtol=0)
    np.testing.assert_allclose(ml.cpu().numpy().reshape(-1), ml_ref, atol=1e-5, rtol=0)


# d = 128: one float4 per lane; 256: two; 36: lanes past d idle; 70: the scalar form
@pytest.mark.parametrize("d", [128, 256, 36, 70])
def test_lse_merge_special_rows_and_in_place(ops, d):
    rows = 1000
    gen = torch.Generator().manual_seed(3)
    oa = torch.randn(rows, d, generator=gen)
    ob = torch.randn(rows, d, generator=gen)
    la = torch.randn(rows, generator=gen) * 5
    lb = torch.randn(rows, generator=gen) * 5
    la[:10] = -math.inf
    lb[5:15] = -math.inf
    oa[:10] = 0
    ob[5:15] = 0
    ref_o, ref_l = oracle.lse_merge(oa, la, ob, lb)
    go, gl = oa.to(dev()), la.to(dev())
    ops.lse_merge(go, gl, ob.to(dev()), lb.to(dev()), out=go, lse_out=gl)  # in place
    torch.cuda.synchronize()
    np.testing.assert_allclose(go.cpu().numpy(), ref_o, atol=1e-5, rtol=0)
    got_l = gl.cpu().numpy()
    assert np.array_equal(np.isinf(got_l), np.isinf(ref_l))
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(got_l[fin], ref_l[fin], atol=1e-5, rtol=0)


@pytest.mark.parametrize("pos", [0, 63, 64, 127, 128, 4095, 4096, 9999])
def test_needle_positions(ops, pos):
    """One key with logit ~ +30 at tile/split boundaries: o must be that key's V."""
    x = small(pos, B=1, N=2, Hq=4, Hkv=2, L=10000)
    q = x["q"]
    scale = x["scale"]
    qv = q[0, 0, 2].double()
    x["k_cache"][0, 1, pos] = (qv * (30.0 / (scale * float(qv.dot(qv))))).to(torch.bfloat16)
    rows = np.array([2])
    g = to_dev(x)
    out, lse = ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], g["parent"],
                               scale=scale)
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                              scale=scale, rows=rows)
    torch.cuda.synchronize()
    o = out.cpu().numpy().reshape(-1, 128)[2]
    assert np.abs(o - x["v_cache"][0, 1, pos].float().numpy()).max() < 2e-2
    assert_attn_close(out, lse, ro, rl, rows)


@pytest.mark.parametrize("needles", [((138, 50.0), (198, 100.0)), ((200, 50.0), (9000, 120.0)),
                                     ((70, 60.0), (4100, 130.0), (8190, 200.0))])
def test_huge_logit_jumps_rescale_o(ops, needles):
    """Keys whose logits jump far above everything before them (by more than 64 in base 2,
    about 44 natural) later in the cache, also in consecutive halves of one tile: O must be
    rescaled while earlier PV products may still be running."""
    x = small(77, B=1, N=2, Hq=4, Hkv=2, L=10000)
    q, scale = x["q"], x["scale"]
    qv = q[0, 0, 2].double()
    for pos, logit in needles:
        x["k_cache"][0, 1, pos] = (qv * (logit / (scale * float(qv.dot(qv))))).to(torch.bfloat16)
    g = to_dev(x)
    out, lse = ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], g["parent"],
                               scale=scale)
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                              scale=scale)
    torch.cuda.synchronize()
    strongest = max(needles, key=lambda n: n[1])[0]
    o = out.cpu().numpy().reshape(-1, 128)[2]
    assert np.abs(o - x["v_cache"][0, 1, strongest].float().numpy()).max() < 2e-2
    assert_attn_close(out, lse, ro, rl)


def test_strided_cache_layout(ops):
    """K/V as [B, L, Hkv, d] memory viewed as [B, Hkv, L, d] (token-major cache)."""
    x = small(8, B=2, L=400, Hq=8, Hkv=4)
    kc = x["k_cache"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    g = to_dev(x)
    gk = x["k_cache"].permute(0, 2, 1, 3).contiguous().to(dev()).permute(0, 2, 1, 3)
    gv = x["v_cache"].permute(0, 2, 1, 3).contiguous().to(dev()).permute(0, 2, 1, 3)
    assert gk.stride() == kc.stride()
    out, lse = ops.verify_attn(g["q"], gk, gv, g["k_draft"], g["v_draft"], g["parent"], scale=x["scale"])
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                              scale=x["scale"])
    torch.cuda.synchronize()
    assert_attn_close(out, lse, ro, rl)


def test_sparse_budget_covering_context_equals_dense(ops):
    x = small(31, L=500)
    g = to_dev(x)
    idx = torch.cat([torch.arange(500, dtype=torch.int32), torch.full((12,), -1, dtype=torch.int32)])
    idx = idx.repeat(2, 1).to(dev())
    so, sl = ops.verify_attn_sparse(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"],
                                    g["parent"], idx, scale=x["scale"])
    do, dl = ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], g["parent"],
                             scale=x["scale"])
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                              scale=x["scale"])
    torch.cuda.synchronize()
    # the sparse and dense paths run different cache kernels: each must meet the oracle,
    # and they agree with each other to the bf16 rounding of P
    assert_attn_close(so, sl, ro, rl)
    assert_attn_close(do, dl, ro, rl)
    assert torch.allclose(so, do, atol=2e-3, rtol=0) and torch.allclose(sl, dl, atol=1e-4, rtol=0)


def test_sparse_ragged_selection(ops):
    x = small(41, B=3, L=2000, N=6)
    ds, ts = W.random_scores(3, 2000, seed=4, ties=6)
    cl = torch.tensor([2000, 1500, 100], dtype=torch.int32)
    g = to_dev(x)
    kw = dict(sink=4, window=64, top_m=128, budget=300)
    idx, cnt = ops.select_topk(ds.to(dev()), ts.to(dev()), ctx_lens=cl.to(dev()), **kw)
    ridx, rcnt, _ = oracle.select(ds, ts, ctx_lens=cl, **kw)
    assert np.array_equal(idx.cpu().numpy(), ridx) and np.array_equal(cnt.cpu().numpy(), rcnt)
    out, lse = ops.verify_attn_sparse(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"],
                                      g["parent"], idx, scale=x["scale"], ctx_lens=cl.to(dev()))
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                              scale=x["scale"], idx=torch.from_numpy(ridx), ctx_lens=cl)
    torch.cuda.synchronize()
    assert_attn_close(out, lse, ro, rl)


def strided_cache(x, sb, sh, st):
    """The cache tensor x [B, Hkv, L, d] copied into a device buffer with element strides (sb, sh, st, 1)."""
    B, H, L, d = x.shape
    flat = torch.zeros((B - 1) * sb + (H - 1) * sh + (L - 1) * st + d, dtype=x.dtype, device=dev())
    view = torch.as_strided(flat, (B, H, L, d), (sb, sh, st, 1))
    view.copy_(x.to(dev()))
    return view


@pytest.mark.parametrize("case", ["g3_warp_kernel", "token_major", "padding_runs", "row_groups", "one_tile",
                                  "padded_rows", "padded_batch"])
def test_sparse_paths(ops, case):
    """Sparse verify on both cache kernels, on cache strides that are multiples of 8 but not of
    d, and on the index patterns each must mask."""
    shapes = {"g3_warp_kernel": dict(B=2, N=7, Hq=12, Hkv=4, L=3000),  # G = 3: warp-level kernel
              "token_major": dict(B=2, N=5, Hq=8, Hkv=4, L=2500),
              # token-major, token rows padded to 576 elements, batches shifted by 8 elements
              "padded_rows": dict(B=3, N=5, Hq=8, Hkv=4, L=2500),
              # head-major with batches shifted by 8 elements
              "padded_batch": dict(B=3, N=5, Hq=8, Hkv=2, L=2500),
              "padding_runs": dict(B=2, N=5, Hq=8, Hkv=2, L=2500),
              "row_groups": dict(B=2, N=40, Hq=16, Hkv=2, L=2600),  # G*N = 320 rows: three row groups
              "one_tile": dict(B=1, N=3, Hq=4, Hkv=1, L=90)}[case]
    x = small(77, depth=5, **shapes)
    B, L = shapes["B"], shapes["L"]
    ds, ts = W.random_scores(B, L, seed=11)
    budget = 80 if case == "one_tile" else 700
    kw = dict(sink=4, window=32, top_m=200 if budget > 100 else 20, budget=budget)
    ridx, _, st = oracle.select(ds, ts, **kw)
    assert st == 0
    if case == "padding_runs":  # unused slots inside the list: -1 runs, a repeat, an out-of-range entry
        ridx = ridx.copy()
        ridx[0, 100:230] = -1
        ridx[1, 128:256] = -1
        ridx[1, 300] = ridx[1, 299]
        ridx[1, 400] = L + 5
    idx = torch.from_numpy(ridx)
    g = to_dev(x)
    k, v = g["k_cache"], g["v_cache"]
    if case == "token_major":
        k = x["k_cache"].permute(0, 2, 1, 3).contiguous().to(dev()).permute(0, 2, 1, 3)
        v = x["v_cache"].permute(0, 2, 1, 3).contiguous().to(dev()).permute(0, 2, 1, 3)
    if case == "padded_rows":
        st = 4 * 128 + 64
        k, v = (strided_cache(x[n], L * st + 8, 128, st) for n in ("k_cache", "v_cache"))
    if case == "padded_batch":
        k, v = (strided_cache(x[n], 2 * L * 128 + 8, L * 128, 128) for n in ("k_cache", "v_cache"))
    out, lse = ops.verify_attn_sparse(g["q"], k, v, g["k_draft"], g["v_draft"], g["parent"], idx.to(dev()),
                                      scale=x["scale"])
    ro, rl, st = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                               scale=x["scale"], idx=idx)
    assert st == (5 if case == "padding_runs" else 0)
    torch.cuda.synchronize()
    assert_attn_close(out, lse, ro, rl)


@pytest.mark.parametrize("slot", [0, 5, 70, 127, 128, 255, 1999])
def test_sparse_needle_at_index_slot(ops, slot):
    """A key with logit ~ +30 behind index slot `slot`: o must be that key's V."""
    x = small(300 + slot, B=1, N=2, Hq=4, Hkv=2, L=9000)
    idx = torch.from_numpy(np.sort(np.random.default_rng(slot).choice(9000, size=2000, replace=False))
                           .astype(np.int32))[None]
    t = int(idx[0, slot])
    qv = x["q"][0, 1, 3].double()
    x["k_cache"][0, 1, t] = (qv * (30.0 / (x["scale"] * float(qv.dot(qv))))).to(torch.bfloat16)
    g = to_dev(x)
    out, lse = ops.verify_attn_sparse(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"],
                                      g["parent"], idx.to(dev()), scale=x["scale"])
    rows = np.array([1 * 4 + 3])
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                              scale=x["scale"], idx=idx, rows=rows)
    torch.cuda.synchronize()
    o = out.cpu().numpy().reshape(-1, 128)[rows[0]]
    assert np.abs(o - x["v_cache"][0, 1, t].float().numpy()).max() < 2e-2
    assert_attn_close(out, lse, ro, rl, rows)


@pytest.mark.parametrize("case", ["ties", "special", "small_ctx", "big_top_m", "zero_top_m", "ties_32k",
                                  "special_32k", "unaligned_rows_32k", "small_ctx_32k", "cluster_40k",
                                  "cluster_ties_40k", "ties_12k", "cluster_100k", "staged_cluster_140k",
                                  "staged_cluster_ties_140k"])
def test_selection_cases_bit_exact(ops, case):
    """Both selection kernels: a 4-CTA cluster per sequence with the keys in registers up to
    64k tokens (one, two, four or eight quads per warp), 8 CTAs up to 128k, the cluster with
    staged keys beyond."""
    B, L = 5, 5000
    if case.endswith("_32k"):
        B, L = 3, 32768
    if case.endswith("_40k"):
        B, L = 3, 40000
    if case.endswith("_12k"):
        B, L = 4, 12000
    if case.endswith("_100k"):
        B, L = 2, 100000
    if case.endswith("_140k"):
        B, L = 2, 140000
    ds, ts = W.random_scores(B, L, seed=7, ties=3 if "ties" in case else 0)
    kw = dict(sink=4, window=64, top_m=512, budget=1024)
    cl = None
    if case.startswith("special"):
        rng = np.random.default_rng(0)
        for arr in (ds, ts):
            pick = rng.choice(B * L, size=2000, replace=False)
            vals = np.array([np.nan, -0.0, 0.0, np.inf, -np.inf], np.float32)
            arr.view(-1)[torch.from_numpy(pick)] = torch.from_numpy(rng.choice(vals, size=2000))
    if case == "small_ctx":
        cl = torch.tensor([5000, 1024, 1025, 68, 0], dtype=torch.int32)
    if case == "small_ctx_32k":
        cl = torch.tensor([32768, 1025, 20001], dtype=torch.int32)
    if case == "big_top_m":
        kw["top_m"] = 5000
    if case == "zero_top_m":
        kw["top_m"] = 0
    gds, gts = ds.to(dev()), ts.to(dev())
    if case == "unaligned_rows_32k":  # row stride of 32771 floats: rows off 16-byte boundaries
        pad = lambda t: torch.nn.functional.pad(t, (0, 3))[:, :L]
        gds, gts = pad(gds), pad(gts)
        assert gds.stride(0) == L + 3
    idx, cnt = ops.select_topk(gds, gts, ctx_lens=None if cl is None else cl.to(dev()), **kw)
    ridx, rcnt, _ = oracle.select(ds, ts, ctx_lens=cl, **kw)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)


def test_bad_inputs_set_the_status_word(ops):
    x = small(51, L=300, tree="chain")
    g = to_dev(x)
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device=dev())
    ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], g["parent"],
                    scale=x["scale"], ws=ws)
    assert ops.read_device_status(ws) == 0
    bad = g["parent"].clone()
    bad[0, 3] = 7  # parent after the node
    out, lse = ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], bad,
                               scale=x["scale"], ws=ws)
    assert ops.read_device_status(ws) == 5
    ro, rl, st = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], bad.cpu(),
                               scale=x["scale"])
    assert st == 5
    assert_attn_close(out, lse, ro, rl)
    idx = torch.tensor([[0, 5, 5, 2, 999, -1], [1, 2, 3, -1, -1, -1]], dtype=torch.int32)
    out, lse = ops.verify_attn_sparse(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"],
                                      g["parent"], idx.to(dev()), scale=x["scale"], ws=ws)
    assert ops.read_device_status(ws) == 5
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                              scale=x["scale"], idx=idx)
    assert_attn_close(out, lse, ro, rl)
    # a clean call clears the word again
    ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], g["parent"],
                    scale=x["scale"], ws=ws)
    assert ops.read_device_status(ws) == 0
    # selection: a context length outside [0, L] is clamped and reported, on both selection
    # kernels (registers up to 128k tokens, staged keys beyond); a clean call reports nothing
    for L in (3000, 140000):
        ds, ts = W.random_scores(3, L, seed=L)
        kw = dict(sink=4, window=16, top_m=64, budget=256)
        sws = torch.full((256,), 255, dtype=torch.uint8, device=dev())
        cl = torch.tensor([L, -5, L + 9], dtype=torch.int32)
        idx, cnt = ops.select_topk(ds.to(dev()), ts.to(dev()), ctx_lens=cl.to(dev()), ws=sws, **kw)
        assert ops.read_device_status(sws) == 5
        ridx, rcnt, st = oracle.select(ds, ts, ctx_lens=cl, **kw)
        assert st == 5 and np.array_equal(idx.cpu().numpy(), ridx) and np.array_equal(cnt.cpu().numpy(), rcnt)
        ops.select_topk(ds.to(dev()), ts.to(dev()), ws=sws, **kw)
        assert ops.read_device_status(sws) == 0


def test_status_word_of_back_to_back_calls(ops):
    """Calls on one workspace with no synchronisation between them: the word holds the last
    call's result. Its clearing kernel may launch while the previous call's kernels run, so it
    must wait for them: a bad tree flagged late by the previous call's merge must not survive
    into a clean call, and a clean call must not hide the bad one after it."""
    x = small(52, L=300, tree="chain")
    g = to_dev(x)
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device=dev())
    bad = g["parent"].clone()
    bad[0, 3] = 7  # parent after the node
    good = g["parent"]

    def call(parent):
        ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], parent,
                        scale=x["scale"], ws=ws)

    for first, second, want in ((bad, good, 0), (good, bad, 5), (bad, bad, 5), (good, good, 0)):
        for _ in range(4):
            call(first)
            call(second)
        assert ops.read_device_status(ws) == want


def test_native_kernels_ran(ops):
    before = ops.kernel_launches()
    x = small(61, L=100)
    g = to_dev(x)
    ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], g["parent"])
    torch.cuda.synchronize()
    assert ops.kernel_launches() >= before + 2


def test_workspace_too_small_is_rejected(ops):
    x = small(71, L=100)
    g = to_dev(x)
    ws = torch.zeros(512, dtype=torch.uint8, device=dev())
    with pytest.raises(ops.SpecError) as e:
        ops.verify_attn(g["q"], g["k_cache"], g["v_cache"], g["k_draft"], g["v_draft"], g["parent"], ws=ws)
    assert e.value.code == 4


# ---------------------------------------------------------------- acceptance and cache commit

def accept_inputs(seed, B, N, Hkv, L, ctx, tree="random"):
    """Random draft trees with small token ids (so that siblings share tokens) and the
    target's tokens made to follow a random root path of each tree."""
    rng = np.random.default_rng(seed)
    if tree == "chain":
        par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    else:
        par = np.stack([np.array([-1] + [int(rng.integers(max(-1, i - 9), i)) for i in range(1, N)], np.int32)
                        for _ in range(B)])
    tok = rng.integers(0, 4, (B, N)).astype(np.int32)
    tn = rng.integers(0, 4, (B, N + 1)).astype(np.int32)
    for b in range(B):
        c = N - 1 if tree == "chain" else int(rng.integers(0, N))
        while c >= 0:
            tn[b, par[b, c] + 1] = tok[b, c]
            c = par[b, c]
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn((B, Hkv, L, 128), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, L, 128), generator=g).to(torch.bfloat16)
    kd = torch.randn((B, N, Hkv, 128), generator=g).to(torch.bfloat16)
    vd = torch.randn((B, N, Hkv, 128), generator=g).to(torch.bfloat16)
    return tok, par, tn, kc, vc, kd, vd, np.asarray(ctx, np.int32)


@pytest.mark.parametrize("case", ["tree", "chain_n256", "n1", "room_runs_out", "bad_ctx", "bad_parent",
                                  "no_commit", "token_major"])
def test_accept_commit_matches_oracle(ops, case):
    """Greedy acceptance and cache commit: path, length, bonus, caches and lengths bit-exact."""
    B, N, Hkv, L = 4, 64, 8, 1024
    tree = "random"
    ctx = [0, 100, 517, 900]
    if case == "chain_n256":
        N, tree = 256, "chain"
        ctx = [0, 3, 500, 768]
    if case == "n1":
        N = 1
    if case == "room_runs_out":
        ctx = [L - 1, L - 2, L, 10]
    if case == "bad_ctx":
        ctx = [-1, L + 5, 7, 8]
    tok, par, tn, kc, vc, kd, vd, ctx = accept_inputs(11 + len(case), B, N, Hkv, L, ctx, tree)
    if case == "bad_parent":
        par[1, 5] = 5
        par[2, 7] = -3
    commit = case != "no_commit"
    want = oracle.accept_commit(tok, par, tn, *((kc.view(torch.int16).numpy(), vc.view(torch.int16).numpy(),
                                                 kd.view(torch.int16).numpy(), vd.view(torch.int16).numpy(), ctx)
                                                if commit else ()))
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    if commit:
        gk, gv = kc.to(dev()), vc.to(dev())
        if case == "token_major":
            gk = kc.permute(0, 2, 1, 3).contiguous().to(dev()).permute(0, 2, 1, 3)
            gv = vc.permute(0, 2, 1, 3).contiguous().to(dev()).permute(0, 2, 1, 3)
        gctx = d(ctx)
        path, length, bonus, status = ops.accept_commit(d(tok), d(par), d(tn), gk, gv, kd.to(dev()), vd.to(dev()), gctx)
    else:
        path, length, bonus, status = ops.accept_commit(d(tok), d(par), d(tn))
    torch.cuda.synchronize()
    assert np.array_equal(path.cpu().numpy(), want[0])
    assert np.array_equal(length.cpu().numpy(), want[1])
    assert np.array_equal(bonus.cpu().numpy(), want[2])
    assert int(status.item()) == want[6]
    assert want[6] == (5 if case in ("room_runs_out", "bad_ctx", "bad_parent") else 0)
    if commit:
        assert np.array_equal(gctx.cpu().numpy(), want[5])
        assert np.array_equal(gk.cpu().contiguous().view(torch.int16).numpy(), want[3])
        assert np.array_equal(gv.cpu().contiguous().view(torch.int16).numpy(), want[4])
        assert want[1].max() > 0  # the planted paths were accepted


# ---------------------------------------------------------------- importance scores

@pytest.mark.parametrize("case", ["ragged", "repeated_heads_g8", "bad_head", "n24_tail", "fma_form_n200",
                                  "draft_lookahead"])
def test_importance_scores_match_oracle(ops, case):
    """Target-historical scores on the listed heads (tensor-core form; fma_form_n200 stages more
    than 256 query rows and takes the portable form). Both sides read the same lse: the attention
    oracle's, rounded to fp32 (the dtype the library takes). draft_lookahead feeds the call a
    drafter's own queries, keys and lse (one KV head, four query heads): the same computation
    gives the draft-lookahead signal."""
    shapes = {"ragged": dict(B=2, N=8, Hq=8, Hkv=2, L=3000),
              "repeated_heads_g8": dict(B=1, N=16, Hq=16, Hkv=2, L=1500),
              "bad_head": dict(B=2, N=4, Hq=8, Hkv=2, L=700),
              "n24_tail": dict(B=2, N=24, Hq=8, Hkv=4, L=1111),
              "fma_form_n200": dict(B=1, N=200, Hq=8, Hkv=2, L=900),
              "draft_lookahead": dict(B=2, N=8, Hq=4, Hkv=1, L=2500)}[case]
    heads = {"ragged": [1, 6], "repeated_heads_g8": [0, 9, 9, 15], "bad_head": [2, 99], "n24_tail": [7, 0, 3],
             "fma_form_n200": [1, 5], "draft_lookahead": [0, 1, 2, 3]}[case]
    x = small(91, depth=3, **shapes)
    B, N, Hq, L = shapes["B"], shapes["N"], shapes["Hq"], shapes["L"]
    ctx = np.array([L, 1234][:B] if case == "ragged" else [L] * B, np.int32)
    _, lse64, st = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                                 scale=x["scale"], ctx_lens=torch.from_numpy(ctx))
    assert st == 0
    lse32 = lse64.astype(np.float32).reshape(B, N, Hq)
    valid = [h for h in heads if 0 <= h < Hq]
    want = oracle.importance_scores(x["q"].float().numpy(), x["k_cache"].float().numpy(), lse32.astype(np.float64),
                                    valid, scale=float(np.float32(x["scale"])), ctx_lens=ctx)
    g = to_dev(x)
    stale = torch.full((1,), 7, dtype=torch.int32, device=dev())  # the call must write the word whole
    score, status = ops.importance_scores(g["q"], g["k_cache"], torch.from_numpy(lse32).to(dev()),
                                          torch.tensor(heads, dtype=torch.int32, device=dev()), scale=x["scale"],
                                          ctx_lens=torch.from_numpy(ctx).to(dev()), status=stale)
    torch.cuda.synchronize()
    got = score.cpu().numpy()
    assert int(status.item()) == (5 if case == "bad_head" else 0)
    for b in range(B):
        assert np.all(got[b, ctx[b]:] == 0.0)
    assert np.allclose(got, want, rtol=1e-4, atol=1e-6), np.abs(got - want).max()
    assert want.max() > 0


# ---------------------------------------------------------------- paged KV cache

def paged_case(seed, B, N, Hq, Hkv, L, bs, token_major=False, depth=4):
    """A contiguous problem and the same cache scattered into a pool of bs-row blocks in a random
    order (noise blocks in between): (x, k_pool view, v_pool view [nblk, Hkv, bs, d] on the device,
    block table, number of pool blocks)."""
    from tests.test_oracle_pins import to_pool

    x = small(seed, B=B, N=N, Hq=Hq, Hkv=Hkv, L=L, depth=depth)
    g = torch.Generator().manual_seed(seed)
    kp, vp, table, nblk = to_pool(x["k_cache"], x["v_cache"], bs, g)
    kp, vp = kp[:nblk], vp[:nblk]
    if token_major:  # pool memory [nblk, bs, Hkv, d], seen as [nblk, Hkv, bs, d]
        gk = kp.permute(0, 2, 1, 3).contiguous().to(dev()).permute(0, 2, 1, 3)
        gv = vp.permute(0, 2, 1, 3).contiguous().to(dev()).permute(0, 2, 1, 3)
    else:
        gk, gv = kp.to(dev()), vp.to(dev())
    return x, kp, vp, gk, gv, table, nblk


@pytest.mark.parametrize("case", ["dense_bs128", "dense_bs256_token_major", "dense_bs16", "dense_g3",
                                  "sparse_bs16", "sparse_bs128_token_major", "bad_block_dense", "bad_block_sparse"])
def test_paged_cache_matches_oracle(ops, case):
    """Paged cache on both cache kernels (tensor-core tiles need blocks of a multiple of 128 rows)
    against the paged oracle, which is pinned to the contiguous one bit for bit."""
    Hq, Hkv = (12, 4) if case == "dense_g3" else (8, 2)
    bs = int(case.split("_bs")[1].split("_")[0]) if "_bs" in case else 128
    B, N, L = 2, 6, 1000
    x, kp, vp, gk, gv, table, nblk = paged_case(100 + bs, B, N, Hq, Hkv, L, bs, "token_major" in case)
    cl = torch.tensor([L, 777], dtype=torch.int32)
    idx = None
    if "sparse" in case:
        ds, ts = W.random_scores(B, L, seed=bs)
        idx, _, _ = oracle.select(ds, ts, ctx_lens=cl, sink=4, window=32, top_m=100, budget=300)
        idx = torch.from_numpy(idx)
    if case.startswith("bad_block"):
        table[1, 3] = nblk  # a block inside sequence 1's context that the pool does not have
    g = to_dev(x)
    out, lse = ops.verify_attn_paged(g["q"], gk, gv, table.to(dev()), g["k_draft"], g["v_draft"], g["parent"], L=L,
                                     idx=None if idx is None else idx.to(dev()), scale=x["scale"],
                                     ctx_lens=cl.to(dev()))
    ro, rl, st = oracle.attend_paged(x["q"], kp, vp, x["k_draft"], x["v_draft"], x["parent"], table, L=L,
                                     scale=x["scale"], ctx_lens=cl, idx=idx)
    assert st == (5 if case.startswith("bad_block") else 0)
    ws = ops.workspace(0, dev(), "verify")
    assert ops.read_device_status(ws) == st
    assert_attn_close(out, lse, ro, rl)


def test_paged_headline_shape_sampled(ops):
    """The headline layer's shape (B=4, L=32k, 32/8 heads, N=64 tree) on a pool of 256-row blocks."""
    w = W.workload(2)
    x = W.make_inputs(w)
    from tests.test_oracle_pins import to_pool

    g0 = torch.Generator().manual_seed(2)
    kp, vp, table, nblk = to_pool(x["k_cache"], x["v_cache"], 256, g0)
    kp, vp = kp[:nblk], vp[:nblk]
    g = to_dev(x)
    out, lse = ops.verify_attn_paged(g["q"], kp.to(dev()), vp.to(dev()), table.to(dev()), g["k_draft"],
                                     g["v_draft"], g["parent"], L=w.L, scale=x["scale"])
    rows = unit_rows(w, 8, seed=5)
    ro, rl, st = oracle.attend_paged(x["q"], kp, vp, x["k_draft"], x["v_draft"], x["parent"], table, L=w.L,
                                     scale=x["scale"], rows=rows)
    assert st == 0
    assert_attn_close(out, lse, ro, rl, rows)


@pytest.mark.parametrize("case", ["dense_tc", "dense_g3", "sparse", "paged"])
def test_bf16_output_is_the_rounded_fp32_output(ops, case):
    """out_dtype bf16: the fp32 result of the same call rounded to nearest even, bit for bit, and
    within the oracle tolerance plus one bf16 rounding of |o|."""
    Hq, Hkv = (12, 4) if case == "dense_g3" else (8, 2)
    x = small(200, B=2, N=5, Hq=Hq, Hkv=Hkv, L=900)
    g = to_dev(x)
    kc, vc, kw, okw = g["k_cache"], g["v_cache"], {}, {}
    if case == "sparse":
        ds, ts = W.random_scores(2, 900, seed=3)
        idx, _, _ = oracle.select(ds, ts, sink=4, window=16, top_m=64, budget=256)
        kw["idx"] = torch.from_numpy(idx).to(dev())
        okw["idx"] = torch.from_numpy(idx)
    if case == "paged":
        from tests.test_oracle_pins import to_pool

        kp, vp, table, nblk = to_pool(x["k_cache"], x["v_cache"], 128, torch.Generator().manual_seed(9))
        kc, vc = kp[:nblk].to(dev()), vp[:nblk].to(dev())
        kw.update(block_table=table.to(dev()), L=900)
    args = (g["q"], kc, vc, g["k_draft"], g["v_draft"], g["parent"])
    o32, l32 = ops.verify_attn_ex(*args, scale=x["scale"], **kw)
    o16, l16 = ops.verify_attn_ex(*args, scale=x["scale"], out_dtype=torch.bfloat16, **kw)
    torch.cuda.synchronize()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(l16, l32)
    ro, rl, _ = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                              scale=x["scale"], **okw)
    o = o16.float().cpu().numpy().reshape(ro.shape)
    assert np.abs(o - ro).max() <= ATOL_O + np.abs(ro).max() * 2.0 ** -8


# ---------------------------------------------------------------- fp8 KV cache


def quantize_e4m3(c):
    """A bf16 cache [B, Hkv, L, d] as E4M3 codes with one fp32 scale per (sequence, KV head): the
    head's largest magnitude maps to 448, the format's largest number."""
    amax = c.float().abs().amax(dim=(2, 3)).clamp_min(1e-30)
    sc = (amax / 448.0).to(torch.float32)
    return (c.float() / sc[:, :, None, None]).to(torch.float8_e4m3fn), sc


def codes_to_pool(kc, vc, bs, gen):
    """The code caches scattered into a pool of bs-row blocks in a random order, noise blocks
    between them: (k_pool, v_pool [nblk, Hkv, bs, d] codes, table [B, nb + 2], nblk)."""
    B, Hkv, L, d = kc.shape
    nb = (L + bs - 1) // bs
    total = B * nb + 3
    perm = torch.randperm(total, generator=gen)
    noise = lambda: torch.randint(0, 120, (total, Hkv, bs, d), generator=gen).to(torch.uint8)
    kp, vp = noise(), noise()
    table = torch.full((B, nb + 2), -7, dtype=torch.int32)
    for b in range(B):
        for j in range(nb):
            blk = int(perm[b * nb + j])
            table[b, j] = blk
            t0, t1 = j * bs, min(L, (j + 1) * bs)
            kp[blk, :, : t1 - t0] = kc[b, :, t0:t1].view(torch.uint8)
            vp[blk, :, : t1 - t0] = vc[b, :, t0:t1].view(torch.uint8)
    return kp, vp, table, total


@pytest.mark.parametrize("case", ["dense", "sparse", "paged_bs16", "sparse_paged_bs64", "g3", "ragged",
                                  "bf16_out", "headline_sampled", "rows128", "rows132", "empty_context"])
def test_fp8_cache_matches_oracle(ops, case):
    """An E4M3 cache with a scale per (sequence, KV head) against the fp8 oracle on the same codes
    and scales (the oracle is pinned to the bf16 one on the numbers the codes stand for). rows128 /
    rows132: 128 and 132 query rows per KV head on the tensor-core kernel (alternate tiles of one
    128-row block, then both pipes with a 4-row second block); empty_context: a sequence with no
    cache token at all."""
    if case == "headline_sampled":
        w = W.workload(2)
        x = W.make_inputs(w)
        B, N, Hq, L = w.B, w.N, w.Hq, w.L
    elif case in ("rows128", "rows132"):
        Hq, Hkv = 8, 2
        B, N, L = 2, (32 if case == "rows128" else 33), 900
        x = small(350 + N, B=B, N=N, Hq=Hq, Hkv=Hkv, L=L, depth=6)
    else:
        Hq, Hkv = (12, 4) if case == "g3" else (8, 2)
        B, N, L = 2, 6, 1000
        x = small(300 + len(case), B=B, N=N, Hq=Hq, Hkv=Hkv, L=L)
    kc, ks = quantize_e4m3(x["k_cache"])
    vc, vs = quantize_e4m3(x["v_cache"])
    g = to_dev(x)
    kw, okw = {}, {}
    rows = sample_rows(B, N, Hq, 384, seed=7) if case == "headline_sampled" else None
    if "sparse" in case:
        ds, ts = W.random_scores(B, L, seed=11)
        idx, _, _ = oracle.select(ds, ts, sink=4, window=16, top_m=64, budget=256)
        kw["idx"] = torch.from_numpy(idx).to(dev())
        okw["idx"] = torch.from_numpy(idx)
    if case in ("ragged", "empty_context"):
        cl = torch.tensor([L, 357] if case == "ragged" else [0, L], dtype=torch.int32)
        kw["ctx_lens"] = cl.to(dev())
        okw["ctx_lens"] = cl
    dk, dv = kc.to(dev()), vc.to(dev())
    if "paged" in case:
        bs = int(case.split("_bs")[1])
        kp, vp, table, nblk = codes_to_pool(kc, vc, bs, torch.Generator().manual_seed(bs))
        dk, dv = kp[:nblk].to(dev()), vp[:nblk].to(dev())
        kw.update(block_table=table.to(dev()), L=L)
    out_dtype = torch.bfloat16 if case == "bf16_out" else torch.float32
    out, lse = ops.verify_attn_ex(g["q"], dk, dv, g["k_draft"], g["v_draft"], g["parent"], scale=x["scale"],
                                  k_scale=ks.to(dev()), v_scale=vs.to(dev()), out_dtype=out_dtype, **kw)
    ro, rl, st = oracle.attend_fp8(x["q"], kc, vc, ks, vs, x["k_draft"], x["v_draft"], x["parent"],
                                   scale=x["scale"], rows=rows, **okw)
    assert st == 0
    torch.cuda.synchronize()
    if case == "bf16_out":
        o = out.float().cpu().numpy().reshape(ro.shape)
        assert np.abs(o - ro).max() <= ATOL_O + np.abs(ro).max() * 2.0 ** -8
    else:
        assert_attn_close(out, lse, ro, rl, rows)


@pytest.mark.parametrize("path", ["tcgen05", "portable"])
def test_fp8_every_code_converts_exactly(ops, path):
    """Caches drawn uniformly from the 254 finite E4M3 codes (zeros of both signs, every
    subnormal, the largest numbers) on the tensor-core kernel (G = 4) and on the warp-level one
    (G = 3): both convert the codes to bf16 without error, so the result is the oracle's."""
    Hq, Hkv = (8, 2) if path == "tcgen05" else (12, 4)
    B, N, L = 2, 6, 700
    x = small(41 if path == "tcgen05" else 43, B=B, N=N, Hq=Hq, Hkv=Hkv, L=L)
    gen = torch.Generator().manual_seed(17)
    finite = torch.tensor([c for c in range(256) if c & 0x7F != 0x7F], dtype=torch.uint8)
    pick = lambda: finite[torch.randint(0, len(finite), (B, Hkv, L, 128), generator=gen)].view(torch.float8_e4m3fn)
    kc, vc = pick(), pick()
    ks = torch.full((B, Hkv), 1.0 / (448 * 8), dtype=torch.float32)
    vs = (torch.rand(B, Hkv, generator=gen) + 0.5).float() / 448
    g = to_dev(x)
    out, lse = ops.verify_attn_ex(g["q"], kc.to(dev()), vc.to(dev()), g["k_draft"], g["v_draft"], g["parent"],
                                  scale=x["scale"], k_scale=ks.to(dev()), v_scale=vs.to(dev()))
    ro, rl, st = oracle.attend_fp8(x["q"], kc, vc, ks, vs, x["k_draft"], x["v_draft"], x["parent"], scale=x["scale"])
    assert st == 0
    torch.cuda.synchronize()
    assert_attn_close(out, lse, ro, rl)


@pytest.mark.parametrize("path", ["tcgen05", "portable"])
def test_fp8_nan_code_in_v_gives_nan_columns(ops, path):
    """A NaN code in V (0x7F or 0xFF) is a NaN in the output column it sits in, for every query
    row of that KV head, as in the oracle; everything else is unchanged."""
    Hq, Hkv = (8, 2) if path == "tcgen05" else (12, 4)
    B, N, L = 2, 4, 600
    x = small(47, B=B, N=N, Hq=Hq, Hkv=Hkv, L=L)
    kc, ks = quantize_e4m3(x["k_cache"])
    vc, vs = quantize_e4m3(x["v_cache"])
    vb = vc.view(torch.uint8).clone()
    vb[0, 1, 500, 7] = 0x7F
    vb[1, 0, 3, 100] = 0xFF
    vc = vb.view(torch.float8_e4m3fn)
    g = to_dev(x)
    out, lse = ops.verify_attn_ex(g["q"], kc.to(dev()), vc.to(dev()), g["k_draft"], g["v_draft"], g["parent"],
                                  scale=x["scale"], k_scale=ks.to(dev()), v_scale=vs.to(dev()))
    ro, rl, st = oracle.attend_fp8(x["q"], kc, vc, ks, vs, x["k_draft"], x["v_draft"], x["parent"], scale=x["scale"])
    torch.cuda.synchronize()
    o = out.cpu().numpy().reshape(ro.shape)
    nan = np.isnan(ro)
    assert nan.any() and np.array_equal(np.isnan(o), nan)
    assert np.abs(o[~nan] - ro[~nan]).max() <= ATOL_O
    assert np.all(np.isfinite(lse.cpu().numpy())) and np.abs(lse.cpu().numpy().reshape(-1) - rl).max() <= ATOL_L


def test_importance_scores_headline_shape(ops):
    """The headline layer (B=4, L=32k, N=64 tree) scored on two heads of different KV heads,
    against the oracle on a sample of tokens of every sequence (all draft queries of each)."""
    w = W.workload(2)
    x = W.make_inputs(w)
    g = to_dev(x)
    # both sides take the attention oracle's lse (every row), rounded to fp32
    _, lse64, st = oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                                 scale=x["scale"])
    assert st == 0
    lse32 = lse64.astype(np.float32).reshape(w.B, w.N, w.Hq)
    heads = [3, 17]
    score, status = ops.importance_scores(g["q"], g["k_cache"], torch.from_numpy(lse32).to(dev()),
                                          torch.tensor(heads, dtype=torch.int32, device=dev()), scale=x["scale"])
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    lse32 = lse32.astype(np.float64)
    toks = np.sort(np.random.default_rng(1).choice(w.L, 300, replace=False))
    kc = x["k_cache"][:, :, toks].float().numpy()
    want = oracle.importance_scores(x["q"].float().numpy(), kc, lse32, heads, scale=float(np.float32(x["scale"])))
    got = score.cpu().numpy()[:, toks]
    assert np.allclose(got, want, rtol=1e-4, atol=1e-7), np.abs(got - want).max()
