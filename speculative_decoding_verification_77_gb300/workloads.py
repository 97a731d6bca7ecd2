"""Seeded synthetic inputs for verification attention.

This module only draws inputs. It holds none of the verification arithmetic
(no attention, no selection, no merge), so both the CUDA path and the CPU
oracle can take their inputs from it without sharing any computation.

Input recipe (all draws on the CPU, in this order, from one
``torch.Generator`` seeded per workload):

1. Q ``[B, N, Hq, d]``             fp32 N(0,1), rounded to bf16 (RNE)
2. K cache ``[B, Hkv, L, d]``      fp32 N(0,1) drawn one sequence ``b`` at a time, rounded to bf16
3. V cache ``[B, Hkv, L, d]``      same
4. K draft ``[B, N, Hkv, d]``      fp32 N(0,1), rounded to bf16
5. V draft ``[B, N, Hkv, d]``      same
6. the parent array (random trees only), one tree per sequence
7. importance scores (sparse workloads only): z_draft then z_target, each
   ``[B, L]`` N(0,1); the score is softmax(4 z) along L in fp32.

Draft trees follow the shapes the pages use:

* chain (a causal block of draft tokens);
* random tree with bounded depth (the parent of node i is uniform over the
  earlier nodes whose depth is below the bound);
* best-first prefix tree built from per-position draft marginals, as in
  BASTION "Metodologia" section 1-2: the path score of node i is the product of
  the marginals along its root path, and the tree grows by repeatedly adding the
  candidate with the highest path score (the expansion the page proves optimal
  for the acceptance surrogate sum of path scores).

Tree convention: ``parent[i] == -1`` means node i is a child of the last cache
token (depth 1); otherwise ``0 <= parent[i] < i``.
"""

from __future__ import annotations

import heapq
from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    """One verification workload: shapes, tree kind and the selection budget."""

    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    N: int
    tree: str  # "chain" | "random" | "best_first"
    depth_max: int = 0  # for "random"
    seed: int = 0
    sparse: bool = False
    sink: int = 0
    window: int = 0
    top_m: int = 0
    budget: int = 0
    d: int = HEAD_DIM
    # best-first marginals: block length and candidates per position
    bf_block: int = 16
    bf_cands: int = 10
    bf_alpha: float = 0.3

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def kv_bytes(self) -> int:
        """K and V cache bytes the cache part must read (bf16)."""
        t = self.budget if self.sparse else self.L
        return 2 * self.B * self.Hkv * t * self.d * 2

    def flops(self) -> int:
        """QK^T + PV flops of the cache part."""
        t = self.budget if self.sparse else self.L
        return 4 * self.B * self.Hq * self.N * t * self.d


def workload(cfg: int, N: int | None = None) -> Workload:
    """The five synthetic workloads, by number (1..5).

    1 tiny dense chain; 2 Llama-3-8B-shaped layer at L=32k (the headline);
    3 sparse hybrid at L=32k, k=2048; 4 Qwen2.5-72B-shaped layer at L=128k;
    5 tree-size sweep at L=16k (N in {1, 4, 16, 64, 256}).
    """
    if cfg == 1:
        return Workload("tiny-dense-B1-L2k-N8-chain", B=1, L=2048, Hq=8, Hkv=2, N=8,
                        tree="chain", seed=1000)
    if cfg == 2:
        return Workload("llama3-8b-layer-B4-L32k-N64-tree", B=4, L=32768, Hq=32, Hkv=8, N=64,
                        tree="random", depth_max=8, seed=2000)
    if cfg == 3:
        return Workload("sparse-hybrid-B16-L32k-k2048-N8-chain", B=16, L=32768, Hq=32, Hkv=8,
                        N=8, tree="chain", seed=3000, sparse=True, sink=4, window=64,
                        top_m=512, budget=2048)
    if cfg == 4:
        return Workload("qwen2.5-72b-layer-B8-L128k-N32-tree", B=8, L=131072, Hq=64, Hkv=8,
                        N=32, tree="random", depth_max=6, seed=4000)
    if cfg == 5:
        n = 64 if N is None else N
        return Workload(f"tree-sweep-B8-L16k-N{n}-best-first", B=8, L=16384, Hq=32, Hkv=8,
                        N=n, tree="best_first", seed=5000 + n)
    raise ValueError(f"unknown workload {cfg}")


# ---------------------------------------------------------------------------
# trees


def chain_parents(N: int) -> list[int]:
    """Chain: node i's parent is i-1; node 0 hangs off the cache."""
    return [-1] + list(range(N - 1))


def random_parents(N: int, depth_max: int, gen: torch.Generator) -> list[int]:
    """Random tree: parent of node i uniform over earlier nodes j with depth(j) < depth_max."""
    parents = [-1]
    depth = [1]
    for i in range(1, N):
        cands = [j for j in range(i) if depth[j] < depth_max]
        if not cands:  # depth_max == 1: every node is a root
            parents.append(-1)
            depth.append(1)
            continue
        pick = int(torch.randint(len(cands), (1,), generator=gen).item())
        j = cands[pick]
        parents.append(j)
        depth.append(depth[j] + 1)
    return parents


@dataclass
class BestFirstTree:
    parents: list[int]
    depth: list[int]  # 1-based depth of each node
    cand: list[int]  # candidate (rank within its position's marginal) of each node
    rho: list[float]  # path score of each node
    marginals: np.ndarray = field(repr=False)  # [block, cands], sorted descending


def best_first_tree(marginals: np.ndarray, N: int) -> BestFirstTree:
    """Grow a prefix tree best-first from per-position marginals q_k.

    ``marginals[k, c]`` is the drafter's probability of candidate c at depth k+1.
    The path score of a node at depth d reached through candidates
    (c_1..c_d) is prod_k marginals[k-1, c_k] (BASTION "Metodologia" section 1,
    path score). The frontier is a max-heap on (path score desc, insertion
    order asc); each pop adds one node, and pushes that node's children at
    the next position. Node ids follow pop order, so parent[i] < i.
    """
    block, ncand = marginals.shape
    heap: list[tuple[float, int, int, int, float]] = []
    counter = 0
    for c in range(ncand):
        r = float(marginals[0, c])
        heapq.heappush(heap, (-r, counter, -1, 0, c))
        counter += 1
    t = BestFirstTree([], [], [], [], marginals)
    while len(t.parents) < N and heap:
        neg_r, _, par, k, c = heapq.heappop(heap)
        node = len(t.parents)
        t.parents.append(par)
        t.depth.append(k + 1)
        t.cand.append(c)
        t.rho.append(-neg_r)
        if k + 1 < block:
            for c2 in range(ncand):
                r2 = (-neg_r) * float(marginals[k + 1, c2])
                heapq.heappush(heap, (-r2, counter, node, k + 1, c2))
                counter += 1
    return t


def dirichlet_marginals(rng: np.random.Generator, block: int, ncand: int, alpha: float) -> np.ndarray:
    """Synthetic block-diffusion marginals: per position a Dirichlet(alpha) draw, sorted descending."""
    q = rng.dirichlet(np.full(ncand, alpha), size=block)
    return -np.sort(-q, axis=1)


# ---------------------------------------------------------------------------
# tensors


def _randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_inputs(w: Workload, *, seed: int | None = None, kv_tokens: int | None = None) -> dict:
    """Draw every input of workload ``w`` on the CPU (see the module docstring).

    Returns a dict of CPU tensors: q, k_cache, v_cache, k_draft, v_draft,
    parent (int32 [B, N]), ctx_lens (int32 [B]) and, for sparse workloads,
    draft_score / target_score (fp32 [B, L]) plus the selection arguments.
    ``kv_tokens`` overrides L (used to draw smaller variants of a workload).
    """
    s = w.seed if seed is None else seed
    g = torch.Generator().manual_seed(s)
    B, N, Hq, Hkv, d = w.B, w.N, w.Hq, w.Hkv, w.d
    L = w.L if kv_tokens is None else kv_tokens
    out: dict = {"workload": w, "L": L}
    out["q"] = _randn_bf16((B, N, Hq, d), g)
    out["k_cache"] = torch.stack([_randn_bf16((Hkv, L, d), g) for _ in range(B)])
    out["v_cache"] = torch.stack([_randn_bf16((Hkv, L, d), g) for _ in range(B)])
    out["k_draft"] = _randn_bf16((B, N, Hkv, d), g)
    out["v_draft"] = _randn_bf16((B, N, Hkv, d), g)
    parents = []
    if w.tree == "chain":
        parents = [chain_parents(N) for _ in range(B)]
    elif w.tree == "random":
        parents = [random_parents(N, w.depth_max, g) for _ in range(B)]
    elif w.tree == "best_first":
        rng = np.random.default_rng(s)
        trees = [best_first_tree(dirichlet_marginals(rng, w.bf_block, w.bf_cands, w.bf_alpha), N)
                 for _ in range(B)]
        out["trees"] = trees
        parents = [t.parents for t in trees]
    else:
        raise ValueError(w.tree)
    out["parent"] = torch.tensor(parents, dtype=torch.int32)
    out["ctx_lens"] = torch.full((B,), L, dtype=torch.int32)
    out["scale"] = float(1.0 / np.sqrt(d))
    if w.sparse:
        zd = torch.randn((B, L), generator=g, dtype=torch.float32)
        zt = torch.randn((B, L), generator=g, dtype=torch.float32)
        out["draft_score"] = torch.softmax(4.0 * zd, dim=-1)
        out["target_score"] = torch.softmax(4.0 * zt, dim=-1)
        out.update(sink=w.sink, window=w.window, top_m=w.top_m, budget=w.budget)
    return out


def random_scores(B: int, L: int, seed: int, *, ties: int = 0) -> tuple[torch.Tensor, torch.Tensor]:
    """Importance scores for selection cases: softmax(4 z) per row.

    With ``ties > 0`` the scores are quantised to ``ties`` levels so that many
    entries compare equal (exercises the lower-index tie rule).
    """
    g = torch.Generator().manual_seed(seed)
    zd = torch.randn((B, L), generator=g, dtype=torch.float32)
    zt = torch.randn((B, L), generator=g, dtype=torch.float32)
    if ties > 0:
        zd = torch.floor(zd * ties / 4.0)
        zt = torch.floor(zt * ties / 4.0)
    return torch.softmax(4.0 * zd, dim=-1), torch.softmax(4.0 * zt, dim=-1)
