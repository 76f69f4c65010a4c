"""Seeded synthetic draft-tree workloads for TreeWY verification of Gated DeltaNet.

This module holds only tree shapes and random draws.  It holds none of the
method's arithmetic (no decay products, no Gram matrices, no state updates), so
that the CPU oracle and the CUDA path can both consume its output without
sharing any computation.

Shapes follow the pages' workloads:

* draft chains of an MTP drafter (TreeWY: Speculative Verification for Gated
  DeltaNet Hybrids, §5 "Setup": depth-3 MTP chain);
* ``draft_tree_widths`` trees, one branching factor per depth level, with the
  first level hanging off the committed state, laid out in DFS pre-order
  (same paper, §4 and Table 2: (3,3,3) gives N = 3 + 9 + 27 = 39);
* per-head sizes dk = dv = 128 with 32 or 64 value heads (same paper, §2 "The
  memory problem": Qwen3.5 35B-A3B and 397B-A17B GDN layers).

Layout of every generated batch (T = total draft nodes over all requests):

* ``node_offset`` int32 [R+1]: request r owns node rows node_offset[r] ..
  node_offset[r+1]-1;
* ``parent`` int32 [T]: parent of each node as a request-local index, -1 for a
  node that hangs off the committed state S0; parents precede children;
* ``q``, ``k`` [T][H][dk], ``v`` [T][H][dv] in bf16 (or fp32), q and k
  L2-normalised in fp32 before rounding;
* ``alpha``, ``beta`` fp32 [T][H];
* ``state`` fp32 [num_slots][H][dv][dk] (dk contiguous), ``state_slot`` int32
  [R] mapping a request to its pool slot;
* ``accepted`` int32 [R]: request-local index of the accepted node, -1 when
  no draft token is accepted.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

MAX_NODES = 64


# --------------------------------------------------------------------------
# Tree shapes (parent arrays, request-local indices, DFS pre-order)
# --------------------------------------------------------------------------

def chain_parents(n: int) -> np.ndarray:
    """A linear draft chain of n nodes: node 0 hangs off S0, node i off i-1."""
    return np.arange(-1, n - 1, dtype=np.int32)


def width_tree_parents(widths: Sequence[int]) -> np.ndarray:
    """Full tree with branching factor widths[l] at depth l, in DFS pre-order.

    The first level has widths[0] nodes that all hang off the committed state,
    so N = sum_l prod_{j<=l} widths[j] (TreeWY paper, §4 and Table 2).
    """
    parents: List[int] = []

    def expand(par: int, level: int) -> None:
        if level == len(widths):
            return
        for _ in range(widths[level]):
            me = len(parents)
            parents.append(par)
            expand(me, level + 1)

    expand(-1, 0)
    return np.asarray(parents, dtype=np.int32)


def complete_binary_parents(depth: int) -> np.ndarray:
    """Complete binary tree of the given depth with a single root, DFS pre-order.

    depth 4 gives 1 + 2 + 4 + 8 = 15 nodes.
    """
    parents: List[int] = []

    def expand(par: int, level: int) -> None:
        me = len(parents)
        parents.append(par)
        if level + 1 < depth:
            expand(me, level + 1)
            expand(me, level + 1)

    expand(-1, 0)
    return np.asarray(parents, dtype=np.int32)


def branches_parents(n_branches: int, branch_len: int) -> np.ndarray:
    """n_branches independent chains of branch_len nodes, all off S0."""
    parents = []
    for b in range(n_branches):
        base = b * branch_len
        parents.append(-1)
        parents.extend(range(base, base + branch_len - 1))
    return np.asarray(parents, dtype=np.int32)


def random_recursive_parents(rng: np.random.Generator, n: int, max_depth: int) -> np.ndarray:
    """Random tree: node 0 hangs off S0; node i>0 picks its parent uniformly
    among earlier nodes whose depth is below max_depth (node 0 has depth 1)."""
    parents = np.empty(n, dtype=np.int32)
    depth = np.empty(n, dtype=np.int64)
    parents[0] = -1
    depth[0] = 1
    for i in range(1, n):
        cand = np.nonzero(depth[:i] < max_depth)[0]
        p = int(cand[rng.integers(0, cand.size)])
        parents[i] = p
        depth[i] = depth[p] + 1
    return parents


def tree_depths(parents: np.ndarray) -> np.ndarray:
    """Depth of every node (a node hanging off S0 has depth 1)."""
    depth = np.zeros(len(parents), dtype=np.int64)
    for i, p in enumerate(parents):
        depth[i] = 1 if p < 0 else depth[p] + 1
    return depth


# --------------------------------------------------------------------------
# Workload configurations
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    R: int
    H: int
    dk: int
    dv: int
    qkv_dtype: str          # "bf16" or "f32"
    tree: str               # "chain4", "binary15", "random16_64_d8", "random64_d8", "branches8x8", "widths"
    s0_std: float
    alpha_range: Tuple[float, float]
    beta: Tuple             # ("sigmoid",) or ("uniform", lo, hi)
    accepted: str           # "fixed1", "prefix", "uniform"
    seed: int
    layers: int = 1
    widths: Tuple[int, ...] = ()

    def with_(self, **kw) -> "WorkloadConfig":
        return dataclasses.replace(self, **kw)


CONFIGS: Dict[str, WorkloadConfig] = {
    # 1 request, 1 head, dk=dv=16, fp32 everything, chain 0->1->2->3, first
    # two nodes accepted.
    "tiny": WorkloadConfig("tiny", 1, 1, 16, 16, "f32", "chain4", 0.1, (0.9, 0.999),
                           ("uniform", 0.1, 0.9), "fixed1", seed=0),
    # MTP-style chain of 4, accepted prefix length uniform in 0..4.
    "chain": WorkloadConfig("chain", 64, 32, 128, 128, "bf16", "chain4", 0.05, (0.9, 0.999),
                            ("sigmoid",), "prefix", seed=2),
    # complete binary tree of depth 4 (N = 15), accepted node uniform.
    "binary": WorkloadConfig("binary", 128, 32, 128, 128, "bf16", "binary15", 0.05, (0.9, 0.999),
                             ("sigmoid",), "uniform", seed=3),
    # wide ragged random trees, N uniform in 16..64, depth <= 8, 30 GDN layers.
    "wide": WorkloadConfig("wide", 256, 32, 128, 128, "bf16", "random16_64_d8", 0.05, (0.9, 0.999),
                           ("sigmoid",), "uniform", seed=4, layers=30),
    # 8 branches of depth 8 sharing the committed root (N = 64), 64 heads.
    "stress": WorkloadConfig("stress", 512, 64, 128, 128, "bf16", "branches8x8", 0.05, (0.8, 0.999),
                             ("uniform", 0.05, 0.95), "uniform", seed=5),
}


def make_trees(cfg: WorkloadConfig, R: Optional[int] = None) -> Tuple[List[np.ndarray], np.ndarray]:
    """Per-request parent arrays and accepted node indices (seeded numpy PCG64)."""
    R = cfg.R if R is None else R
    rng = np.random.default_rng(cfg.seed)
    trees: List[np.ndarray] = []
    for _ in range(R):
        if cfg.tree == "chain4":
            trees.append(chain_parents(4))
        elif cfg.tree == "binary15":
            trees.append(complete_binary_parents(4))
        elif cfg.tree == "random16_64_d8":
            n = int(rng.integers(16, 65))
            trees.append(random_recursive_parents(rng, n, 8))
        elif cfg.tree == "random64_d8":
            trees.append(random_recursive_parents(rng, 64, 8))
        elif cfg.tree == "branches8x8":
            trees.append(branches_parents(8, 8))
        elif cfg.tree == "widths":
            trees.append(width_tree_parents(cfg.widths))
        else:
            raise ValueError(f"unknown tree kind {cfg.tree}")
    accepted = np.empty(R, dtype=np.int32)
    for r, par in enumerate(trees):
        n = len(par)
        if cfg.accepted == "fixed1":
            accepted[r] = min(1, n - 1)
        elif cfg.accepted == "prefix":
            accepted[r] = int(rng.integers(0, n + 1)) - 1
        elif cfg.accepted == "uniform":
            accepted[r] = int(rng.integers(0, n)) if n > 0 else -1
        else:
            raise ValueError(f"unknown accepted rule {cfg.accepted}")
    return trees, accepted


@dataclass
class Workload:
    """One layer's worth of synthetic inputs (torch tensors on one device)."""
    R: int
    H: int
    dk: int
    dv: int
    T: int
    max_nodes: int
    qkv_dtype: str
    trees: List[np.ndarray]
    node_offset: torch.Tensor
    parent: torch.Tensor
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    alpha: torch.Tensor
    beta: torch.Tensor
    state: torch.Tensor
    state_slot: torch.Tensor
    accepted: torch.Tensor

    @property
    def num_slots(self) -> int:
        return int(self.state.shape[0])

    def to(self, device) -> "Workload":
        kw = {}
        for f in dataclasses.fields(self):
            val = getattr(self, f.name)
            kw[f.name] = val.to(device) if isinstance(val, torch.Tensor) else val
        return Workload(**kw)

    def request_state(self, r: int) -> torch.Tensor:
        """The committed state block [H][dv][dk] of request r."""
        return self.state[int(self.state_slot[r])]


def assemble(trees: Sequence[np.ndarray], accepted: np.ndarray, H: int, dk: int, dv: int,
             qkv_dtype: str, s0_std: float, alpha_range: Tuple[float, float], beta: Tuple,
             seed: int, device="cpu", max_nodes: Optional[int] = None,
             extra_slots: int = 0, state_dtype: str = "f32") -> Workload:
    """Draw the per-node and per-head tensors for the given trees.

    Draw order (one torch generator seeded with ``seed``): slot permutation,
    S0, q, k, v, alpha, beta.  q and k are drawn N(0,1) in fp32 and divided by
    their L2 norm (no epsilon) before rounding to the qkv dtype (round to
    nearest even); beta of kind "sigmoid" is sigmoid(N(0,1)) evaluated in fp64
    and rounded to fp32.  A bf16 state pool (``state_dtype="bf16"``) is the
    same fp32 draw rounded to nearest even bf16.
    """
    R = len(trees)
    sizes = np.array([len(t) for t in trees], dtype=np.int64)
    T = int(sizes.sum())
    node_offset = np.zeros(R + 1, dtype=np.int32)
    node_offset[1:] = np.cumsum(sizes)
    parent = np.concatenate(trees).astype(np.int32) if T else np.zeros(0, np.int32)
    if max_nodes is None:
        max_nodes = int(sizes.max()) if R else 1
        max_nodes = max(max_nodes, 1)

    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    num_slots = R + extra_slots
    perm = torch.randperm(num_slots, generator=g, device=dev)[:R].to(torch.int32)

    state = torch.randn(num_slots, H, dv, dk, generator=g, device=dev, dtype=torch.float32) * s0_std
    if state_dtype == "bf16":
        state = state.to(torch.bfloat16)
    elif state_dtype != "f32":
        raise ValueError(f"state_dtype {state_dtype!r} is not 'f32' or 'bf16'")

    def unit(shape):
        x = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
        return x / x.norm(dim=-1, keepdim=True)

    tdt = torch.bfloat16 if qkv_dtype == "bf16" else torch.float32
    q = unit((T, H, dk)).to(tdt)
    k = unit((T, H, dk)).to(tdt)
    v = torch.randn(T, H, dv, generator=g, device=dev, dtype=torch.float32).to(tdt)
    lo, hi = alpha_range
    alpha = (torch.rand(T, H, generator=g, device=dev, dtype=torch.float32) * (hi - lo) + lo)
    if beta[0] == "sigmoid":
        b = torch.sigmoid(torch.randn(T, H, generator=g, device=dev, dtype=torch.float64)).to(torch.float32)
    elif beta[0] == "uniform":
        b = torch.rand(T, H, generator=g, device=dev, dtype=torch.float32) * (beta[2] - beta[1]) + beta[1]
    elif beta[0] == "const":
        b = torch.full((T, H), float(beta[1]), device=dev, dtype=torch.float32)
    else:
        raise ValueError(beta)
    # alpha and beta must lie in (0, 1); rounding of the affine map can touch
    # an end point only with negligible probability, but clamp for safety.
    alpha = alpha.clamp(min=float(np.nextafter(np.float32(0), np.float32(1))),
                        max=float(np.nextafter(np.float32(1), np.float32(0))))
    return Workload(
        R=R, H=H, dk=dk, dv=dv, T=T, max_nodes=int(max_nodes), qkv_dtype=qkv_dtype,
        trees=[np.asarray(t, dtype=np.int32) for t in trees],
        node_offset=torch.from_numpy(node_offset).to(dev),
        parent=torch.from_numpy(parent).to(dev),
        q=q, k=k, v=v, alpha=alpha, beta=b, state=state, state_slot=perm,
        accepted=torch.from_numpy(np.asarray(accepted, dtype=np.int32)).to(dev),
    )


def generate(cfg: WorkloadConfig, R: Optional[int] = None, layer: int = 0, device="cpu",
             extra_slots: int = 0, state_dtype: str = "f32") -> Workload:
    """Seeded inputs for one GDN layer of a configuration (optionally fewer requests).

    Trees and accepted nodes depend only on (cfg.seed, R); tensors use the
    seed ``cfg.seed * 1000 + layer`` so every layer of a step draws fresh data.
    """
    trees, accepted = make_trees(cfg, R)
    return assemble(trees, accepted, cfg.H, cfg.dk, cfg.dv, cfg.qkv_dtype, cfg.s0_std,
                    cfg.alpha_range, cfg.beta, seed=cfg.seed * 1000 + layer, device=device,
                    extra_slots=extra_slots, state_dtype=state_dtype)


def as_float64(x: torch.Tensor) -> np.ndarray:
    """Exact widening of a (bf16 or fp32) tensor to a float64 numpy array."""
    return x.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)
