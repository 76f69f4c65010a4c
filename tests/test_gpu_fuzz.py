"""Randomised GPU parity: every seed draws a batch shape (requests, heads,
head sizes, q/k/v and state dtypes, tree capacity, tree shapes including
chains, stars, deep paths and empty trees, accepted nodes) and runs verify +
commit and the two-round fused path through the C ABI against the oracle.

Tolerances as in tests/gpu_helpers.py (o, U: 2e-3 of the largest reference
value; state: 1e-3 of the largest reference value) plus, for a bf16 pool,
the per-element rounding bound 2^-8 |S| of the stored state.
"""
import numpy as np
import pytest
import torch

from gdn_speculative_tree_gb300 import binding
from gdn_speculative_tree_gb300 import workloads as wl
from oracle import gdn_tree_oracle as orc
from tests.gpu_helpers import np32

pytestmark = pytest.mark.gpu

SHAPES = [(128, 128, "bf16"), (128, 128, "f32"), (64, 64, "bf16"), (32, 96, "bf16"), (5, 7, "f32")]


def draw_tree(rng, cap):
    kind = rng.integers(0, 6)
    n = int(rng.integers(0, cap + 1))
    if kind == 0 or n == 0:
        return np.zeros(0, np.int32)                         # an empty tree
    if kind == 1:
        return wl.chain_parents(n)
    if kind == 2:
        return np.full(n, -1, np.int32)                     # all nodes on S0
    if kind == 3:
        return np.array([-1] + [0] * (n - 1), np.int32)     # a star under node 0
    return np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32)


def draw_batch(seed, caps=(16, 32, 64)):
    rng = np.random.default_rng(1000 + seed)
    dk, dv, qkv = SHAPES[int(rng.integers(0, len(SHAPES)))]
    sd = "bf16" if rng.integers(0, 2) else "f32"
    cap = int(rng.choice(list(caps)))
    R = int(rng.integers(1, 9))
    H = int(rng.integers(1, 4))
    trees = [draw_tree(rng, cap) for _ in range(R)]
    acc = [int(rng.integers(-1, len(t))) if len(t) else -1 for t in trees]
    return rng, dict(H=H, dk=dk, dv=dv, qkv=qkv, sd=sd, cap=cap, trees=trees, acc=acc)


def assemble(p, trees, acc, seed):
    return wl.assemble(trees, np.asarray(acc, np.int32), p["H"], p["dk"], p["dv"], p["qkv"], 0.05,
                       (0.85, 0.999), ("uniform", 0.05, 0.95), seed=seed, max_nodes=p["cap"],
                       extra_slots=1, state_dtype=p["sd"]).to("cuda")


def f64(x):
    return np32(x).astype(np.float64)


def check_state(S_gpu, S_ref, sd):
    bound = 1e-3 * np.abs(S_ref).max() + (2.0 ** -8 * np.abs(S_ref) if sd == "bf16" else 0.0)
    assert np.all(np.abs(S_gpu - S_ref) <= bound + 1e-30)


SMALL_CAPS = (4, 8)  # the small-tree kernel's capacities (dk = dv = 128, bf16 q/k/v)
MID_CAPS = (9, 12, 16)  # the warp-MMA kernel's range below the tcgen05 kernel's


def seeded(seed, base_small, base_mid, base):
    """Batch parameters for a seed: "small<i>" and "mid<i>" draw capacities of
    the small-tree and warp-MMA kernels, integers the general mix."""
    if isinstance(seed, str):
        kind, i = ("small", int(seed[5:])) if seed.startswith("small") else ("mid", int(seed[3:]))
        s2 = (base_small if kind == "small" else base_mid) + i
        rng, p = draw_batch(s2, caps=SMALL_CAPS if kind == "small" else MID_CAPS)
        return rng, p, s2
    rng, p = draw_batch(base + seed)
    return rng, p, seed


@pytest.mark.parametrize("seed", list(range(48)) + [f"small{i}" for i in range(24)] +
                         [f"mid{i}" for i in range(16)])
def test_fuzz_verify_commit(cuda_lib, seed):
    _, p, seed = seeded(seed, 3000, 5000, 0)
    w = assemble(p, p["trees"], p["acc"], seed)
    S0_pool = w.state.cpu()
    tv = binding.TreeVerifier(w)
    tv.verify()
    tv.commit()
    torch.cuda.synchronize()
    assert not tv.status.any(), (p, tv.status.tolist())
    o, U = np32(tv.o), np32(tv.U)
    node = w.node_offset.cpu().numpy()
    o_err = o_max = u_err = u_max = 0.0
    for r in range(w.R):
        lo, hi = int(node[r]), int(node[r + 1])
        slot = int(w.state_slot[r])
        S0 = f64(S0_pool[slot])
        ref = orc.verify_request(S0, w.parent[lo:hi].cpu().numpy(), f64(w.q[lo:hi]), f64(w.k[lo:hi]),
                                 f64(w.v[lo:hi]), f64(w.alpha[lo:hi]), f64(w.beta[lo:hi]))
        if hi > lo:
            o_err = max(o_err, float(np.abs(o[lo:hi] - ref.o).max()))
            o_max = max(o_max, float(np.abs(ref.o).max()))
            u_err = max(u_err, float(np.abs(U[lo:hi] - ref.U).max()))
            u_max = max(u_max, float(np.abs(ref.U).max()))
        S_ref = orc.commit_request(S0, ref, p["acc"][r])
        check_state(f64(w.state[slot]), S_ref, p["sd"])
    assert o_err <= 2e-3 * max(o_max, 1e-30), (p["dk"], p["dv"], p["qkv"], p["sd"], o_err, o_max)
    assert u_err <= 2e-3 * max(u_max, 1e-30), (u_err, u_max)


@pytest.mark.parametrize("seed", list(range(24)) + [f"small{i}" for i in range(16)] +
                         [f"mid{i}" for i in range(12)])
def test_fuzz_fused_two_rounds(cuda_lib, seed):
    rng, p, seed = seeded(seed, 4000, 6000, 100)
    R = len(p["trees"])
    nxt_trees = [draw_tree(rng, p["cap"]) for _ in range(R)]
    prev = assemble(p, p["trees"], p["acc"], 2 * seed)
    nxt = assemble(p, nxt_trees, [-1] * R, 2 * seed + 1)
    nxt.state = prev.state
    nxt.state_slot = prev.state_slot
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    S0_pool = prev.state.cpu()
    tn = binding.TreeVerifier(nxt)
    binding.treewy_commit_verify(tp.batch, prev.accepted, tn.batch)
    torch.cuda.synchronize()
    assert not tn.status.any() and not tp.status.any()
    o = np32(tn.o)
    pn, nn = prev.node_offset.cpu().numpy(), nxt.node_offset.cpu().numpy()
    o_err = o_max = 0.0
    for r in range(R):
        slot = int(prev.state_slot[r])
        S0 = f64(S0_pool[slot])
        lo, hi = int(pn[r]), int(pn[r + 1])
        ref_p = orc.verify_request(S0, prev.parent[lo:hi].cpu().numpy(), f64(prev.q[lo:hi]),
                                   f64(prev.k[lo:hi]), f64(prev.v[lo:hi]), f64(prev.alpha[lo:hi]),
                                   f64(prev.beta[lo:hi]))
        S_a = orc.commit_request(S0, ref_p, p["acc"][r])
        check_state(f64(prev.state[slot]), S_a, p["sd"])
        S_pool = orc.commit_request(S0, ref_p, p["acc"][r], state_dtype=p["sd"])
        lo, hi = int(nn[r]), int(nn[r + 1])
        if hi == lo:
            continue
        ref = orc.verify_request(S_pool, nxt.parent[lo:hi].cpu().numpy(), f64(nxt.q[lo:hi]),
                                 f64(nxt.k[lo:hi]), f64(nxt.v[lo:hi]), f64(nxt.alpha[lo:hi]),
                                 f64(nxt.beta[lo:hi]))
        o_err = max(o_err, float(np.abs(o[lo:hi] - ref.o).max()))
        o_max = max(o_max, float(np.abs(ref.o).max()))
    assert o_err <= 2e-3 * max(o_max, 1e-30), (p["dk"], p["dv"], p["qkv"], p["sd"], o_err, o_max)


# ------------------------------------------------------------ error reporting

BT, TMN, BA, BS = (binding.STATUS_BAD_TREE, binding.STATUS_TOO_MANY_NODES,
                   binding.STATUS_BAD_ACCEPTED, binding.STATUS_BAD_SLOT)


@pytest.mark.parametrize("flags", [0, binding.FLAG_FORCE_GENERIC])
@pytest.mark.parametrize("seed", range(12))
def test_fuzz_error_reporting(cuda_lib, seed, flags):
    """Requests carrying one planted error each (a parent index out of range,
    a tree above the batch's capacity, a pool slot out of range, an accepted
    index outside the tree) get exactly their status bits and keep their
    outputs and state; every other request matches the oracle."""
    rng = np.random.default_rng(5000 + seed)
    cap = int(rng.choice([4, 8, 16, 32]))
    R = int(rng.integers(4, 10))
    kinds = [int(rng.integers(0, 5)) for _ in range(R)]   # 0 clean, 1 parent, 2 size, 3 slot, 4 accepted
    trees, acc = [], []
    for kind in kinds:
        n = int(rng.integers(cap + 1, 65)) if kind == 2 else int(rng.integers(2, cap + 1))
        t = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32)
        if kind == 1:
            j = int(rng.integers(1, n))
            t[j] = j                                   # a node is its own parent
        trees.append(t)
        acc.append(n if kind == 4 else int(rng.integers(0, n)))
    sd = "bf16" if rng.integers(0, 2) else "f32"
    w = wl.assemble(trees, np.asarray(acc, np.int32), 2, 128, 128, "bf16", 0.05, (0.85, 0.999),
                    ("uniform", 0.05, 0.95), seed=seed, max_nodes=cap, extra_slots=1,
                    state_dtype=sd).to("cuda")
    slots = w.state_slot.clone()
    for r, kind in enumerate(kinds):
        if kind == 3:
            slots[r] = w.num_slots                     # outside the pool
    w.state_slot.copy_(slots)
    S_before = w.state.clone()
    tv = binding.TreeVerifier(w, flags=flags)
    tv.o.fill_(float("nan"))
    tv.U.fill_(float("nan"))
    tv.verify()
    tv.commit()
    torch.cuda.synchronize()
    expect = {0: 0, 1: BT, 2: TMN, 3: BS, 4: BA}
    assert tv.status.cpu().tolist() == [expect[k] for k in kinds], (kinds, tv.status.tolist())
    node = w.node_offset.cpu().numpy()
    o, U = np32(tv.o), np32(tv.U)
    S0_pool = S_before.cpu()
    for r, kind in enumerate(kinds):
        lo, hi = int(node[r]), int(node[r + 1])
        if kind in (1, 2, 3):
            assert np.isnan(o[lo:hi]).all() and np.isnan(U[lo:hi]).all(), (r, kind)
            continue
        slot = int(w.state_slot[r])
        S0 = f64(S0_pool[slot])
        ref = orc.verify_request(S0, w.parent[lo:hi].cpu().numpy(), f64(w.q[lo:hi]), f64(w.k[lo:hi]),
                                 f64(w.v[lo:hi]), f64(w.alpha[lo:hi]), f64(w.beta[lo:hi]))
        assert np.abs(o[lo:hi] - ref.o).max() <= 2e-3 * np.abs(ref.o).max(), (r, kind)
        if kind == 4:
            assert torch.equal(w.state[slot], S_before[slot])  # refused commit
        else:
            check_state(f64(w.state[slot]), orc.commit_request(S0, ref, acc[r]), sd)
    for r, kind in enumerate(kinds):                          # states of refused requests
        if kind in (1, 2):
            s = int(w.state_slot[r])
            assert torch.equal(w.state[s], S_before[s]), (r, kind)
