"""GPU parity of the small-tree verification (batches whose trees have at most
8 nodes: the warp-MMA kernel for dk = dv = 128 with bf16 q/k/v; 4-node and
8-node capacities) against the
oracle on the same seeded inputs: every size from 1 to 8 in chain, star,
forest and random shapes, ragged batches with empty trees, gates at the ends
of their range, a bf16 state pool, the commit-into-verify call, device-side
errors, CUDA-graph replay, and agreement with the tensor-core kernel on the
same inputs.  Tolerances as in gpu_helpers (o, U: 2e-3 of the largest
reference value; committed state 1e-3; gamma 1e-5 relative).
"""
import types

import numpy as np
import pytest
import torch

from gdn_speculative_tree_gb300 import binding
from gdn_speculative_tree_gb300 import workloads as wl
from oracle import gdn_tree_oracle as orc
from tests.gpu_helpers import (CudaRun, FLT_MIN, G_TOL, O_TOL, U_TOL, assert_within, compare, np32,
                               oracle_request)

pytestmark = pytest.mark.gpu

SMALL = 8  # node capacity of the small-tree kernel


def custom(trees, accepted, seed=101, H=3, alpha=(0.9, 0.999), beta=("sigmoid",), max_nodes=None,
           extra_slots=2, state_dtype="f32"):
    w = wl.assemble([np.asarray(t, np.int32) for t in trees], np.asarray(accepted, np.int32), H, 128,
                    128, "bf16", 0.05, alpha, beta, seed=seed, max_nodes=max_nodes,
                    extra_slots=extra_slots, state_dtype=state_dtype)
    return w.to("cuda")


def random_tree(rng, n):
    return np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32) if n else \
        np.zeros(0, np.int32)


def shapes(cap=SMALL):
    """Chains, stars (every node a child of the root), forests (every node a
    root) and two random trees of every size 1..cap."""
    rng = np.random.default_rng(8 + cap)
    trees = []
    for n in range(1, cap + 1):
        trees.append(wl.chain_parents(n))
        trees.append(np.array([-1] + [0] * (n - 1), np.int32))
        trees.append(np.full(n, -1, np.int32))
        trees.append(random_tree(rng, n))
        trees.append(random_tree(rng, n))
    acc = [int(rng.integers(-1, len(t))) for t in trees]
    return trees, acc


@pytest.mark.parametrize("cap", [4, SMALL])
def test_small_every_size_and_shape(cuda_lib, cap):
    """Both capacities: up to 4 nodes (keys and queries in one 8-wide tile) and
    up to 8 (two tiles)."""
    trees, acc = shapes(cap)
    w = custom(trees, acc)
    assert w.max_nodes == cap
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"small shapes, capacity {cap}")


@pytest.mark.parametrize("sizes,H", [([0, 3, 0, 8, 1, 0, 5], 5), ([4] * 7 + [0], 1), ([1, 1, 2, 0], 7)])
def test_small_ragged_with_empty_trees(cuda_lib, sizes, H):
    rng = np.random.default_rng(sum(sizes) + H)
    trees = [random_tree(rng, n) for n in sizes]
    acc = [len(t) - 1 for t in trees]
    w = custom(trees, acc, H=H, max_nodes=SMALL)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"ragged {sizes}")


@pytest.mark.parametrize("alpha,beta", [((1.0, 1.0), ("const", 1.0)),
                                        ((0.9, 0.999), ("const", 0.0)),
                                        ((0.01, 0.05), ("uniform", 0.05, 0.95)),
                                        ((0.999999, 0.9999999), ("uniform", 0.9999, 0.99999))])
@pytest.mark.parametrize("cap", [4, SMALL])
def test_small_gate_edges(cuda_lib, alpha, beta, cap):
    trees, acc = shapes(cap)
    w = custom(trees, acc, alpha=alpha, beta=beta, seed=37)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"gates {alpha} {beta}")


def test_small_agrees_with_tensor_cores(cuda_lib):
    """The same batch through the small-tree kernel (max_nodes 8) and the
    tcgen05 kernel (max_nodes 64): both within tolerance of the oracle, and of
    each other."""
    trees, acc = shapes()
    w_small = custom(trees, acc, seed=5)
    w_tc = custom(trees, acc, seed=5)
    small = CudaRun(w_small)
    tc = CudaRun(w_tc, max_nodes=64)
    assert not small.status.any() and not tc.status.any()
    assert_within(compare(w_small, small, range(w_small.R)), "small kernel")
    assert_within(compare(w_tc, tc, range(w_tc.R)), "tensor-core kernel")
    scale = float(np.abs(tc.o).max())
    assert float(np.abs(small.o - tc.o).max()) <= 2 * O_TOL * scale
    assert float(np.abs(small.U - tc.U).max()) <= 2 * U_TOL * float(np.abs(tc.U).max())
    assert np.array_equal(small.gamma, tc.gamma)  # the same products of alpha in the same order


def test_small_deterministic(cuda_lib):
    trees, acc = shapes()
    w = custom(trees, acc)
    tv = binding.TreeVerifier(w)
    tv.verify()
    o1, u1 = tv.o.clone(), tv.U.clone()
    tv.verify()
    torch.cuda.synchronize()
    assert torch.equal(o1, tv.o) and torch.equal(u1, tv.U)


@pytest.mark.parametrize("cap", [4, SMALL])
def test_small_bf16_state(cuda_lib, cap):
    """A bf16 state pool: verification reads the bf16 S0 exactly (o and U to
    the fp32 tolerances), the commit rounds S_a once to bf16:
    |S_gpu - S_ref| <= 2^-8 |S_ref| + 1e-3 max|S_ref| (8 significant bits,
    round to nearest, plus the fp32 bound before the rounding)."""
    trees, acc = shapes(cap)
    w = custom(trees, acc, seed=71, state_dtype="bf16")
    run = CudaRun(w, flags=binding.FLAG_STATE_BF16)
    assert not run.status.any()
    slot = w.state_slot.cpu().numpy()
    o_err = o_max = u_err = u_max = g_err = 0.0
    for r in range(w.R):
        lo, hi, S0, ref = oracle_request(w, r, run.S0_pool)
        o_err = max(o_err, float(np.abs(run.o[lo:hi] - ref.o).max()))
        o_max = max(o_max, float(np.abs(ref.o).max()))
        u_err = max(u_err, float(np.abs(run.U[lo:hi] - ref.U).max()))
        u_max = max(u_max, float(np.abs(ref.U).max()))
        g_err = max(g_err, float((np.abs(run.gamma[lo:hi] - ref.gamma) /
                                  np.maximum(ref.gamma, FLT_MIN)).max()))
        S_ref = orc.commit_request(S0, ref, int(acc[r]))
        S_gpu = np32(w.state[int(slot[r])]).astype(np.float64)
        bound = 2.0 ** -8 * np.abs(S_ref) + 1e-3 * np.abs(S_ref).max()
        assert np.all(np.abs(S_gpu - S_ref) <= bound), r
    assert o_err <= O_TOL * o_max, (o_err, o_max)
    assert u_err <= U_TOL * u_max, (u_err, u_max)
    assert g_err <= G_TOL, g_err


def test_small_bad_inputs_set_status_and_spare_others(cuda_lib):
    rng = np.random.default_rng(13)
    trees = [random_tree(rng, n) for n in (6, 7, 8, 5, 4, 7)]
    trees[1][4] = 5                        # parent after child
    trees[5][6] = 6                        # parent is the node itself
    acc = [3, 2, 1, 5, 0, 1]               # request 3: accepted outside its 5-node tree
    w = custom(trees, acc, max_nodes=SMALL, extra_slots=2)
    slots = w.state_slot.clone()
    slots[4] = -1                          # outside the pool
    w.state_slot.copy_(slots)
    tv = binding.TreeVerifier(w, max_nodes=7)  # request 2 (8 nodes) exceeds it
    tv.o.fill_(float("nan"))
    tv.U.fill_(float("nan"))
    S_before = w.state.clone()
    tv.verify()
    tv.commit()
    torch.cuda.synchronize()
    st = tv.status.cpu().tolist()
    assert st[0] == 0
    assert st[1] & binding.STATUS_BAD_TREE
    assert st[2] & binding.STATUS_TOO_MANY_NODES
    assert st[3] == binding.STATUS_BAD_ACCEPTED
    assert st[4] & binding.STATUS_BAD_SLOT
    assert st[5] & binding.STATUS_BAD_TREE
    node = w.node_offset.cpu().tolist()
    for r in (1, 2, 4, 5):
        assert torch.isnan(tv.o[node[r]:node[r + 1]]).all()
        assert torch.isnan(tv.U[node[r]:node[r + 1]]).all()
    for r in (1, 2, 3, 5):  # state untouched where the commit was refused
        s = int(w.state_slot[r])
        assert torch.equal(w.state[s], S_before[s])
    for r in (0, 3):        # verified normally
        lo, hi, S0, ref = oracle_request(w, r, S_before.cpu())
        assert np.abs(np32(tv.o[lo:hi]) - ref.o).max() <= O_TOL * np.abs(ref.o).max()


def two_rounds(prev_trees, next_trees, accepted, H=3, seed=43, cap=SMALL, state_dtype="f32"):
    """Two rounds over the same requests sharing one state pool; the previous
    round's trees may be larger than 8 nodes, the next round's are not."""
    R = len(prev_trees)
    prev = wl.assemble([np.asarray(t, np.int32) for t in prev_trees], np.asarray(accepted, np.int32),
                       H, 128, 128, "bf16", 0.05, (0.9, 0.999), ("sigmoid",), seed=seed,
                       extra_slots=3, state_dtype=state_dtype).to("cuda")
    nxt = wl.assemble([np.asarray(t, np.int32) for t in next_trees], np.full(R, -1, np.int32),
                      H, 128, 128, "bf16", 0.05, (0.9, 0.999), ("sigmoid",), seed=seed + 1,
                      max_nodes=cap, extra_slots=3, state_dtype=state_dtype).to("cuda")
    nxt.state = prev.state
    nxt.state_slot = prev.state_slot
    return prev, nxt


def run_commit_verify(prev, nxt):
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    assert not tp.status.any()
    S0_pool = prev.state.cpu()
    tn = binding.TreeVerifier(nxt)
    binding.treewy_commit_verify(tp.batch, prev.accepted, tn.batch)
    torch.cuda.synchronize()
    return tn, S0_pool


def check_two_rounds(prev, nxt, tn, S0_pool, requests, bf16=False, refused=(), verified=True):
    """The oracle commits the previous round (unless refused) and verifies the
    next one from the state the pool then holds: S_a (rounded to bf16 for a
    bf16 pool, |S_gpu - S_ref| <= 2^-8 |S_ref| + 1e-3 max|S_ref|; fp32: 1e-3
    max|S_ref|)."""
    o, U = np32(tn.o), np32(tn.U)
    pn, nn = prev.node_offset.cpu().numpy(), nxt.node_offset.cpu().numpy()
    acc = prev.accepted.cpu().numpy()
    for r in requests:
        slot = int(prev.state_slot[r])
        S0 = np32(S0_pool[slot]).astype(np.float64)
        S_gpu = np32(prev.state[slot]).astype(np.float64)
        if r in refused or int(acc[r]) < 0:
            assert np.array_equal(S_gpu, S0), r
            S_next = S0
        else:
            lo, hi = int(pn[r]), int(pn[r + 1])
            ref_prev = orc.verify_request(S0, prev.parent[lo:hi].cpu().numpy(), np32(prev.q[lo:hi]),
                                          np32(prev.k[lo:hi]), np32(prev.v[lo:hi]),
                                          np32(prev.alpha[lo:hi]), np32(prev.beta[lo:hi]))
            Sa = orc.commit_request(S0, ref_prev, int(acc[r]))
            if bf16:
                bound = 2.0 ** -8 * np.abs(Sa) + 1e-3 * np.abs(Sa).max()
                assert np.all(np.abs(S_gpu - Sa) <= bound), r
                S_next = orc.commit_request(S0, ref_prev, int(acc[r]), state_dtype="bf16")
            else:
                assert np.abs(S_gpu - Sa).max() <= 1e-3 * np.abs(Sa).max(), r
                S_next = Sa
        lo2, hi2 = int(nn[r]), int(nn[r + 1])
        if hi2 == lo2 or not verified:
            continue
        ref = orc.verify_request(S_next, nxt.parent[lo2:hi2].cpu().numpy(), np32(nxt.q[lo2:hi2]),
                                 np32(nxt.k[lo2:hi2]), np32(nxt.v[lo2:hi2]), np32(nxt.alpha[lo2:hi2]),
                                 np32(nxt.beta[lo2:hi2]))
        assert np.abs(o[lo2:hi2] - ref.o).max() <= O_TOL * np.abs(ref.o).max(), r
        assert np.abs(U[lo2:hi2] - ref.U).max() <= U_TOL * np.abs(ref.U).max(), r


@pytest.mark.parametrize("cap", [4, SMALL])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_small_commit_verify_matches_oracle(cuda_lib, cap, state_dtype):
    """treewy_commit_verify whose next trees have at most 4 or 8 nodes: accepted
    paths from the root only to 64 entries (eight update passes of the fused
    kernel for an fp32 pool; a bf16 pool with previous trees above 8 nodes
    takes the commit and the verification as two calls), no commit, empty
    next trees; S_a and the next round's o and U against the oracle run as
    commit-then-verify."""
    rng = np.random.default_rng(17 + cap)
    prev_trees = [random_tree(rng, n) for n in (40, 4, 64, 8, 1, 12, 9)]
    prev_trees[2] = wl.chain_parents(64)
    prev_trees[6] = wl.chain_parents(9)     # a path of kSeg + 1 entries
    next_trees = [random_tree(rng, n) for n in (cap, 2, 0, 1, cap - 1, 3, cap)]
    accepted = [39, -1, 63, 5, 0, 11, 8]
    prev, nxt = two_rounds(prev_trees, next_trees, accepted, cap=cap, state_dtype=state_dtype)
    tn, S0_pool = run_commit_verify(prev, nxt)
    assert not tn.status.any(), tn.status.tolist()
    check_two_rounds(prev, nxt, tn, S0_pool, range(len(prev_trees)), bf16=state_dtype == "bf16")


@pytest.mark.parametrize("cap", [4, SMALL])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_small_commit_verify_short_paths(cuda_lib, cap, state_dtype):
    """Both rounds with trees of at most 8 nodes (the fused kernel for either
    pool; a bf16 pool's S_a rounded once): chains, stars and random trees,
    accepted nodes from the root to the deepest node."""
    rng = np.random.default_rng(41 + cap)
    prev_trees = [wl.chain_parents(8), np.array([-1] + [0] * 7, np.int32), random_tree(rng, 5),
                  random_tree(rng, 8), wl.chain_parents(3), random_tree(rng, 1)]
    next_trees = [random_tree(rng, n) for n in (cap, 1, cap, 2, 0, cap - 1)]
    accepted = [7, 6, 4, 5, -1, 0]
    prev, nxt = two_rounds(prev_trees, next_trees, accepted, cap=cap, state_dtype=state_dtype, seed=9)
    assert prev.max_nodes <= SMALL
    tn, S0_pool = run_commit_verify(prev, nxt)
    assert not tn.status.any(), tn.status.tolist()
    check_two_rounds(prev, nxt, tn, S0_pool, range(len(prev_trees)), bf16=state_dtype == "bf16")


def test_small_commit_verify_refusals(cuda_lib):
    """Each half runs exactly when its separate call would: an accepted index
    outside the previous tree, a previous parent after its node and a state
    slot outside the pool refuse the commit (state unchanged, COMMIT_REFUSED
    beside the reason; the bad slot skips the verification too), while a bad
    next tree (parent after its node, more nodes than the capacity) skips
    only the verification and still commits."""
    rng = np.random.default_rng(29)
    prev_trees = [random_tree(rng, n) for n in (6, 7, 5, 8, 6, 4)]
    prev_trees[2] = prev_trees[2].copy()
    prev_trees[2][3] = 4                    # previous tree: parent after its node
    next_trees = [random_tree(rng, n) for n in (4, 3, 4, 4, 6, 2)]
    next_trees[3] = next_trees[3].copy()
    next_trees[3][2] = 3                    # next tree: parent after its node
    accepted = [5, 7, 2, 6, 3, 1]           # request 1: outside its 7-node tree
    prev, nxt = two_rounds(prev_trees, next_trees, accepted, cap=SMALL)
    slots = prev.state_slot.clone()
    slots[5] = prev.num_slots               # outside the pool
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    S0_pool = prev.state.cpu()
    prev.state_slot.copy_(slots)
    nxt.state_slot = prev.state_slot
    tn = binding.TreeVerifier(nxt, max_nodes=4)   # request 4 (6 nodes) exceeds it
    tn.o.fill_(float("nan"))
    binding.treewy_commit_verify(tp.batch, prev.accepted, tn.batch)
    torch.cuda.synchronize()
    st = tn.status.cpu().tolist()
    R_ = binding.STATUS_COMMIT_REFUSED
    assert st[0] == 0, st
    assert st[1] == binding.STATUS_BAD_ACCEPTED | R_, st
    assert st[2] == binding.STATUS_BAD_TREE | R_, st
    assert st[3] == binding.STATUS_BAD_TREE, st
    assert st[4] == binding.STATUS_TOO_MANY_NODES, st
    assert st[5] == binding.STATUS_BAD_SLOT | R_, st
    nn = nxt.node_offset.cpu().tolist()
    for r in (3, 4, 5):
        assert torch.isnan(tn.o[nn[r]:nn[r + 1]]).all(), r
    check_two_rounds(prev, nxt, tn, S0_pool, [0, 1, 2], refused=(1, 2))
    # committed although not verified
    check_two_rounds(prev, nxt, tn, S0_pool, [3, 4], verified=False)


def test_small_commit_verify_equals_separate_calls(cuda_lib):
    """The chain workload, two layers on one state pool: the fused call
    against verify(prev), commit(prev), verify(next)."""
    cfg = wl.CONFIGS["chain"]
    pa = wl.generate(cfg, R=48).to("cuda")
    na = wl.generate(cfg, R=48, layer=1).to("cuda")
    pb = wl.generate(cfg, R=48).to("cuda")
    nb = wl.generate(cfg, R=48, layer=1).to("cuda")
    na.state, na.state_slot = pa.state, pa.state_slot
    nb.state, nb.state_slot = pb.state, pb.state_slot
    tn, _ = run_commit_verify(pa, na)
    tpb = binding.TreeVerifier(pb)
    tpb.verify()
    tpb.commit()
    tnb = binding.TreeVerifier(nb)
    tnb.verify()
    torch.cuda.synchronize()
    assert not tn.status.any() and not tnb.status.any()
    ds = (pa.state - pb.state).abs().max().item()
    assert ds <= 1e-4 * pb.state.abs().max().item(), ds
    do = (tn.o - tnb.o).abs().max().item()
    assert do <= 1e-3 * tnb.o.abs().max().item(), do


def test_small_graph_replay_matches_eager(cuda_lib):
    """The chain workload's verify + commit captured in a CUDA graph and
    replayed: the oracle's results within the tolerances, and the eager
    launches' bit for bit."""
    cfg = wl.CONFIGS["chain"]
    w_eager = wl.generate(cfg, R=24).to("cuda")
    run = CudaRun(w_eager)
    w = wl.generate(cfg, R=24).to("cuda")
    assert w.max_nodes <= SMALL
    S0 = w.state.clone()
    tv = binding.TreeVerifier(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tv.verify(s)
        w.state.copy_(S0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tv.verify()
        tv.commit()
    w.state.copy_(S0)
    tv.o.fill_(float("nan"))
    tv.U.fill_(float("nan"))
    tv.gamma.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert not tv.status.any()
    replay = types.SimpleNamespace(o=np32(tv.o), U=np32(tv.U), gamma=np32(tv.gamma),
                                   S0_pool=S0.cpu(), S_after=w.state)
    assert_within(compare(w, replay, range(w.R)), "chain graph replay")
    assert torch.equal(tv.o.cpu(), torch.from_numpy(run.o))
    assert torch.equal(w.state.cpu(), run.S_after.cpu())


def test_small_commit_verify_chain_full_size(cuda_lib):
    """The chain workload at full size (64 requests x 32 heads, the launch
    configuration of the per-workload study): two layers on one state pool,
    the fused call against the oracle run as commit-then-verify on every
    request."""
    cfg = wl.CONFIGS["chain"]
    prev = wl.generate(cfg).to("cuda")
    nxt = wl.generate(cfg, layer=1).to("cuda")
    nxt.state, nxt.state_slot = prev.state, prev.state_slot
    assert prev.max_nodes <= SMALL and nxt.max_nodes <= SMALL
    assert (prev.accepted.cpu() == -1).any()   # the no-op commit is exercised
    tn, S0_pool = run_commit_verify(prev, nxt)
    assert not tn.status.any(), tn.status.tolist()
    check_two_rounds(prev, nxt, tn, S0_pool, range(prev.R))
