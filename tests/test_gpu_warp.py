"""GPU parity of the warp-MMA verification (batches whose trees have 9 to 32
nodes: dk = dv = 128 with bf16 q/k/v; capacities 16 and 32, the latter with
an fp32 state streamed through a ring of three of its four boxes) against the
oracle on the same seeded inputs: every size from 1 to 16 (and 32) in chain,
star, forest and random shapes (chains longer than 8 take the kernel's general
root-path recurrence, shorter paths its register form), the smallest
capacities routed to it (9, 17), ragged batches with empty trees, gates at the
ends of their range,
a bf16 state pool, device-side errors, CUDA-graph replay, agreement with
the small-tree and tcgen05 kernels on the same inputs, and the commit fused
in front (paths of 1 to 64 entries, both pools, refusals, against the two
separate calls, the binary workload at full size).  Tolerances as in
gpu_helpers (o, U: 2e-3 of the largest reference value; committed state
1e-3; gamma 1e-5 relative).
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
from tests.test_gpu_small import (check_two_rounds, custom, random_tree, run_commit_verify, shapes,
                                  two_rounds)

pytestmark = pytest.mark.gpu

CAP = 16   # node capacity of the warp-MMA kernel's fused form
CAP2 = 32  # ... and of its plain verification


@pytest.mark.parametrize("cap", [CAP, CAP2])
def test_warp_every_size_and_shape(cuda_lib, cap):
    trees, acc = shapes(cap)
    w = custom(trees, acc, H=2 if cap > CAP else 3)
    assert w.max_nodes == cap
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"warp kernel shapes, capacity {cap}")


@pytest.mark.parametrize("max_nodes,sizes", [(9, [9, 1, 9, 0, 4]), (16, [16]), (12, [12, 11, 3]),
                                             (17, [17, 1, 17, 0, 9]), (32, [32]), (24, [24, 20, 18])])
def test_warp_capacities(cuda_lib, max_nodes, sizes):
    """The smallest capacities routed to the kernel's two instances (9, 17)
    and full trees at them."""
    rng = np.random.default_rng(max_nodes + len(sizes))
    trees = [random_tree(rng, n) for n in sizes]
    if len(sizes) == 1:
        trees = [wl.chain_parents(sizes[0])]  # the longest root path
    acc = [len(t) - 1 for t in trees]
    w = custom(trees, acc, H=2, max_nodes=max_nodes)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"capacity {max_nodes}, sizes {sizes}")


@pytest.mark.parametrize("sizes,H", [([0, 13, 0, 16, 1, 0, 9], 5), ([15] * 7 + [0], 1), ([10, 2, 14, 0], 7),
                                     ([0, 29, 0, 32, 1, 0, 17], 5), ([31] * 5 + [0], 1)])
def test_warp_ragged_with_empty_trees(cuda_lib, sizes, H):
    rng = np.random.default_rng(sum(sizes) + H)
    trees = [random_tree(rng, n) for n in sizes]
    acc = [len(t) - 1 for t in trees]
    w = custom(trees, acc, H=H, max_nodes=CAP if max(sizes) <= CAP else CAP2)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"ragged {sizes}")


@pytest.mark.parametrize("alpha,beta", [((1.0, 1.0), ("const", 1.0)),
                                        ((0.9, 0.999), ("const", 0.0)),
                                        ((0.01, 0.05), ("uniform", 0.05, 0.95)),
                                        ((0.999999, 0.9999999), ("uniform", 0.9999, 0.99999))])
@pytest.mark.parametrize("cap", [CAP, CAP2])
def test_warp_gate_edges(cuda_lib, alpha, beta, cap):
    trees, acc = shapes(cap)
    w = custom(trees, acc, alpha=alpha, beta=beta, seed=41)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"gates {alpha} {beta}")


def test_warp_agrees_with_other_kernels(cuda_lib):
    """The same batch through the warp-MMA kernel (max_nodes 16 and 32) and
    the tcgen05 kernel (max_nodes 64), and its trees of at most 8 nodes
    through the small-tree kernel as well: all within tolerance of the oracle
    and of each other, with identical decays (the same products of alpha in
    the same order)."""
    trees, acc = shapes(CAP)
    runs = {}
    for name, mn in (("warp", 16), ("warp32", 32), ("tcgen05", 64)):
        w = custom(trees, acc, seed=5)
        runs[name] = (w, CudaRun(w, max_nodes=mn))
    for name, (w, run) in runs.items():
        assert not run.status.any(), name
        assert_within(compare(w, run, range(w.R)), name)
    warp, tc = runs["warp"][1], runs["tcgen05"][1]
    assert float(np.abs(warp.o - tc.o).max()) <= 2 * O_TOL * float(np.abs(tc.o).max())
    assert float(np.abs(warp.U - tc.U).max()) <= 2 * U_TOL * float(np.abs(tc.U).max())
    assert np.array_equal(warp.gamma, tc.gamma)
    w32 = runs["warp32"][1]
    assert float(np.abs(w32.o - tc.o).max()) <= 2 * O_TOL * float(np.abs(tc.o).max())
    assert np.array_equal(w32.gamma, tc.gamma)
    small_trees = [t for t in trees if len(t) <= 8]
    small_acc = [a for t, a in zip(trees, acc) if len(t) <= 8]
    ws, ww = custom(small_trees, small_acc, seed=9), custom(small_trees, small_acc, seed=9)
    small, warp8 = CudaRun(ws), CudaRun(ww, max_nodes=16)
    assert not small.status.any() and not warp8.status.any()
    assert_within(compare(ww, warp8, range(ww.R)), "warp kernel, trees of at most 8 nodes")
    assert float(np.abs(warp8.o - small.o).max()) <= 2 * O_TOL * float(np.abs(small.o).max())
    assert np.array_equal(warp8.gamma, small.gamma)


def test_warp_deterministic(cuda_lib):
    trees, acc = shapes(CAP)
    w = custom(trees, acc)
    tv = binding.TreeVerifier(w)
    tv.verify()
    o1, u1 = tv.o.clone(), tv.U.clone()
    tv.verify()
    torch.cuda.synchronize()
    assert torch.equal(o1, tv.o) and torch.equal(u1, tv.U)


@pytest.mark.parametrize("cap", [CAP, CAP2])
def test_warp_bf16_state(cuda_lib, cap):
    """A bf16 state pool: verification reads the bf16 S0 exactly (o and U to
    the fp32 tolerances), the commit rounds S_a once to bf16:
    |S_gpu - S_ref| <= 2^-8 |S_ref| + 1e-3 max|S_ref|."""
    trees, acc = shapes(cap)
    w = custom(trees, acc, seed=73, state_dtype="bf16")
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


@pytest.mark.parametrize("cap", [CAP, CAP2])
def test_warp_bad_inputs_set_status_and_spare_others(cuda_lib, cap):
    rng = np.random.default_rng(29 + cap)
    k = cap - CAP                          # sizes shifted into the capacity tested
    trees = [random_tree(rng, n + k) for n in (12, 15, 16, 10, 9, 14)]
    trees[1][11] = 13 + k                  # parent after child
    trees[5][13] = 13                      # parent is the node itself
    acc = [3, 2, 1, 10 + k, 0, 1]          # request 3: accepted outside its tree
    w = custom(trees, acc, max_nodes=cap, extra_slots=2)
    slots = w.state_slot.clone()
    slots[4] = -1                          # outside the pool
    w.state_slot.copy_(slots)
    tv = binding.TreeVerifier(w, max_nodes=cap - 1)  # request 2 (cap nodes) exceeds it
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
        assert np.abs(np32(tv.U[lo:hi]) - ref.U).max() <= U_TOL * np.abs(ref.U).max()


def test_warp_graph_replay_matches_eager(cuda_lib):
    """The binary-tree workload's verify + commit captured in a CUDA graph and
    replayed: the oracle's results within the tolerances, and the eager
    launches' bit for bit."""
    cfg = wl.CONFIGS["binary"]
    w_eager = wl.generate(cfg, R=12).to("cuda")
    run = CudaRun(w_eager)
    w = wl.generate(cfg, R=12).to("cuda")
    assert 8 < w.max_nodes <= CAP
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
    assert_within(compare(w, replay, range(w.R)), "binary graph replay")
    assert torch.equal(tv.o.cpu(), torch.from_numpy(run.o))
    assert torch.equal(w.state.cpu(), run.S_after.cpu())


@pytest.mark.parametrize("cap", [CAP, CAP2])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_warp_commit_verify_matches_oracle(cuda_lib, state_dtype, cap):
    """treewy_commit_verify whose next trees have 9 to 16 nodes: accepted paths
    from the root only to 64 entries (four update passes of 16 entries for an
    fp32 pool; a bf16 pool with previous trees above 16 nodes takes the commit
    and the verification as two calls), no commit, empty next trees;
    S_a and the next round's o and U against the oracle run as
    commit-then-verify."""
    rng = np.random.default_rng(23)
    prev_trees = [random_tree(rng, n) for n in (40, 4, 64, 8, 1, 12, 9, 16)]
    prev_trees[2] = wl.chain_parents(64)
    prev_trees[6] = wl.chain_parents(17)    # a path of one pass + 1 entry
    next_trees = [random_tree(rng, n) for n in (cap, 2, 0, 1, cap - 1, 3, 9, 12)]
    next_trees[0] = wl.chain_parents(cap)   # the longest next root path
    accepted = [39, -1, 63, 5, 0, 11, 16, 15]
    prev, nxt = two_rounds(prev_trees, next_trees, accepted, cap=cap, state_dtype=state_dtype)
    tn, S0_pool = run_commit_verify(prev, nxt)
    assert not tn.status.any(), tn.status.tolist()
    check_two_rounds(prev, nxt, tn, S0_pool, range(len(prev_trees)), bf16=state_dtype == "bf16")


@pytest.mark.parametrize("cap", [CAP, CAP2])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_warp_commit_verify_short_paths(cuda_lib, state_dtype, cap):
    """Previous trees of at most 16 nodes (one update pass with every node's U
    and key row requested up front; a bf16 pool's S_a rounded once), next
    trees of up to 16: chains, stars, binary and random trees, accepted nodes
    from the root to the deepest node."""
    rng = np.random.default_rng(43)
    prev_trees = [wl.chain_parents(16), np.array([-1] + [0] * 15, np.int32), random_tree(rng, 5),
                  random_tree(rng, 12), wl.chain_parents(3), random_tree(rng, 1),
                  wl.complete_binary_parents(4), wl.chain_parents(8)]
    next_trees = [random_tree(rng, n) for n in (cap, 1, 11, 2, 0, cap - 1, 15, 9)]
    accepted = [15, 9, 4, 11, -1, 0, 14, 7]
    prev, nxt = two_rounds(prev_trees, next_trees, accepted, cap=cap, state_dtype=state_dtype, seed=11)
    assert prev.max_nodes <= 16
    tn, S0_pool = run_commit_verify(prev, nxt)
    assert not tn.status.any(), tn.status.tolist()
    check_two_rounds(prev, nxt, tn, S0_pool, range(len(prev_trees)), bf16=state_dtype == "bf16")


def test_warp_commit_verify_refusals(cuda_lib):
    """Each half runs exactly when its separate call would: an accepted index
    outside the previous tree, a previous parent after its node and a state
    slot outside the pool refuse the commit (state unchanged, COMMIT_REFUSED
    beside the reason; the bad slot skips the verification too), while a bad
    next tree (parent after its node, more nodes than the capacity) skips
    only the verification and still commits."""
    rng = np.random.default_rng(31)
    prev_trees = [random_tree(rng, n) for n in (6, 7, 5, 12, 6, 4)]
    prev_trees[2] = prev_trees[2].copy()
    prev_trees[2][3] = 4                    # previous tree: parent after its node
    next_trees = [random_tree(rng, n) for n in (12, 3, 9, 14, 16, 10)]
    next_trees[3] = next_trees[3].copy()
    next_trees[3][12] = 13                  # next tree: parent after its node
    accepted = [5, 7, 2, 11, 3, 1]          # request 1: outside its 7-node tree
    prev, nxt = two_rounds(prev_trees, next_trees, accepted, cap=CAP)
    slots = prev.state_slot.clone()
    slots[5] = prev.num_slots               # outside the pool
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    S0_pool = prev.state.cpu()
    prev.state_slot.copy_(slots)
    nxt.state_slot = prev.state_slot
    tn = binding.TreeVerifier(nxt, max_nodes=15)   # request 4 (16 nodes) exceeds it
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


def test_warp_commit_verify_equals_separate_calls(cuda_lib):
    """The binary-tree workload, two layers on one state pool: the fused call
    against verify(prev), commit(prev), verify(next)."""
    cfg = wl.CONFIGS["binary"]
    pa = wl.generate(cfg, R=24).to("cuda")
    na = wl.generate(cfg, R=24, layer=1).to("cuda")
    pb = wl.generate(cfg, R=24).to("cuda")
    nb = wl.generate(cfg, R=24, layer=1).to("cuda")
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


def test_warp_commit_verify_binary_full_size(cuda_lib):
    """The binary-tree workload at full size (128 requests x 32 heads, the
    launch configuration of the per-workload study): two layers on one state
    pool, the fused call against the oracle run as commit-then-verify on
    every request."""
    cfg = wl.CONFIGS["binary"]
    prev = wl.generate(cfg).to("cuda")
    nxt = wl.generate(cfg, layer=1).to("cuda")
    nxt.state, nxt.state_slot = prev.state, prev.state_slot
    assert 8 < nxt.max_nodes <= CAP
    tn, S0_pool = run_commit_verify(prev, nxt)
    assert not tn.status.any(), tn.status.tolist()
    check_two_rounds(prev, nxt, tn, S0_pool, range(prev.R))
