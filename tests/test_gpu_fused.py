"""GPU parity of treewy_commit_verify (the previous round's commit fused into the
next round's verification) against the oracle run as commit-then-verify on the
same seeded inputs, and against the two separate library calls.
"""
import numpy as np
import pytest
import torch

from gdn_speculative_tree_gb300 import binding
from gdn_speculative_tree_gb300 import workloads as wl
from oracle import gdn_tree_oracle as orc
from tests.gpu_helpers import np32

pytestmark = pytest.mark.gpu


def rounds(prev_trees, next_trees, accepted, H=4, dk=128, dv=128, qkv="bf16", seed=41, max_nodes=64):
    """Two rounds over the same requests sharing one state pool."""
    R = len(prev_trees)
    assert len(next_trees) == R
    prev = wl.assemble([np.asarray(t, np.int32) for t in prev_trees], np.asarray(accepted, np.int32),
                       H, dk, dv, qkv, 0.05, (0.9, 0.999), ("sigmoid",), seed=seed, max_nodes=max_nodes,
                       extra_slots=3).to("cuda")
    nxt = wl.assemble([np.asarray(t, np.int32) for t in next_trees], np.full(R, -1, np.int32),
                      H, dk, dv, qkv, 0.05, (0.9, 0.999), ("sigmoid",), seed=seed + 1, max_nodes=max_nodes,
                      extra_slots=3).to("cuda")
    nxt.state = prev.state
    nxt.state_slot = prev.state_slot
    return prev, nxt


def random_tree(rng, n):
    return np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32) if n else \
        np.zeros(0, np.int32)


def oracle_commit(prev, S0_pool, r):
    """Oracle: the state committed from the previous round's tree."""
    S0 = np32(S0_pool[int(prev.state_slot[r])])
    pn = prev.node_offset.cpu().numpy()
    lo, hi = int(pn[r]), int(pn[r + 1])
    ref_prev = orc.verify_request(S0, prev.parent[lo:hi].cpu().numpy(), np32(prev.q[lo:hi]),
                                  np32(prev.k[lo:hi]), np32(prev.v[lo:hi]), np32(prev.alpha[lo:hi]),
                                  np32(prev.beta[lo:hi]))
    return orc.commit_request(S0, ref_prev, int(prev.accepted[r]))


def oracle_two_rounds(prev, nxt, S0_pool, r):
    """Oracle: S_a from the previous round's tree, then the next round from S_a."""
    slot = int(prev.state_slot[r])
    S0 = np32(S0_pool[slot])
    pn = prev.node_offset.cpu().numpy()
    lo, hi = int(pn[r]), int(pn[r + 1])
    ref_prev = orc.verify_request(S0, prev.parent[lo:hi].cpu().numpy(), np32(prev.q[lo:hi]),
                                  np32(prev.k[lo:hi]), np32(prev.v[lo:hi]), np32(prev.alpha[lo:hi]),
                                  np32(prev.beta[lo:hi]))
    Sa = orc.commit_request(S0, ref_prev, int(prev.accepted[r]))
    nn = nxt.node_offset.cpu().numpy()
    lo2, hi2 = int(nn[r]), int(nn[r + 1])
    ref_next = orc.verify_request(Sa, nxt.parent[lo2:hi2].cpu().numpy(), np32(nxt.q[lo2:hi2]),
                                  np32(nxt.k[lo2:hi2]), np32(nxt.v[lo2:hi2]), np32(nxt.alpha[lo2:hi2]),
                                  np32(nxt.beta[lo2:hi2]))
    return Sa, ref_next, (lo2, hi2)


def run_fused(prev, nxt):
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    assert not tp.status.any()
    S0_pool = prev.state.cpu()
    tn = binding.TreeVerifier(nxt)
    binding.treewy_commit_verify(tp.batch, prev.accepted, tn.batch)
    torch.cuda.synchronize()
    return tp, tn, S0_pool


def check(prev, nxt, tn, S0_pool, requests):
    o = np32(tn.o)
    U = np32(tn.U)
    o_err = o_max = s_err = s_max = u_err = u_max = 0.0
    for r in requests:
        Sa, ref, (lo, hi) = oracle_two_rounds(prev, nxt, S0_pool, r)
        S_gpu = np32(prev.state[int(prev.state_slot[r])])
        s_err = max(s_err, float(np.abs(S_gpu - Sa).max()))
        s_max = max(s_max, float(np.abs(Sa).max()))
        if hi > lo:
            o_err = max(o_err, float(np.abs(o[lo:hi] - ref.o).max()))
            o_max = max(o_max, float(np.abs(ref.o).max()))
            u_err = max(u_err, float(np.abs(U[lo:hi] - ref.U).max()))
            u_max = max(u_max, float(np.abs(ref.U).max()))
    assert s_err <= 1e-3 * s_max, (s_err, s_max)
    assert o_err <= 2e-3 * o_max, (o_err, o_max)
    assert u_err <= 2e-3 * u_max, (u_err, u_max)


def test_fused_matches_oracle_mixed(cuda_lib):
    rng = np.random.default_rng(61)
    prev_trees = [random_tree(rng, n) for n in (12, 40, 64, 5, 30, 17, 9, 64)]
    prev_trees[7] = wl.chain_parents(64)  # a 64-long accepted path (several staged segments)
    next_trees = [random_tree(rng, n) for n in (20, 0, 33, 64, 1, 17, 48, 10)]
    accepted = [5, 39, -1, 4, 29, 0, 8, 63]
    prev, nxt = rounds(prev_trees, next_trees, accepted)
    tp, tn, S0_pool = run_fused(prev, nxt)
    assert not tn.status.any(), tn.status.tolist()
    check(prev, nxt, tn, S0_pool, range(len(prev_trees)))


@pytest.mark.parametrize("max_nodes", [16, 32])
def test_fused_small_buckets(cuda_lib, max_nodes):
    """The 16- and 32-node capacity buckets (the update's operand tile after
    the lists, and in the K/Q region whose boxes wait for it): accepted paths
    of one and two 16-entry segments (a chain as long as the capacity), a
    commit of the root only, a request without commit, an empty next tree."""
    rng = np.random.default_rng(200 + max_nodes)
    prev_trees = [random_tree(rng, n) for n in (max_nodes // 2, 3, max_nodes - 1, 1)]
    prev_trees.append(wl.chain_parents(max_nodes))
    next_trees = [random_tree(rng, n) for n in (max_nodes, 5, 0, max_nodes // 2, 2)]
    accepted = [max_nodes // 2 - 1, -1, max_nodes - 2, 0, max_nodes - 1]
    prev, nxt = rounds(prev_trees, next_trees, accepted, H=3, seed=31, max_nodes=max_nodes)
    tp, tn, S0_pool = run_fused(prev, nxt)
    assert not tn.status.any()
    check(prev, nxt, tn, S0_pool, range(len(prev_trees)))


def test_fused_matches_separate_calls(cuda_lib):
    cfg = wl.CONFIGS["wide"]
    trees, acc = wl.make_trees(cfg, R=10)
    rng = np.random.default_rng(3)
    nxt_trees = [random_tree(rng, int(rng.integers(16, 65))) for _ in range(10)]
    prev_a, nxt_a = rounds(trees, nxt_trees, acc, H=8, seed=7)
    prev_b, nxt_b = rounds(trees, nxt_trees, acc, H=8, seed=7)
    # fused
    tp, tn, _ = run_fused(prev_a, nxt_a)
    # separate: verify(prev), commit(prev), verify(next)
    tpb = binding.TreeVerifier(prev_b)
    tpb.verify()
    tpb.commit()
    tnb = binding.TreeVerifier(nxt_b)
    tnb.verify()
    torch.cuda.synchronize()
    assert not tn.status.any() and not tnb.status.any()
    ds = (prev_a.state - prev_b.state).abs().max().item()
    assert ds <= 1e-4 * prev_b.state.abs().max().item(), ds
    do = (tn.o - tnb.o).abs().max().item()
    assert do <= 1e-3 * tnb.o.abs().max().item(), do


def check_next_from_unchanged(nxt, tn, S_before, r):
    """Request r's next round verified from its unchanged state (refused commit)."""
    nn = nxt.node_offset.cpu().numpy()
    lo, hi = int(nn[r]), int(nn[r + 1])
    ref = orc.verify_request(np32(S_before[int(nxt.state_slot[r])]), nxt.parent[lo:hi].cpu().numpy(),
                             np32(nxt.q[lo:hi]), np32(nxt.k[lo:hi]), np32(nxt.v[lo:hi]),
                             np32(nxt.alpha[lo:hi]), np32(nxt.beta[lo:hi]))
    o_err = float(np.abs(np32(tn.o[lo:hi]) - ref.o).max())
    assert o_err <= 2e-3 * float(np.abs(ref.o).max()), o_err


def test_fused_bad_previous_round_refuses_commit_only(cuda_lib):
    """Tensor-core path: an accepted index outside the previous tree refuses
    that request's commit (state unchanged, COMMIT_REFUSED beside the reason)
    and the request is verified from its unchanged state, as the separate
    calls would do."""
    rng = np.random.default_rng(5)
    prev_trees = [random_tree(rng, 10), random_tree(rng, 12), random_tree(rng, 8)]
    next_trees = [random_tree(rng, 9), random_tree(rng, 11), random_tree(rng, 7)]
    prev, nxt = rounds(prev_trees, next_trees, [3, 12, 2])   # request 1: accepted outside its tree
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    S_before = prev.state.clone()
    tn = binding.TreeVerifier(nxt)
    binding.treewy_commit_verify(tp.batch, prev.accepted, tn.batch)
    torch.cuda.synchronize()
    st = tn.status.cpu().tolist()
    assert st[0] == 0 and st[2] == 0
    assert st[1] == binding.STATUS_BAD_ACCEPTED | binding.STATUS_COMMIT_REFUSED, st
    s1 = int(prev.state_slot[1])
    assert torch.equal(prev.state[s1], S_before[s1])
    check(prev, nxt, tn, S_before.cpu(), [0, 2])
    check_next_from_unchanged(nxt, tn, S_before.cpu(), 1)


@pytest.mark.parametrize("dk,dv,qkv", [(128, 128, "bf16"), (128, 128, "f32"), (64, 48, "bf16")])
def test_fused_bad_next_tree_still_commits(cuda_lib, dk, dv, qkv):
    """An error in the next round's tree skips that request's verification
    but not the previous round's commit: a tree above the batch's capacity,
    a parent index out of range and a node range past T each leave S_a
    written (no COMMIT_REFUSED) and the request's outputs untouched, on the
    tensor-core kernel and on the fallback shapes."""
    rng = np.random.default_rng(dk + dv)
    prev_trees = [random_tree(rng, n) for n in (10, 14, 9, 12)]
    next_trees = [random_tree(rng, n) for n in (6, 40, 9, 7)]
    next_trees[2] = next_trees[2].copy()
    next_trees[2][5] = 7                      # parent after the node
    prev, nxt = rounds(prev_trees, next_trees, [4, 13, 8, 11], H=3, dk=dk, dv=dv, qkv=qkv)
    nxt.max_nodes = 32                        # request 1 (40 nodes) exceeds the capacity
    T = int(nxt.node_offset[-1])
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    S0_pool = prev.state.cpu()
    tn = binding.TreeVerifier(nxt, max_nodes=32)
    tn.o.fill_(float("nan"))
    # request 3's node range runs past the rows the batch declares
    tn.batch.T = T - 2
    binding.treewy_commit_verify(tp.batch, prev.accepted, tn.batch)
    torch.cuda.synchronize()
    st = tn.status.cpu().tolist()
    assert st[0] == 0, st
    assert st[1] == binding.STATUS_TOO_MANY_NODES, st
    assert st[2] == binding.STATUS_BAD_TREE, st
    assert st[3] == binding.STATUS_BAD_TREE, st
    nn = nxt.node_offset.cpu().tolist()
    for r in (1, 2, 3):
        assert torch.isnan(tn.o[nn[r]:min(nn[r + 1], T)]).all(), r
    # every request's commit happened
    s_err = s_max = 0.0
    for r in range(4):
        Sa = oracle_commit(prev, S0_pool, r)
        S_gpu = np32(prev.state[int(prev.state_slot[r])])
        s_err = max(s_err, float(np.abs(S_gpu - Sa).max()))
        s_max = max(s_max, float(np.abs(Sa).max()))
    assert s_err <= 1e-3 * s_max, (s_err, s_max)
    check(prev, nxt, tn, S0_pool, [0])


@pytest.mark.parametrize("dk,dv,qkv", [(128, 128, "f32"), (64, 48, "bf16")])
def test_fused_fallback_shapes(cuda_lib, dk, dv, qkv):
    rng = np.random.default_rng(dk)
    prev_trees = [random_tree(rng, n) for n in (7, 20, 3)]
    next_trees = [random_tree(rng, n) for n in (5, 0, 9)]
    prev, nxt = rounds(prev_trees, next_trees, [6, 19, -1], H=2, dk=dk, dv=dv, qkv=qkv)
    tp, tn, S0_pool = run_fused(prev, nxt)
    assert not tn.status.any()
    check(prev, nxt, tn, S0_pool, range(3))


def test_fused_full_size_sampled(cuda_lib):
    """The benchmark's layer size and launch configuration (256 requests x 32
    heads, N 16..64): the previous round is one layer, the next round another
    layer's draws on the same state pool; sampled requests (all heads) against
    the oracle's commit-then-verify."""
    cfg = wl.CONFIGS["wide"]
    prev = wl.generate(cfg, device="cuda")
    nxt = wl.generate(cfg, layer=1, device="cuda")
    nxt.state = prev.state
    nxt.state_slot = prev.state_slot
    tp, tn, S0_pool = run_fused(prev, nxt)
    assert not tn.status.any()
    rng = np.random.default_rng(2024)
    reqs = sorted(set(rng.choice(cfg.R, 3, replace=False).tolist()) | {cfg.R - 1})
    check(prev, nxt, tn, S0_pool, reqs)


def test_fused_fallback_bad_previous_round(cuda_lib):
    """Outside the tensor-core path: a refused commit reports in next's status
    and leaves the state unchanged; that request is still verified from it."""
    rng = np.random.default_rng(8)
    prev_trees = [random_tree(rng, 6), random_tree(rng, 9)]
    next_trees = [random_tree(rng, 5), random_tree(rng, 4)]
    prev, nxt = rounds(prev_trees, next_trees, [2, 9], H=2, qkv="f32")  # request 1: a >= N
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    S_before = prev.state.clone()
    tn = binding.TreeVerifier(nxt)
    binding.treewy_commit_verify(tp.batch, prev.accepted, tn.batch)
    torch.cuda.synchronize()
    st = tn.status.cpu().tolist()
    assert st[0] == 0 and st[1] == binding.STATUS_BAD_ACCEPTED | binding.STATUS_COMMIT_REFUSED, st
    assert not tp.status.any()
    s1 = int(prev.state_slot[1])
    assert torch.equal(prev.state[s1], S_before[s1])
    check(prev, nxt, tn, S_before.cpu(), [0])
    check_next_from_unchanged(nxt, tn, S_before.cpu(), 1)
