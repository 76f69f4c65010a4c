"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, element by element, for the five workload shapes (full
size where the oracle finishes in seconds, sampled requests at full size
otherwise), random and degenerate trees, both kernels, the storeall
comparator, device-side error reporting and CUDA-graph replay.
"""
import types

import numpy as np
import pytest
import torch

from gdn_speculative_tree_gb300 import binding
from gdn_speculative_tree_gb300 import workloads as wl
from oracle import gdn_tree_oracle as orc
from tests.gpu_helpers import CudaRun, assert_within, compare, np32, oracle_request

pytestmark = pytest.mark.gpu


def cpu_then_cuda(name, R=None, **over):
    cfg = wl.CONFIGS[name].with_(**over) if over else wl.CONFIGS[name]
    return wl.generate(cfg, R=R).to("cuda")


# ------------------------------------------------------------ the five shapes

def test_tiny_chain_fp32(cuda_lib):
    w = cpu_then_cuda("tiny")
    run = CudaRun(w)
    assert run.status.tolist() == [0]
    assert_within(compare(w, run, [0]), "tiny")


def test_chain_full(cuda_lib):
    w = cpu_then_cuda("chain")
    run = CudaRun(w)
    assert not run.status.any()
    assert (w.accepted == -1).any()  # the no-op commit is exercised
    assert_within(compare(w, run, range(w.R)), "chain")


def test_binary_full(cuda_lib):
    w = cpu_then_cuda("binary")
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), "binary")


def test_wide_reduced_all_requests(cuda_lib):
    w = cpu_then_cuda("wide", R=12)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), "wide R=12")


def test_stress_reduced_all_requests(cuda_lib):
    w = cpu_then_cuda("stress", R=3)
    run = CudaRun(w)
    assert_within(compare(w, run, range(w.R)), "stress R=3")


@pytest.mark.parametrize("name,nsample", [("wide", 64), ("stress", 16)])
def test_full_size_sampled(cuda_lib, oracle_pool, name, nsample):
    """Full-size workload in the launch configuration the benchmark times;
    the oracle checks a sample of requests (all heads each), the first and
    last request among them, on a pool of worker processes."""
    cfg = wl.CONFIGS[name]
    w = wl.generate(cfg, device="cuda")
    run = CudaRun(w)
    assert not run.status.any()
    rng = np.random.default_rng(1234)
    reqs = sorted(set(rng.choice(w.R, nsample - 2, replace=False).tolist()) | {0, w.R - 1})
    assert_within(compare(w, run, reqs, pool=oracle_pool), name)


# ------------------------------------------------------------ trees and edges

def custom(trees, accepted, seed=77, H=4, dk=128, dv=128, qkv="bf16", alpha=(0.9, 0.999),
           beta=("sigmoid",), max_nodes=None, extra_slots=0):
    w = wl.assemble([np.asarray(t, np.int32) for t in trees], np.asarray(accepted, np.int32), H, dk,
                    dv, qkv, 0.05, alpha, beta, seed=seed, max_nodes=max_nodes,
                    extra_slots=extra_slots)
    return w.to("cuda")


def random_trees(rng, sizes):
    out = []
    for n in sizes:
        out.append(np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32)
                   if n else np.zeros(0, np.int32))
    return out


MIXED_SIZES = [1, 2, 5, 16, 17, 33, 64, 0, 48, 31]


def mixed_trees(rng):
    trees = random_trees(rng, MIXED_SIZES)
    trees.append(wl.chain_parents(64))                    # depth 64
    trees.append(np.full(64, -1, np.int32))               # 64 roots, depth 1
    trees.append(wl.width_tree_parents((3, 3, 3)))        # Table 2's widest shape
    trees.append(wl.branches_parents(8, 8))
    acc = [int(rng.integers(-1, len(t))) if len(t) else -1 for t in trees]
    acc[-1] = 63
    acc[-4] = 63
    return trees, acc


@pytest.mark.parametrize("flags", [0, binding.FLAG_FORCE_GENERIC])
def test_random_and_degenerate_trees(cuda_lib, flags):
    rng = np.random.default_rng(5)
    trees, acc = mixed_trees(rng)
    w = custom(trees, acc)
    run = CudaRun(w, flags=flags)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"mixed flags={flags}")


@pytest.mark.parametrize("alpha,beta", [((0.999999, 0.9999999), ("uniform", 0.9999, 0.99999)),
                                        ((0.5, 0.6), ("uniform", 1e-4, 2e-4)),
                                        ((0.8, 0.999), ("uniform", 0.05, 0.95))])
def test_gate_edges(cuda_lib, alpha, beta):
    rng = np.random.default_rng(9)
    trees, acc = mixed_trees(rng)
    w = custom(trees, acc, alpha=alpha, beta=beta, seed=31)
    run = CudaRun(w)
    assert_within(compare(w, run, range(w.R)), f"gates {alpha} {beta}")


@pytest.mark.parametrize("alpha,beta", [((1.0, 1.0), ("const", 1.0)),     # no decay, full writes
                                        ((0.9, 0.999), ("const", 0.0)),   # no writes: U = 0
                                        ((0.01, 0.05), ("uniform", 0.05, 0.95))])  # strong decay
def test_degenerate_gates_on_chains_and_trees(cuda_lib, alpha, beta):
    """Gates at the ends of their range, on 64-node chains (paths past the
    register-held length of 8) beside random trees: alpha at 1 (clamped to the
    largest float below 1), beta exactly 1 or 0, and decays that underflow
    gamma along a long chain."""
    rng = np.random.default_rng(23)
    trees = [wl.chain_parents(64), wl.chain_parents(9)] + random_trees(rng, [64, 33, 5])
    acc = [63, 8, int(rng.integers(0, 64)), 32, 0]
    w = custom(trees, acc, alpha=alpha, beta=beta, seed=37, H=3)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"gates {alpha} {beta}")


@pytest.mark.parametrize("max_nodes,sizes", [(16, [1, 7, 16, 9, 16, 3]), (32, [17, 32, 1, 30])])
def test_smaller_tree_capacity(cuda_lib, max_nodes, sizes):
    rng = np.random.default_rng(max_nodes)
    trees = random_trees(rng, sizes)
    acc = [len(t) - 1 for t in trees]
    w = custom(trees, acc, max_nodes=max_nodes, H=3)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"max_nodes={max_nodes}")


@pytest.mark.parametrize("sizes", [[5, 33], [40, 1, 63], [17], [64, 49]])
def test_key_rows_padded_past_the_batch(cuda_lib, sizes):
    """The key/query boxes cover each tree's rows rounded up to 16: the padding
    rows are the next request's (or zero fill past the batch's last node) and
    must not reach any output."""
    rng = np.random.default_rng(sum(sizes))
    trees = random_trees(rng, sizes)
    acc = [len(t) - 1 for t in trees]
    w = custom(trees, acc, H=2, max_nodes=64)
    assert int(w.node_offset[-1]) % 16 != 0  # the last tree reads past the batch
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"padding rows {sizes}")


@pytest.mark.parametrize("dk,dv,qkv", [(128, 128, "f32"), (48, 80, "bf16"), (16, 16, "bf16"),
                                       (128, 64, "bf16"), (3, 5, "f32")])
def test_generic_head_sizes(cuda_lib, dk, dv, qkv):
    rng = np.random.default_rng(dk + dv)
    trees = random_trees(rng, [9, 23, 1, 40])
    acc = [4, 22, 0, -1]
    w = custom(trees, acc, dk=dk, dv=dv, qkv=qkv, H=2)
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), f"dk={dk} dv={dv} {qkv}")


def test_deterministic(cuda_lib):
    w = cpu_then_cuda("wide", R=8)
    a = binding.TreeVerifier(w)
    a.verify()
    o1, u1 = a.o.clone(), a.U.clone()
    a.verify()
    torch.cuda.synchronize()
    assert torch.equal(o1, a.o) and torch.equal(u1, a.U)


# ------------------------------------------------------------ storeall comparator

def run_storeall(w, chunks=1):
    snaps = torch.empty(w.T, w.H, w.dv, w.dk, device="cuda", dtype=torch.float32)
    o = torch.full((w.T, w.H, w.dv), float("nan"), device="cuda")
    status = torch.zeros(w.R, device="cuda", dtype=torch.int32)
    node = w.node_offset.cpu().tolist()
    bounds = np.linspace(0, w.R, chunks + 1).astype(int)
    S0 = w.state.cpu()
    for c in range(chunks):
        r0, r1 = int(bounds[c]), int(bounds[c + 1])
        if r1 == r0:
            continue
        b = binding.make_batch(node_offset=w.node_offset[r0:], parent=w.parent, q=w.q, k=w.k,
                               v=w.v, alpha=w.alpha, beta=w.beta, state=w.state,
                               state_slot=w.state_slot[r0:], o=o, U=o, status=status[r0:],
                               max_nodes=w.max_nodes)
        b.R = r1 - r0
        sub = snaps[node[r0]:node[r1]]
        binding.treewy_storeall_verify(b, sub)
        binding.treewy_storeall_commit(b, sub, w.accepted[r0:])
    torch.cuda.synchronize()
    return snaps, o, status, S0


@pytest.mark.parametrize("name,R,chunks", [("binary", 6, 1), ("stress", 2, 2), ("wide", 5, 3),
                                           ("tiny", None, 1)])
def test_storeall_matches_oracle(cuda_lib, name, R, chunks):
    w = cpu_then_cuda(name, R=R)
    snaps, o, status, S0 = run_storeall(w, chunks)
    assert not status.any()
    node = w.node_offset.cpu().numpy()
    for r in range(w.R):
        lo, hi, S0r, ref = oracle_request(w, r, S0)
        scale_s = np.abs(ref.states).max()
        assert np.abs(np32(snaps[lo:hi]) - ref.states).max() <= 1e-3 * scale_s
        assert np.abs(np32(o[lo:hi]) - ref.o).max() <= 2e-3 * np.abs(ref.o).max()
        S_ref = orc.commit_request(S0r, ref, int(w.accepted[r]))
        S_gpu = np32(w.state[int(w.state_slot[r])])
        assert np.abs(S_gpu - S_ref).max() <= 1e-3 * np.abs(S_ref).max()


@pytest.mark.parametrize("qkv", ["bf16", "f32"])
def test_storeall_tree_shapes(cuda_lib, qkv):
    """The 128 x 128 comparator walks each tree in DFS pre-order and reloads a
    parent's snapshot only after a branch point: a 64-deep chain, 64 nodes
    off S0, the (3,3,3) width tree, 8 branches of 8, random trees and a
    single node, against the oracle's per-node states."""
    rng = np.random.default_rng(29)
    trees = [wl.chain_parents(64), np.full(64, -1, np.int32), wl.width_tree_parents((3, 3, 3)),
             wl.branches_parents(8, 8), np.zeros(1, np.int32) - 1] + random_trees(rng, [17, 40, 64])
    acc = [int(rng.integers(-1, len(t))) for t in trees]
    w = custom(trees, acc, H=2, qkv=qkv, max_nodes=64)
    snaps, o, status, S0 = run_storeall(w, 2)
    assert not status.any()
    for r in range(w.R):
        lo, hi, S0r, ref = oracle_request(w, r, S0)
        scale_s = np.abs(ref.states).max()
        assert np.abs(np32(snaps[lo:hi]) - ref.states).max() <= 1e-3 * scale_s, r
        assert np.abs(np32(o[lo:hi]) - ref.o).max() <= 2e-3 * np.abs(ref.o).max(), r
        S_ref = orc.commit_request(S0r, ref, int(w.accepted[r]))
        assert np.abs(np32(w.state[int(w.state_slot[r])]) - S_ref).max() <= 1e-3 * np.abs(S_ref).max()


def test_storeall_and_treewy_commit_agree(cuda_lib):
    w1 = cpu_then_cuda("binary", R=10)
    w2 = cpu_then_cuda("binary", R=10)
    CudaRun(w1)
    run_storeall(w2)
    d = (w1.state - w2.state).abs().max().item()
    assert d <= 1e-3 * w2.state.abs().max().item()


# ------------------------------------------------------------ device-side errors

def test_bad_inputs_set_status_and_spare_others(cuda_lib):
    rng = np.random.default_rng(3)
    trees = random_trees(rng, [10, 12, 20, 8, 9])
    trees[1][5] = 7                       # parent after child
    acc = [3, 2, 1, 8, 0]                 # request 3: accepted outside its 8-node tree
    w = custom(trees, acc, max_nodes=64, extra_slots=2)
    slots = w.state_slot.clone()
    slots[4] = w.num_slots                # outside the pool
    w.state_slot.copy_(slots)
    tv = binding.TreeVerifier(w, max_nodes=16)  # request 2 (20 nodes) exceeds it
    tv.o.fill_(float("nan"))
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
    node = w.node_offset.cpu().tolist()
    for r in (1, 2, 4):
        assert torch.isnan(tv.o[node[r]:node[r + 1]]).all()
    for r in (1, 2, 3):   # state untouched where commit refused
        s = int(w.state_slot[r])
        assert torch.equal(w.state[s], S_before[s])
    # request 0 is still correct
    lo, hi, S0, ref = oracle_request(w, 0, S_before.cpu())
    assert np.abs(np32(tv.o[lo:hi]) - ref.o).max() <= 2e-3 * np.abs(ref.o).max()


# ------------------------------------------------------------ CUDA graphs

def test_graph_replay_matches_eager(cuda_lib):
    """Verify + commit captured once in a CUDA graph and replayed: the replay
    matches the oracle within the tolerances and the eager launches bit for
    bit, on a ragged tree batch (the case the pages say vLLM could not
    capture)."""
    w_eager = cpu_then_cuda("wide", R=16)
    run = CudaRun(w_eager)
    w = cpu_then_cuda("wide", R=16)
    S0 = w.state.clone()
    tv = binding.TreeVerifier(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tv.verify(s)  # warm-up outside capture (first-call set-up)
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
    assert_within(compare(w, replay, range(w.R)), "graph replay")
    assert torch.equal(tv.o.cpu(), torch.from_numpy(run.o))
    assert torch.equal(w.state.cpu(), run.S_after.cpu())


def test_batch_of_empty_trees(cuda_lib):
    """T = 0: every per-node tensor is empty (NULL data pointers); verify,
    commit, the fused path and storeall accept it, a = -1 leaves the states
    alone, and an accepted index in an empty tree is reported."""
    w = custom([np.zeros(0, np.int32)] * 3, [-1, -1, -1], H=2, extra_slots=1)
    assert w.T == 0
    S0 = w.state.clone()
    tv = binding.TreeVerifier(w)
    tv.verify()
    tv.commit()
    binding.treewy_commit_verify(tv.batch, w.accepted, tv.batch)
    snaps = torch.empty(0, w.H, w.dv, w.dk, device="cuda")
    binding.treewy_storeall_verify(tv.batch, snaps)
    binding.treewy_storeall_commit(tv.batch, snaps, w.accepted)
    torch.cuda.synchronize()
    assert not tv.status.any()
    assert torch.equal(w.state, S0)
    bad = torch.tensor([0, -1, -1], dtype=torch.int32, device="cuda")
    tv.commit(bad)
    torch.cuda.synchronize()
    assert tv.status.cpu().tolist() == [binding.STATUS_BAD_ACCEPTED, 0, 0]
    assert torch.equal(w.state, S0)
