"""GPU parity of a bf16 state pool (TREEWY_FLAG_STATE_BF16) against the oracle
on the same seeded inputs: verification, commit, the fused commit-into-verify,
both kernels (tensor-core and CUDA-core) and the scalar commit path.

Tolerances.  o and U as for an fp32 pool (max-abs error at most 2e-3 of the
largest reference value): verification reads the bf16 S0 as exact values.
The committed state is a bf16 number, so per element
    |S_gpu - S_ref| <= 2^-8 |S_ref| + 1e-3 max|S_ref|,
2^-8 being the relative rounding bound of 8 significant bits (round to
nearest) and 1e-3 max|S_ref| the fp32 pool's bound for the arithmetic before
the rounding; S_ref is the oracle's unrounded S_a.
"""
import numpy as np
import pytest
import torch

from gdn_speculative_tree_gb300 import binding
from gdn_speculative_tree_gb300 import workloads as wl
from oracle import gdn_tree_oracle as orc
from tests.gpu_helpers import CudaRun, FLT_MIN, O_TOL, U_TOL, G_TOL, np32, oracle_request

pytestmark = pytest.mark.gpu

S_REL = 2.0 ** -8
S_ABS = 1e-3


def random_trees(rng, sizes):
    return [np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32)
            if n else np.zeros(0, np.int32) for n in sizes]


def custom(trees, accepted, seed=91, H=4, dk=128, dv=128, qkv="bf16", extra_slots=2):
    w = wl.assemble([np.asarray(t, np.int32) for t in trees], np.asarray(accepted, np.int32), H, dk,
                    dv, qkv, 0.05, (0.9, 0.999), ("sigmoid",), seed=seed, max_nodes=64,
                    extra_slots=extra_slots, state_dtype="bf16")
    return w.to("cuda")


def check_run(w, run, requests):
    assert w.state.dtype == torch.bfloat16
    acc = w.accepted.cpu().numpy()
    slot = w.state_slot.cpu().numpy()
    o_err = o_max = u_err = u_max = g_err = 0.0
    for r in requests:
        lo, hi, S0, ref = oracle_request(w, r, run.S0_pool)
        if hi > lo:
            o_err = max(o_err, float(np.abs(run.o[lo:hi] - ref.o).max()))
            o_max = max(o_max, float(np.abs(ref.o).max()))
            u_err = max(u_err, float(np.abs(run.U[lo:hi] - ref.U).max()))
            u_max = max(u_max, float(np.abs(ref.U).max()))
            g_err = max(g_err, float((np.abs(run.gamma[lo:hi] - ref.gamma) /
                                      np.maximum(ref.gamma, FLT_MIN)).max()))
        S_ref = orc.commit_request(S0, ref, int(acc[r]))
        S_gpu = np32(w.state[int(slot[r])]).astype(np.float64)
        bound = S_REL * np.abs(S_ref) + S_ABS * np.abs(S_ref).max()
        assert np.all(np.abs(S_gpu - S_ref) <= bound), (r, float(np.abs(S_gpu - S_ref).max()))
        if int(acc[r]) < 0:
            assert np.array_equal(S_gpu, S0)
    assert o_err <= O_TOL * o_max, (o_err, o_max)
    assert u_err <= U_TOL * u_max, (u_err, u_max)
    assert g_err <= G_TOL, g_err


@pytest.mark.parametrize("flags", [0, binding.FLAG_FORCE_GENERIC])
def test_bf16_state_mixed_trees(cuda_lib, flags):
    rng = np.random.default_rng(12)
    trees = random_trees(rng, [1, 2, 5, 16, 17, 33, 64, 0, 48, 31])
    trees.append(wl.chain_parents(64))          # 64-long accepted path: 4 commit passes
    trees.append(np.full(64, -1, np.int32))
    trees.append(wl.width_tree_parents((3, 3, 3)))
    acc = [int(rng.integers(-1, len(t))) if len(t) else -1 for t in trees]
    acc[10] = 63
    acc[3] = -1
    w = custom(trees, acc)
    run = CudaRun(w, flags=flags)
    assert not run.status.any()
    check_run(w, run, range(w.R))


@pytest.mark.parametrize("dk,dv,qkv", [(128, 128, "f32"), (48, 80, "bf16"), (3, 5, "f32"),
                                       (16, 16, "bf16")])
def test_bf16_state_generic_head_sizes(cuda_lib, dk, dv, qkv):
    """CUDA-core verify; commit through the 8-wide vector path (dk % 8 == 0)
    and the scalar path (dk = 3), including a path longer than one pass."""
    rng = np.random.default_rng(dk * 7 + dv)
    trees = random_trees(rng, [9, 23, 1, 40]) + [wl.chain_parents(40)]
    acc = [4, 22, 0, -1, 39]
    w = custom(trees, acc, dk=dk, dv=dv, qkv=qkv, H=2)
    run = CudaRun(w)
    assert not run.status.any()
    check_run(w, run, range(w.R))


def test_bf16_state_wide_full_size_sampled(cuda_lib):
    cfg = wl.CONFIGS["wide"]
    w = wl.generate(cfg, device="cuda", state_dtype="bf16")
    run = CudaRun(w)
    assert not run.status.any()
    rng = np.random.default_rng(77)
    reqs = sorted(set(rng.choice(w.R, 4, replace=False).tolist()) | {w.R - 1})
    check_run(w, run, reqs)


def test_bf16_state_fused_two_rounds(cuda_lib):
    """treewy_commit_verify with a bf16 pool: the oracle commits the previous
    round, rounds S_a to bf16 (the value the pool holds) and verifies the next
    round from it."""
    rng = np.random.default_rng(63)
    prev_trees = random_trees(rng, [12, 40, 64, 5, 30, 17, 9])
    prev_trees.append(wl.chain_parents(64))     # a 64-entry path: several staged segments
    next_trees = random_trees(rng, [20, 0, 33, 64, 1, 17, 48, 10])
    accepted = [5, 39, -1, 4, 29, 0, 8, 63]
    R = len(prev_trees)
    prev = wl.assemble(prev_trees, np.asarray(accepted, np.int32), 4, 128, 128, "bf16", 0.05,
                       (0.9, 0.999), ("sigmoid",), seed=5, max_nodes=64, extra_slots=3,
                       state_dtype="bf16").to("cuda")
    nxt = wl.assemble(next_trees, np.full(R, -1, np.int32), 4, 128, 128, "bf16", 0.05,
                      (0.9, 0.999), ("sigmoid",), seed=6, max_nodes=64, extra_slots=3,
                      state_dtype="bf16").to("cuda")
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
    pn = prev.node_offset.cpu().numpy()
    nn = nxt.node_offset.cpu().numpy()
    o_err = o_max = 0.0
    for r in range(R):
        slot = int(prev.state_slot[r])
        S0 = np32(S0_pool[slot]).astype(np.float64)
        lo, hi = int(pn[r]), int(pn[r + 1])
        ref_prev = orc.verify_request(S0, prev.parent[lo:hi].cpu().numpy(), np32(prev.q[lo:hi]),
                                      np32(prev.k[lo:hi]), np32(prev.v[lo:hi]),
                                      np32(prev.alpha[lo:hi]), np32(prev.beta[lo:hi]))
        S_a = orc.commit_request(S0, ref_prev, accepted[r])
        S_gpu = np32(prev.state[slot]).astype(np.float64)
        bound = S_REL * np.abs(S_a) + S_ABS * np.abs(S_a).max()
        assert np.all(np.abs(S_gpu - S_a) <= bound), r
        S_pool = orc.commit_request(S0, ref_prev, accepted[r], state_dtype="bf16")
        lo2, hi2 = int(nn[r]), int(nn[r + 1])
        if hi2 == lo2:
            continue
        ref = orc.verify_request(S_pool, nxt.parent[lo2:hi2].cpu().numpy(), np32(nxt.q[lo2:hi2]),
                                 np32(nxt.k[lo2:hi2]), np32(nxt.v[lo2:hi2]),
                                 np32(nxt.alpha[lo2:hi2]), np32(nxt.beta[lo2:hi2]))
        o_err = max(o_err, float(np.abs(o[lo2:hi2] - ref.o).max()))
        o_max = max(o_max, float(np.abs(ref.o).max()))
    assert o_err <= O_TOL * o_max, (o_err, o_max)


@pytest.mark.parametrize("max_nodes", [16, 32])
def test_bf16_state_fused_small_buckets(cuda_lib, max_nodes):
    """treewy_commit_verify with a bf16 pool on the 16- and 32-node capacity
    buckets, with accepted paths of one and two 16-entry segments (a chain as
    long as the capacity): the committed bf16 state and the next round's
    outputs against the oracle."""
    rng = np.random.default_rng(100 + max_nodes)
    prev_trees = random_trees(rng, [max_nodes // 2, 3, max_nodes - 1, 1])
    prev_trees.append(wl.chain_parents(max_nodes))
    next_trees = random_trees(rng, [max_nodes, 5, 0, max_nodes // 2, 2])
    accepted = [max_nodes // 2 - 1, -1, max_nodes - 2, 0, max_nodes - 1]
    R = len(prev_trees)
    prev = wl.assemble(prev_trees, np.asarray(accepted, np.int32), 3, 128, 128, "bf16", 0.05,
                       (0.9, 0.999), ("sigmoid",), seed=21, max_nodes=max_nodes, extra_slots=2,
                       state_dtype="bf16").to("cuda")
    nxt = wl.assemble(next_trees, np.full(R, -1, np.int32), 3, 128, 128, "bf16", 0.05,
                      (0.9, 0.999), ("sigmoid",), seed=22, max_nodes=max_nodes, extra_slots=2,
                      state_dtype="bf16").to("cuda")
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
    pn = prev.node_offset.cpu().numpy()
    nn = nxt.node_offset.cpu().numpy()
    o_err = o_max = 0.0
    for r in range(R):
        slot = int(prev.state_slot[r])
        S0 = np32(S0_pool[slot]).astype(np.float64)
        lo, hi = int(pn[r]), int(pn[r + 1])
        ref_prev = orc.verify_request(S0, prev.parent[lo:hi].cpu().numpy(), np32(prev.q[lo:hi]),
                                      np32(prev.k[lo:hi]), np32(prev.v[lo:hi]),
                                      np32(prev.alpha[lo:hi]), np32(prev.beta[lo:hi]))
        S_a = orc.commit_request(S0, ref_prev, accepted[r])
        S_gpu = np32(prev.state[slot]).astype(np.float64)
        bound = S_REL * np.abs(S_a) + S_ABS * np.abs(S_a).max()
        assert np.all(np.abs(S_gpu - S_a) <= bound), r
        S_pool = orc.commit_request(S0, ref_prev, accepted[r], state_dtype="bf16")
        lo2, hi2 = int(nn[r]), int(nn[r + 1])
        if hi2 == lo2:
            continue
        ref = orc.verify_request(S_pool, nxt.parent[lo2:hi2].cpu().numpy(), np32(nxt.q[lo2:hi2]),
                                 np32(nxt.k[lo2:hi2]), np32(nxt.v[lo2:hi2]),
                                 np32(nxt.alpha[lo2:hi2]), np32(nxt.beta[lo2:hi2]))
        o_err = max(o_err, float(np.abs(o[lo2:hi2] - ref.o).max()))
        o_max = max(o_max, float(np.abs(ref.o).max()))
    assert o_err <= O_TOL * o_max, (o_err, o_max)


def test_bf16_state_fused_equals_separate_calls(cuda_lib):
    """Fused and separate paths store the same bf16 state up to one bf16 step
    (the fused kernel forms the rank-|path| update on the tensor cores, c_j u_j
    as two bf16 terms accumulated in fp32, the separate commit with fp32 FMAs;
    both round once to bf16) and give the same outputs."""
    cfg = wl.CONFIGS["wide"]
    trees, acc = wl.make_trees(cfg, R=10)
    rng = np.random.default_rng(4)
    nxt_trees = random_trees(rng, [int(rng.integers(16, 65)) for _ in range(10)])

    def pair():
        p = wl.assemble(trees, acc, 8, 128, 128, "bf16", 0.05, (0.9, 0.999), ("sigmoid",), seed=8,
                        max_nodes=64, extra_slots=2, state_dtype="bf16").to("cuda")
        n = wl.assemble(nxt_trees, np.full(10, -1, np.int32), 8, 128, 128, "bf16", 0.05,
                        (0.9, 0.999), ("sigmoid",), seed=9, max_nodes=64, extra_slots=2,
                        state_dtype="bf16").to("cuda")
        n.state = p.state
        n.state_slot = p.state_slot
        return p, n

    pa, na = pair()
    pb, nb = pair()
    ta = binding.TreeVerifier(pa)
    ta.verify()
    tna = binding.TreeVerifier(na)
    binding.treewy_commit_verify(ta.batch, pa.accepted, tna.batch)
    tb = binding.TreeVerifier(pb)
    tb.verify()
    tb.commit()
    tnb = binding.TreeVerifier(nb)
    tnb.verify()
    torch.cuda.synchronize()
    assert not tna.status.any() and not tnb.status.any()
    ds = (pa.state.float() - pb.state.float()).abs()
    Sb = pb.state.float().abs()
    # at most one bf16 step apart (the two f32 values may round to neighbours),
    # or, where S_a is near zero after cancellation, within the committed
    # state tolerance of each other
    assert bool((ds <= 2.0 ** -7 * Sb + S_ABS * Sb.max()).all())
    do = (tna.o - tnb.o).abs().max().item()
    assert do <= 1e-3 * tnb.o.abs().max().item(), do


@pytest.mark.parametrize("dk,dv,qkv", [(128, 128, "f32"), (64, 48, "bf16")])
def test_bf16_state_fused_fallback_shapes(cuda_lib, dk, dv, qkv):
    """Shapes outside the tensor-core path: treewy_commit_verify runs the
    commit and the verification back to back; results as the oracle's
    commit, rounding to bf16, then verification."""
    rng = np.random.default_rng(dk + dv)
    prev_trees = random_trees(rng, [7, 20, 3])
    next_trees = random_trees(rng, [5, 0, 9])
    accepted = [6, 19, -1]
    prev = wl.assemble(prev_trees, np.asarray(accepted, np.int32), 2, dk, dv, qkv, 0.05,
                       (0.9, 0.999), ("sigmoid",), seed=12, max_nodes=64, extra_slots=1,
                       state_dtype="bf16").to("cuda")
    nxt = wl.assemble(next_trees, np.full(3, -1, np.int32), 2, dk, dv, qkv, 0.05, (0.9, 0.999),
                      ("sigmoid",), seed=13, max_nodes=64, extra_slots=1,
                      state_dtype="bf16").to("cuda")
    nxt.state = prev.state
    nxt.state_slot = prev.state_slot
    tp = binding.TreeVerifier(prev)
    tp.verify()
    torch.cuda.synchronize()
    S0_pool = prev.state.cpu()
    tn = binding.TreeVerifier(nxt)
    binding.treewy_commit_verify(tp.batch, prev.accepted, tn.batch)
    torch.cuda.synchronize()
    assert not tn.status.any()
    pn, nn = prev.node_offset.cpu().numpy(), nxt.node_offset.cpu().numpy()
    o = np32(tn.o)
    for r in range(3):
        slot = int(prev.state_slot[r])
        S0 = np32(S0_pool[slot]).astype(np.float64)
        lo, hi = int(pn[r]), int(pn[r + 1])
        ref_prev = orc.verify_request(S0, prev.parent[lo:hi].cpu().numpy(), np32(prev.q[lo:hi]),
                                      np32(prev.k[lo:hi]), np32(prev.v[lo:hi]),
                                      np32(prev.alpha[lo:hi]), np32(prev.beta[lo:hi]))
        S_a = orc.commit_request(S0, ref_prev, accepted[r])
        S_gpu = np32(prev.state[slot]).astype(np.float64)
        assert np.all(np.abs(S_gpu - S_a) <= S_REL * np.abs(S_a) + S_ABS * np.abs(S_a).max()), r
        lo2, hi2 = int(nn[r]), int(nn[r + 1])
        if hi2 == lo2:
            continue
        S_pool = orc.commit_request(S0, ref_prev, accepted[r], state_dtype="bf16")
        ref = orc.verify_request(S_pool, nxt.parent[lo2:hi2].cpu().numpy(), np32(nxt.q[lo2:hi2]),
                                 np32(nxt.k[lo2:hi2]), np32(nxt.v[lo2:hi2]),
                                 np32(nxt.alpha[lo2:hi2]), np32(nxt.beta[lo2:hi2]))
        assert np.abs(o[lo2:hi2] - ref.o).max() <= O_TOL * np.abs(ref.o).max(), r
