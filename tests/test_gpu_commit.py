"""GPU checks of the two commit kernels: the bulk-copy kernel (dk = dv = 128,
state tile staged by TMA) against the oracle and against the portable
register-streaming kernel (TREEWY_FLAG_FORCE_GENERIC).  Both accumulate
gamma_a S0 + sum_j c_j u_j k_j^T in f32 in the same order (path from the
accepted node to the root) and round once, so their states are bit-identical.
"""
import numpy as np
import pytest
import torch

from gdn_speculative_tree_gb300 import binding
from gdn_speculative_tree_gb300 import workloads as wl
from tests.gpu_helpers import CudaRun, assert_within, compare

pytestmark = pytest.mark.gpu


def trees_with_long_paths(rng):
    trees = [np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32)
             for n in (1, 7, 16, 33, 64, 20)]
    trees += [wl.chain_parents(64), wl.chain_parents(17), wl.branches_parents(8, 8)]
    acc = [0, 6, -1, 32, 63, 19, 63, 16, 63]
    return trees, acc


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_commit_kernels_bit_identical(cuda_lib, state_dtype):
    rng = np.random.default_rng(19)
    trees, acc = trees_with_long_paths(rng)

    def make():
        return wl.assemble(trees, np.asarray(acc, np.int32), 8, 128, 128, "bf16", 0.05, (0.8, 0.999),
                           ("sigmoid",), seed=3, max_nodes=64, extra_slots=2,
                           state_dtype=state_dtype).to("cuda")

    wa, wb = make(), make()
    ta = binding.TreeVerifier(wa)
    tb = binding.TreeVerifier(wb, flags=binding.FLAG_FORCE_GENERIC)
    ta.verify()
    tb.verify()
    torch.cuda.synchronize()
    assert torch.equal(ta.U, tb.U) or (ta.U - tb.U).abs().max().item() <= 1e-3 * tb.U.abs().max().item()
    # the same U into both commits so that only the commit kernels differ
    tb.U.copy_(ta.U)
    ta.commit()
    tb.commit()
    torch.cuda.synchronize()
    assert not ta.status.any() and not tb.status.any()
    assert torch.equal(wa.state, wb.state)


def test_commit_tma_wide_oracle(cuda_lib):
    w = wl.generate(wl.CONFIGS["wide"], R=16).to("cuda")
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), "wide R=16, bulk-copy commit")


def test_commit_tma_f32_keys(cuda_lib):
    """f32 q/k/v (CUDA-core verify) with the bulk-copy commit."""
    rng = np.random.default_rng(2)
    trees, acc = trees_with_long_paths(rng)
    w = wl.assemble(trees, np.asarray(acc, np.int32), 2, 128, 128, "f32", 0.05, (0.9, 0.999),
                    ("sigmoid",), seed=4, max_nodes=64).to("cuda")
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), "f32 keys")
