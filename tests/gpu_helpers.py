"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and run the oracle on the same seeded inputs, then compare element by element.

Tolerances: max-abs error of o at most 2e-3 x max|o_ref| and of the committed
state at most 1e-3 x max|S_ref|, both taken over the compared set; the
pseudo-values U at most 2e-3 x max|U_ref|; path decays gamma to 1e-5
relative to max(gamma_ref, 2^-126): gamma is an fp32 output, so a decay
below fp32's smallest normal number underflows there (a product of 64 gates
of ~0.03 is ~1e-97) and is compared against that bound instead.
"""
from __future__ import annotations

import numpy as np
import torch

from gdn_speculative_tree_gb300 import binding
from oracle import gdn_tree_oracle as orc

O_TOL = 2e-3
S_TOL = 1e-3
U_TOL = 2e-3
G_TOL = 1e-5
FLT_MIN = 2.0 ** -126  # smallest normal fp32 number


def np32(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu").to(torch.float32).numpy()


class CudaRun:
    """Verify + commit of one Workload on the GPU (Workload tensors on cuda).

    Keeps a CPU copy of the state pool as it was before the in-place commit.
    """

    def __init__(self, wl, flags: int = 0, accepted=None, max_nodes=None, commit=True):
        self.S0_pool = wl.state.cpu()
        self.tv = binding.TreeVerifier(wl, flags=flags, max_nodes=max_nodes)
        self.tv.verify()
        if commit:
            self.tv.commit(accepted)
        torch.cuda.synchronize()
        self.o = np32(self.tv.o)
        self.U = np32(self.tv.U)
        self.gamma = np32(self.tv.gamma)
        self.status = self.tv.status.cpu().numpy()
        self.S_after = wl.state


def oracle_request(wl, r, S0_pool):
    node = wl.node_offset.cpu().numpy()
    lo, hi = int(node[r]), int(node[r + 1])
    S0 = np32(S0_pool[int(wl.state_slot[r])])
    parent = wl.parent[lo:hi].cpu().numpy()
    res = orc.verify_request(S0, parent, np32(wl.q[lo:hi]), np32(wl.k[lo:hi]), np32(wl.v[lo:hi]),
                             np32(wl.alpha[lo:hi]), np32(wl.beta[lo:hi]))
    return lo, hi, S0, res


def _oracle_results(wl, run, requests, acc, pool):
    """(lo, hi, S0, o, U, gamma, S_commit) per request: one by one here, or as
    jobs of an oracle process pool."""
    node = wl.node_offset.cpu().numpy()
    slot = wl.state_slot.cpu().numpy()
    requests = list(requests)
    if pool is None:
        for r in requests:
            lo, hi, S0, ref = oracle_request(wl, r, run.S0_pool)
            yield lo, hi, S0, ref.o, ref.U, ref.gamma, orc.commit_request(S0, ref, int(acc[r]))
        return
    from oracle import pool as opool
    jobs = opool.jobs_from_arrays(node, wl.parent.cpu().numpy(), np32(wl.q), np32(wl.k), np32(wl.v),
                                  np32(wl.alpha), np32(wl.beta), np32(run.S0_pool), slot, acc,
                                  requests)
    for r, (o, U, g, S_c) in zip(requests, pool.map(jobs)):
        lo, hi = int(node[r]), int(node[r + 1])
        yield lo, hi, None, o, U, g, S_c


def compare(wl, run: CudaRun, requests, accepted=None, check_commit=True, pool=None):
    """Error ratios of o, U, gamma and the committed state over `requests`
    (``pool``: an oracle.pool.OraclePool that runs the requests in parallel)."""
    acc = (wl.accepted if accepted is None else accepted).cpu().numpy()
    slot = wl.state_slot.cpu().numpy()
    o_err = o_max = u_err = u_max = g_err = s_err = s_max = 0.0
    for r, (lo, hi, _S0, ref_o, ref_U, ref_g, S_ref) in zip(
            list(requests), _oracle_results(wl, run, requests, acc, pool)):
        o_err = max(o_err, float(np.abs(run.o[lo:hi] - ref_o).max(initial=0)))
        o_max = max(o_max, float(np.abs(ref_o).max(initial=0)))
        u_err = max(u_err, float(np.abs(run.U[lo:hi] - ref_U).max(initial=0)))
        u_max = max(u_max, float(np.abs(ref_U).max(initial=0)))
        if hi > lo:
            g_err = max(g_err, float((np.abs(run.gamma[lo:hi] - ref_g) /
                                      np.maximum(ref_g, FLT_MIN)).max()))
        if check_commit:
            S_gpu = np32(run.S_after[int(slot[r])])
            s_err = max(s_err, float(np.abs(S_gpu - S_ref).max()))
            s_max = max(s_max, float(np.abs(S_ref).max()))
    return {"o": o_err / max(o_max, 1e-30), "U": u_err / max(u_max, 1e-30), "gamma": g_err,
            "S": s_err / max(s_max, 1e-30) if check_commit else 0.0, "o_abs": o_err, "S_abs": s_err}


def assert_within(res, label=""):
    assert res["o"] <= O_TOL, (label, res)
    assert res["S"] <= S_TOL, (label, res)
    assert res["U"] <= U_TOL, (label, res)
    assert res["gamma"] <= G_TOL, (label, res)
