"""Plain fp64 CPU oracle for TreeWY speculative verification of Gated DeltaNet.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import or run this module.
The product path (the CUDA library and its Python binding) never calls it and
shares no code with it; the only thing both sides share is the seeded input
generator, which holds none of the method's arithmetic.

What it computes is the definition, not the fast method.  For every request
and value head it walks the draft tree node by node (parents precede
children) and applies the gated delta rule to the parent's state:

    S_n = alpha_n * S_par (I - beta_n k_n k_n^T) + beta_n v_n k_n^T,
    o_n = S_n q_n,

where S_par is the committed state S0 for a node that hangs off it (parent
-1) and the parent's state otherwise.  Sources:

* gated delta rule and read-out: "TreeWY: Speculative Verification for Gated
  DeltaNet Hybrids", §1 "Background", Eq. (1); the technical review of that
  paper (zhongzhuzhou.org, 2026-09-05), §2.4, Eq. (3), which prints the
  bracket that the paper's text extraction lost;
* a node's state depends on its root-to-node path only (review §3.2, "not
  siblings, not descendants"); the committed state after accepting node a
  is S_a, and S0 unchanged when nothing is accepted (paper §3 "Reconstruct
  on commit"; review §3.3, Eq. (6));
* the pseudo-value that the fast method stores instead of states is, by its
  definition, u_n = beta_n (v_n - alpha_n S_par k_n) (paper §3 "Key rewrite";
  review §3.1, Eq. (4));
* the cumulative decay gamma_n is the product of alpha over the root-to-n path,
  n included (paper §3 Eq. (2) text "cumulative decay from S0 to t"; review
  §3.2, Algorithm step 1).

The snapshot-per-node comparator ("storeall", paper §2 approach (i)) keeps
exactly the per-node states S_n that this walk produces, and rolls back by
selecting S_a; the oracle returns those states for it.

Products and sums are numpy fp64 (matrix-vector products via einsum over the
independent heads of one request: a library primitive applied per head).
Parity: pinned by the tests in tests/test_oracle_pins.py (closed form of the
pages solved by dense LU on every topology with N <= 5, chain equals the
sequential token loop, sibling/branch invariance, beta = 0, the exact-write
case beta = alpha = 1, and hand-derived values in tests/golden/).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional, Sequence

import numpy as np


@dataclass
class RequestResult:
    """Oracle outputs for one request (all arrays fp64).

    o:      [N][H][dv] per-node outputs o_n = S_n q_n
    U:      [N][H][dv] pseudo-values u_n = beta_n (v_n - alpha_n S_par k_n)
    gamma:  [N][H]     cumulative path decays
    states: [N][H][dv][dk] per-node states S_n (the storeall snapshots)
    """
    o: np.ndarray
    U: np.ndarray
    gamma: np.ndarray
    states: np.ndarray


def check_tree(parent: Sequence[int]) -> None:
    """A draft tree is valid when every parent index is -1 or an earlier node."""
    for n, p in enumerate(parent):
        if not (-1 <= int(p) < n):
            raise ValueError(f"node {n} has parent {p}; parents must precede children")


def verify_request(S0: np.ndarray, parent: Sequence[int], q: np.ndarray, k: np.ndarray,
                   v: np.ndarray, alpha: np.ndarray, beta: np.ndarray) -> RequestResult:
    """Walk one request's draft tree with the gated delta rule (all heads at once).

    S0: [H][dv][dk]; parent: [N]; q, k: [N][H][dk]; v: [N][H][dv];
    alpha, beta: [N][H].  Every array is converted to fp64.
    """
    check_tree(parent)
    S0 = np.asarray(S0, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    alpha = np.asarray(alpha, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    N = len(parent)
    H, dv, dk = S0.shape
    states = np.empty((N, H, dv, dk))
    o = np.empty((N, H, dv))
    U = np.empty((N, H, dv))
    gamma = np.empty((N, H))
    for n in range(N):
        p = int(parent[n])
        S_par = S0 if p < 0 else states[p]
        a = alpha[n][:, None, None]
        b = beta[n][:, None, None]
        kn = k[n]
        # what the parent state predicts for this key: S_par k_n
        pred = np.einsum("hij,hj->hi", S_par, kn)
        # gated delta rule: alpha S_par (I - beta k k^T) + beta v k^T
        S_n = a * (S_par - b * pred[:, :, None] * kn[:, None, :]) + b * v[n][:, :, None] * kn[:, None, :]
        states[n] = S_n
        o[n] = np.einsum("hij,hj->hi", S_n, q[n])
        # pseudo-value (definition): beta (v - alpha S_par k)
        U[n] = beta[n][:, None] * (v[n] - alpha[n][:, None] * pred)
        # cumulative decay over the root-to-n path, n included
        gamma[n] = alpha[n] * (1.0 if p < 0 else gamma[p])
    return RequestResult(o=o, U=U, gamma=gamma, states=states)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value, ties to even.

    bfloat16 has the binary32 exponent range and 8 significant bits.  Writing
    x = m 2^e with 1/2 <= |m| < 1, its neighbours in bfloat16 are the
    multiples of 2^(e-8), so the nearest one is rint(m 2^8) 2^(e-8), with
    numpy's rint rounding halves to even.  The rounding is taken once, from
    fp64 (no intermediate fp32).  Only normal-range values occur here;
    anything below the smallest normal bfloat16 or above the largest finite
    one raises.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    nz = x != 0
    if np.any(nz & ((e < -125) | (e > 128))) or not np.all(np.isfinite(x)):
        raise ValueError("value outside the normal bfloat16 range")
    out = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    if np.any(np.isinf(out)):
        raise ValueError("value rounds past the largest finite bfloat16")
    return out


def commit_request(S0: np.ndarray, result: RequestResult, accepted: int,
                   state_dtype: str = "f32") -> np.ndarray:
    """The state that becomes the next round's S0: S_a, or S0 when a = -1.

    With a bf16 state pool (the serving dtype of the GDN state, TreeWY paper
    §2 "The memory problem": 2 bytes per element) the committed value is S_a
    rounded to the nearest bf16 (ties to even); S0 of a bf16 pool is already
    a bf16 value and is returned unchanged for a = -1.
    """
    a = int(accepted)
    if a < 0:
        return np.array(S0, dtype=np.float64, copy=True)
    if a >= result.states.shape[0]:
        raise ValueError(f"accepted node {a} outside the tree")
    S_a = result.states[a].copy()
    if state_dtype == "bf16":
        return round_to_bf16(S_a)
    if state_dtype != "f32":
        raise ValueError(f"state_dtype {state_dtype!r}")
    return S_a


def verify_batch(node_offset: np.ndarray, parent: np.ndarray, q: np.ndarray, k: np.ndarray,
                 v: np.ndarray, alpha: np.ndarray, beta: np.ndarray, state: np.ndarray,
                 state_slot: np.ndarray, requests: Optional[Sequence[int]] = None
                 ) -> Dict[int, RequestResult]:
    """Oracle for a batch laid out like the library's inputs (see workloads).

    Returns {request index: RequestResult}; ``requests`` restricts the work to
    a subset (used for sampled checks of full-size workloads).
    """
    out: Dict[int, RequestResult] = {}
    R = len(node_offset) - 1
    todo = range(R) if requests is None else requests
    for r in todo:
        lo, hi = int(node_offset[r]), int(node_offset[r + 1])
        S0 = state[int(state_slot[r])]
        out[r] = verify_request(S0, parent[lo:hi], q[lo:hi], k[lo:hi], v[lo:hi],
                                alpha[lo:hi], beta[lo:hi])
    return out
