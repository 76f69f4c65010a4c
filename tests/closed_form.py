"""Independent routes to the gated-delta-rule tree results, used to pin the oracle.

Written separately from the oracle and sharing nothing with it:

* ``closed_form_head``: the pages' closed form.  Build the ancestor-masked
  system of "TreeWY: Speculative Verification for Gated DeltaNet Hybrids",
  §3 Eq. (2) with dense matrices, solve it with a general LU solve
  (numpy.linalg.solve, deliberately not forward substitution), then read
  states and outputs from the decayed-attention closed form of the technical
  review, §3.1 Eq. (5) restricted to ancestors (§3.2) and Eq. (6).  Decay
  ratios are formed by division g_t / g_i, as printed.
* ``sequential_gdn``: the gated delta rule applied token by token to a chain,
  with the transition written as an explicit matrix
  T_t = alpha_t (I - beta_t k_t k_t^T) (paper §1 Eq. (1), review §2.4 Eq. (3)).
"""
from __future__ import annotations

import numpy as np


def ancestor_sets(parent):
    """Strict ancestors of every node, by walking parent pointers."""
    out = []
    for n in range(len(parent)):
        anc = []
        p = int(parent[n])
        while p >= 0:
            anc.append(p)
            p = int(parent[p])
        out.append(anc)
    return out


def closed_form_head(S0, parent, q, k, v, alpha, beta):
    """One head.  S0 [dv][dk]; q,k [N][dk]; v [N][dv]; alpha,beta [N].

    Returns (o [N][dv], Vt [N][dv], g [N], S [N][dv][dk]).
    """
    N = len(parent)
    anc = ancestor_sets(parent)
    g = np.array([np.prod([alpha[j] for j in anc[t] + [t]]) for t in range(N)])
    G = np.zeros((N, N))
    for t in range(N):
        for i in anc[t]:
            G[t, i] = (g[t] / g[i]) * float(k[t] @ k[i])
    S0k = (S0 @ k.T).T                                  # row t is S0 k_t
    R = beta[:, None] * v - (beta * g)[:, None] * S0k
    system = np.eye(N) + np.diag(beta) @ G
    Vt = np.linalg.solve(system, R) if N else np.zeros_like(v)
    S = np.empty((N,) + S0.shape)
    o = np.empty_like(v)
    for t in range(N):
        St = g[t] * S0
        for i in anc[t] + [t]:
            St = St + (g[t] / g[i]) * np.outer(Vt[i], k[i])
        S[t] = St
        o[t] = St @ q[t]
    return o, Vt, g, S


def sequential_gdn(S0, q, k, v, alpha, beta):
    """Token-by-token gated delta rule along a chain (explicit transition matrix)."""
    dk = S0.shape[1]
    S = np.array(S0, dtype=np.float64)
    outs, states = [], []
    for t in range(len(alpha)):
        Tt = alpha[t] * (np.eye(dk) - beta[t] * np.outer(k[t], k[t]))
        S = S @ Tt + beta[t] * np.outer(v[t], k[t])
        states.append(S.copy())
        outs.append(S @ q[t])
    return np.array(outs), np.array(states)
