"""The oracle's process pool adds no arithmetic: its results equal the
one-by-one calls bit for bit, in job order, with either start method."""
import numpy as np
import pytest

from gdn_speculative_tree_gb300 import workloads as wl
from oracle import gdn_tree_oracle as orc
from oracle import pool as opool


@pytest.mark.parametrize("method", ["spawn", "fork"])
def test_pool_equals_serial(method):
    w = wl.generate(wl.CONFIGS["wide"].with_(H=2, dk=16, dv=8), R=5)
    f = wl.as_float64
    node = w.node_offset.numpy()
    acc = w.accepted.numpy()
    jobs = opool.jobs_from_arrays(node, w.parent.numpy(), f(w.q), f(w.k), f(w.v), f(w.alpha),
                                  f(w.beta), f(w.state), w.state_slot.numpy(), acc, range(w.R))
    with opool.OraclePool(workers=2, method=method) as pool:
        got = pool.map(jobs)
        assert pool.map(jobs, keep=False) == [None] * w.R
    for r, (o, U, g, S_c) in enumerate(got):
        lo, hi = int(node[r]), int(node[r + 1])
        S0 = f(w.state[int(w.state_slot[r])])
        ref = orc.verify_request(S0, w.parent.numpy()[lo:hi], f(w.q[lo:hi]), f(w.k[lo:hi]),
                                 f(w.v[lo:hi]), f(w.alpha[lo:hi]), f(w.beta[lo:hi]))
        assert np.array_equal(o, ref.o) and np.array_equal(U, ref.U)
        assert np.array_equal(g, ref.gamma)
        assert np.array_equal(S_c, orc.commit_request(S0, ref, int(acc[r])))


def test_host_cores_positive():
    assert opool.host_cores() >= 1
