"""The fp64 oracle over many requests at once, on every host core.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may use it.  It adds no arithmetic: each job is one call of
``gdn_tree_oracle.verify_request`` followed by ``commit_request`` for one
request (all its heads), and jobs are independent, so they are spread over a
pool of worker processes.

Start method: ``spawn`` by default, which is safe in a process that has
already used the GPU (a process forked after CUDA initialisation must not
touch the device, and a pool forked then can hang).  ``fork`` is accepted for
a pool created before the first GPU call: its workers then share the parent's
already imported modules instead of importing them again.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

from oracle import gdn_tree_oracle as orc

# (S0 [H][dv][dk], parent [N], q [N][H][dk], k [N][H][dk], v [N][H][dv],
#  alpha [N][H], beta [N][H], accepted, state_dtype)
Job = Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray, np.ndarray, np.ndarray, np.ndarray,
            int, str]


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux hosts
        return os.cpu_count() or 1


def _single_threaded() -> None:
    # one request per worker: keep any threaded math library to one thread
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"


def run_job(job: Job, keep: bool = True):
    """Verify one request and commit its accepted node.

    Returns (o, U, gamma, S_commit) in fp64, or None when ``keep`` is false
    (timing runs: the result is computed and dropped in the worker).
    """
    S0, parent, q, k, v, alpha, beta, accepted, state_dtype = job
    res = orc.verify_request(S0, parent, q, k, v, alpha, beta)
    S_c = orc.commit_request(S0, res, int(accepted), state_dtype=state_dtype)
    if not keep:
        return None
    return res.o, res.U, res.gamma, S_c


def _run_keep(job: Job):
    return run_job(job, True)


def _run_drop(job: Job):
    return run_job(job, False)


class OraclePool:
    """A pool of worker processes running oracle jobs (one request each)."""

    def __init__(self, workers: Optional[int] = None, method: str = "spawn"):
        self.workers = max(1, int(workers or host_cores()))
        ctx = mp.get_context(method)
        self._pool = ctx.Pool(self.workers, initializer=_single_threaded)

    def map(self, jobs: Sequence[Job], keep: bool = True) -> List:
        """Results in job order (see run_job)."""
        fn = _run_keep if keep else _run_drop
        return self._pool.map(fn, jobs, chunksize=1)

    def close(self) -> None:
        if self._pool is not None:
            self._pool.close()
            self._pool.join()
            self._pool = None

    def __enter__(self) -> "OraclePool":
        return self

    def __exit__(self, *exc) -> None:
        self.close()


def jobs_from_arrays(node_offset: np.ndarray, parent: np.ndarray, q: np.ndarray, k: np.ndarray,
                     v: np.ndarray, alpha: np.ndarray, beta: np.ndarray, state: np.ndarray,
                     state_slot: np.ndarray, accepted: np.ndarray, requests: Iterable[int],
                     state_dtype: str = "f32") -> List[Job]:
    """One job per request of a batch laid out like the library's inputs."""
    jobs: List[Job] = []
    for r in requests:
        lo, hi = int(node_offset[r]), int(node_offset[r + 1])
        jobs.append((state[int(state_slot[r])], parent[lo:hi], q[lo:hi], k[lo:hi], v[lo:hi],
                     alpha[lo:hi], beta[lo:hi], int(accepted[r]), state_dtype))
    return jobs
