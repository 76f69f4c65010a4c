"""World-size-2 checks of the benchmark's multi-rank host logic on CPU (gloo):
each rank holds an independent batch (weak scaling; same tree shapes, its own
seeded data), and the timing reductions take the max (time) and the sum
(nodes) over ranks with no collective on the data path.
"""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from gdn_speculative_tree_gb300 import workloads as wl
    try:
        w_, r_, l_ = bench.dist_setup(world)
        assert (w_, r_) == (world, rank)
        bench.barrier(world)
        mx = bench.max_over_ranks(float(rank + 1) * 10.0, world)
        sm = bench.sum_over_ranks(float(rank + 1), world)
        cfg = wl.CONFIGS["wide"]
        w = wl.generate(cfg, R=3, layer=0 + 1000 * rank)
        q.put((rank, mx, sm, [len(t) for t in w.trees], float(w.q.float().sum())))
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions_and_sharding():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(world))
    assert all(o[1] == 20.0 for o in out)          # max over ranks
    assert all(o[2] == 3.0 for o in out)           # sum over ranks
    assert out[0][3] == out[1][3]                  # same tree shapes on every rank
    assert out[0][4] != out[1][4]                  # independent data per rank
