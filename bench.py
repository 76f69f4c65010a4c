"""Benchmark of the TreeWY verify + commit hot path on GB300.

One step = one speculative round of the wide ragged tree workload: 256
requests x 32 value heads, dk = dv = 128, one random draft tree per request
with N uniform in 16..64 nodes and depth <= 8, verified and committed in each
of 30 GDN layers (30 treewy_verify launches, then 30 treewy_commit launches,
every layer with its own state pool and inputs, all resident in HBM).

Metric: verified draft nodes per second = (draft nodes in the batch, summed
over ranks) / (time of one step).  Each layer's inputs (about 1.1 GB) are far
larger than L2, so no flush is needed between steps.  Also reported: verify
and commit GB/s on the algorithmic bytes, the roofline fraction of the
dominant kernel against the measured HBM copy bandwidth, the end-to-end rate
with host-resident inputs/outputs, the storeall comparator on the same
inputs, and the CPU oracle on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs its own independent
batch (weak scaling, no collective on the data path); ranks meet at a barrier
around the timed region and rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gdn_speculative_tree_gb300 import workloads as wl  # noqa: E402

METRIC = "verified draft nodes/sec (30 GDN layers verify+commit, 256 req x 32 heads, N 16..64)"
UNIT = "nodes/s"
CONFIG_NAME = "wide"
LAYERS = 30
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "verify_tc_wide_traffic.json")
KERNEL_SOURCES = ["gdn_speculative_tree_gb300/csrc/verify_tc.cuh",
                  "gdn_speculative_tree_gb300/csrc/verify_tc.cu",
                  "gdn_speculative_tree_gb300/csrc/treewy_device.cuh",
                  "gdn_speculative_tree_gb300/csrc/treewy_api.cu",
                  "gdn_speculative_tree_gb300/csrc/treewy_internal.h"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------- bytes model

def tree_stats(trees, accepted):
    """Per-request N, and path length of the accepted node (0 if none)."""
    Ns, plen = [], []
    for par, a in zip(trees, accepted):
        Ns.append(len(par))
        d = 0
        cur = int(a)
        while cur >= 0:
            d += 1
            cur = int(par[cur])
        plen.append(d)
    return np.array(Ns), np.array(plen)


def verify_bytes(Ns, H, state_bytes=65536):
    # per (request, head): S0 read (64 KiB fp32 / 32 KiB bf16) + per node q,k,v
    # (768 B bf16), alpha, beta (8 B), o and U written (1024 B fp32), gamma
    # (4 B); parents once per request
    return int(H * (state_bytes * len(Ns) + 1804 * Ns.sum()) + 4 * Ns.sum())


def commit_bytes(plen, H, state_bytes=65536):
    # per (request, head) with an accepted node: state read + written
    # + per path node u (512 B), k (256 B), alpha (4 B); nothing when a = -1
    live = plen > 0
    return int(H * (2 * state_bytes * live.sum() + 772 * plen.sum()))


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock and throttle reasons) every 25 ms; each
    sample is stamped with the host time it arrived, and the summary keeps
    only those between mark_start() and mark_end() (the timed region)."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "25",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # let the sampler start before the timed region begins
            deadline = time.time() + 2.0
            while not self.lines and time.time() < deadline:
                time.sleep(0.02)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        time.sleep(0.05)  # the sample that covers the last instants

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines or self.t0 is None or self.t1 is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for stamp, ln in list(self.lines):
            if not (self.t0 <= stamp <= self.t1 + 0.03):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "sm_mhz_min": min(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle leg

def oracle_jobs(cfg, n_requests: int, layers: int):
    """Oracle jobs for the first n_requests of every layer (CPU tensors).

    Trees depend only on the workload's seed and the request count, so every
    layer of the sample has the same trees; returns (jobs, draft nodes of the
    sample)."""
    from oracle import pool as opool
    jobs, nodes = [], 0
    for l in range(layers):
        w = wl.generate(cfg, R=n_requests, layer=l)
        f32 = lambda x: x.float().numpy()  # noqa: E731
        jobs += opool.jobs_from_arrays(w.node_offset.numpy(), w.parent.numpy(), f32(w.q), f32(w.k),
                                       f32(w.v), w.alpha.numpy(), w.beta.numpy(), w.state.numpy(),
                                       w.state_slot.numpy(), w.accepted.numpy(), range(w.R))
        nodes = int(w.node_offset[-1])
    return jobs, nodes


def oracle_sample(pool, cfg, n_requests: int, layers: int):
    """Time the oracle (verify + commit of every request in every layer of
    the sample) on the pool's workers.  Returns (nodes, wall seconds)."""
    jobs, nodes = oracle_jobs(cfg, n_requests, layers)
    t0 = time.perf_counter()
    pool.map(jobs, keep=False)
    return nodes, time.perf_counter() - t0


def cpu_baseline(pool, n_requests: int):
    cfg = wl.CONFIGS[CONFIG_NAME]
    nodes, dt = oracle_sample(pool, cfg, n_requests, LAYERS)
    return {"value": nodes / dt, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
            "sample": f"fp64 numpy oracle, first {n_requests} requests x {cfg.H} heads of the "
                      f"workload through all {LAYERS} layers ({nodes} nodes, {dt:.2f} s wall), "
                      f"one request-layer per job on {pool.workers} worker processes"}


def run_reference(args, world, rank, pool):
    """The oracle as the reference arm: every step verifies and commits a
    bounded sample of the workload (its first requests, all heads) through
    all 30 layers on every host core, timed as it runs."""
    if rank != 0:
        return
    cfg = wl.CONFIGS[CONFIG_NAME]
    n_req = args.ref_requests
    jobs, nodes = oracle_jobs(cfg, n_req, LAYERS)
    for _ in range(args.warmup):
        pool.map(jobs, keep=False)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        pool.map(jobs, keep=False)
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = nodes / t
    sample = (f"first {n_req} requests x {cfg.H} heads of the workload ({nodes} nodes) through all "
              f"{LAYERS} layers per step, one request-layer per job on {pool.workers} worker processes")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1000.0,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "wide ragged trees (256 req x 32 heads, N 16..64, depth<=8, "
                                   "30 GDN layers); each timed step is a bounded sample",
                       "sample_requests": n_req, "layers": LAYERS},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg

def run_ours(args, world, rank, local, pool=None):
    from gdn_speculative_tree_gb300 import binding
    from gdn_speculative_tree_gb300 import build as _build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    torch.cuda.set_device(local)
    _build.build()
    binding.load()
    dev = torch.device("cuda", local)
    cfg = wl.CONFIGS[CONFIG_NAME]
    layers = args.layers

    # inputs of every layer resident in HBM; trees are shared by the layers
    work = []
    for l in range(layers):
        w = wl.generate(cfg, layer=l + 1000 * rank, device=dev)
        work.append(binding.TreeVerifier(w))
    trees, accepted = work[0].wl.trees, work[0].wl.accepted.cpu().numpy()
    Ns, plen = tree_stats(trees, accepted)
    H = cfg.H
    vb, cb = verify_bytes(Ns, H), commit_bytes(plen, H)
    nodes = int(Ns.sum())

    stream = torch.cuda.current_stream()

    def new_events():
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(layers)]

    def step(ev_v=None, ev_c=None):
        for l, tv in enumerate(work):
            if ev_v is not None:
                ev_v[l][0].record(stream)
            tv.verify(stream)
            if ev_v is not None:
                ev_v[l][1].record(stream)
        for l, tv in enumerate(work):
            if ev_c is not None:
                ev_c[l][0].record(stream)
            tv.commit(None, stream)
            if ev_c is not None:
                ev_c[l][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for tv in work:
        if tv.status.any().item():
            raise SystemExit(f"device status bits set: {tv.status.unique().tolist()}")

    # timed region: kernel launches on `stream`, inputs resident in HBM; the
    # per-launch events sit on the same stream and are read after the region
    events = [(new_events(), new_events()) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:  # sampling starts before the barrier
        barrier(world)
        torch.cuda.synchronize()
        clk.mark_start()
        start.record(stream)
        for ev_v, ev_c in events:
            step(ev_v, ev_c)
        end.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
        barrier(world)
    total_ms = start.elapsed_time(end)
    v_ms = [a.elapsed_time(b) for ev_v, _ in events for a, b in ev_v]
    c_ms = [a.elapsed_time(b) for _, ev_c in events for a, b in ev_c]
    ms_per_step = max_over_ranks(total_ms / args.steps, world)
    all_nodes = sum_over_ranks(nodes, world)
    value = all_nodes / (ms_per_step / 1e3)

    peak, peak_kind = read_peaks()
    v_avg = sum(v_ms) / len(v_ms)
    c_avg = sum(c_ms) / len(c_ms)
    v_gbs = vb / (v_avg * 1e-3) / 1e9
    c_gbs = cb / (c_avg * 1e-3) / 1e9
    traffic = None
    if os.path.exists(PROFILE_TRAFFIC):
        with open(PROFILE_TRAFFIC) as f:
            prof = json.load(f)
        if prof.get("kernel_hash") == kernel_hash():
            traffic = prof.get("traffic_bytes_per_launch")

    # end to end through the public API: per step, pinned host inputs of all
    # layers copied in, verify + commit, outputs o of all layers copied out
    e2e = run_e2e(args, work, stream, world)
    fused = run_fused(args, work, stream, world, vb, cb, plen, H, peak)

    storeall = run_storeall(work[0], stream) if rank == 0 and not args.no_storeall else None
    cpu = cpu_baseline(pool, args.cpu_requests) if pool is not None else None

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, shapes of the pages' workloads)",
        "config": {"workload": "wide ragged trees: 256 requests x 32 value heads per GPU, dk=dv=128, "
                               "N~U{16..64}, depth<=8, fp32 state, bf16 q/k/v, 30 GDN layers per step",
                   "R": cfg.R, "H": H, "layers": layers, "nodes_per_layer": nodes,
                   "l2": "no flush: each layer's inputs (~1.1 GB) exceed the 129 MB L2"},
        "roofline": {"bound": "hbm", "achieved": v_gbs, "peak": peak, "unit": "GB/s",
                     "frac": v_gbs / peak, "traffic": traffic,
                     "kernel": "verify_tc_kernel<64>", "algorithmic_bytes_per_launch": vb,
                     "avg_launch_ms": v_avg, "peak_kind": f"{peak_kind} hbm_gbs"},
        "commit": {"achieved_gbs": c_gbs, "frac": c_gbs / peak, "avg_launch_ms": c_avg,
                   "algorithmic_bytes_per_launch": cb},
        "verify_nodes_per_s_per_layer": nodes / (v_avg * 1e-3),
        "head_verifies_per_s": cfg.R * H / (v_avg * 1e-3),
        "head_node_verifies_per_s": nodes * H / (v_avg * 1e-3),
        "gpu_launches": 2 * layers * args.steps,
        "e2e": e2e,
        "fused": fused,
        "storeall": storeall,
        "cpu_baseline": cpu,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_fused(args, work, stream, world, vb, cb, plen, H, peak):
    """Steady-state step with the previous round's commit fused into the verify:
    30 treewy_commit_verify launches per step (the same work per step as
    30 verify + 30 commit launches once the loop runs)."""
    from gdn_speculative_tree_gb300 import binding

    def step(ev=None):
        for l, tv in enumerate(work):
            if ev is not None:
                ev[l][0].record(stream)
            binding.treewy_commit_verify(tv.batch, tv.wl.accepted, tv.batch, stream)
            if ev is not None:
                ev[l][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in work] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for ev in events:
        step(ev)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(end) / args.steps, world)
    lay = [a.elapsed_time(b) for ev in events for a, b in ev]
    layer_ms = sum(lay) / len(lay)
    for tv in work:
        if tv.status.any().item():
            raise SystemExit(f"device status bits set in the fused step: {tv.status.unique().tolist()}")
    nodes = sum_over_ranks(int(work[0].wl.node_offset[-1]), world)
    # one state read per committing head is shared by the commit and the verify
    fb = vb + cb - int(H * 65536 * int((plen > 0).sum()))
    return {"value": nodes / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "layer_ms": layer_ms,
            "algorithmic_bytes_per_launch": fb, "achieved_gbs": fb / (layer_ms * 1e-3) / 1e9,
            "frac": fb / (layer_ms * 1e-3) / 1e9 / peak,
            "note": "treewy_commit_verify per layer: commit of the previous round inside this "
                    "round's verify (one state read per head instead of two)"}


def run_e2e(args, work, stream, world):
    """End to end through the public API: per step, every layer's inputs are
    copied in from pinned host memory, verified and committed, and its o is
    copied back.  Separate streams pipeline the layers: host-to-device copies of
    layer l+1 and device-to-host copies of layer l-1 run while layer l
    computes (events order each layer's copy-in, compute and copy-out, and a
    layer's buffers are not overwritten before the previous step is done with
    them)."""
    from gdn_speculative_tree_gb300 import binding
    hosts = []
    h2d = d2h = 0
    for tv in work:
        w = tv.wl
        ins = {name: getattr(w, name).cpu().pin_memory()
               for name in ("node_offset", "parent", "q", "k", "v", "alpha", "beta", "accepted")}
        out = torch.empty(tv.o.shape, dtype=tv.o.dtype).pin_memory()
        hosts.append((ins, out))
        h2d += sum(x.numel() * x.element_size() for x in ins.values())
        d2h += out.numel() * out.element_size()
    dev = work[0].o.device
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    L = len(work)
    ev_in = [torch.cuda.Event() for _ in range(L)]
    ev_done = [torch.cuda.Event() for _ in range(L)]
    ev_out = [torch.cuda.Event() for _ in range(L)]
    first = [True]

    def step():
        for l, (tv, (ins, out)) in enumerate(zip(work, hosts)):
            w = tv.wl
            if not first[0]:
                s_in.wait_event(ev_done[l])      # the previous step's compute of this layer
            with torch.cuda.stream(s_in):
                for name, x in ins.items():
                    getattr(w, name).copy_(x, non_blocking=True)
                ev_in[l].record(s_in)
            stream.wait_event(ev_in[l])
            if not first[0]:
                stream.wait_event(ev_out[l])     # o of the previous step has left
            binding.treewy_verify(tv.batch, stream)
            binding.treewy_commit(tv.batch, tv.wl.accepted, stream)
            ev_done[l].record(stream)
            s_out.wait_event(ev_done[l])
            with torch.cuda.stream(s_out):
                out.copy_(tv.o, non_blocking=True)
                ev_out[l].record(s_out)
        first[0] = False

    step()
    torch.cuda.synchronize()
    steps = max(2, min(args.steps, 10))
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    dt = max_over_ranks((time.perf_counter() - t0) / steps, world)
    nodes = sum_over_ranks(int(work[0].wl.node_offset[-1]), world)
    return {"value": nodes / dt, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": dt * 1e3, "steps": steps,
            "note": "pinned host inputs (q,k,v,alpha,beta,tree,accepted) of all layers copied in and "
                    "o of all layers copied out each step, pipelined across layers over a compute, "
                    "a copy-in and a copy-out stream; the state pool is model state and stays resident on the device"}


def run_storeall(tv, stream):
    """storeall comparator on layer 0's inputs: snapshot-per-node verify and
    rollback, timed with CUDA events (state restored afterwards)."""
    from gdn_speculative_tree_gb300 import binding
    w = tv.wl
    T, H = w.T, w.H
    need = T * H * w.dv * w.dk * 4
    free, _ = torch.cuda.mem_get_info()
    if need > 0.8 * free:
        return {"skipped": f"snapshots need {need / 1e9:.1f} GB, free {free / 1e9:.1f} GB"}
    snaps = torch.empty(T, H, w.dv, w.dk, device=w.q.device, dtype=torch.float32)
    S_save = w.state.clone()
    o = torch.empty_like(tv.o)
    status = torch.zeros_like(tv.status)
    b = binding.make_batch(node_offset=w.node_offset, parent=w.parent, q=w.q, k=w.k, v=w.v,
                           alpha=w.alpha, beta=w.beta, state=w.state, state_slot=w.state_slot,
                           o=o, U=o, status=status, max_nodes=w.max_nodes)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    vt, ct = [], []
    for i in range(4):
        ev[0].record(stream)
        binding.treewy_storeall_verify(b, snaps, stream)
        ev[1].record(stream)
        binding.treewy_storeall_commit(b, snaps, w.accepted, stream)
        ev[2].record(stream)
        ev[2].synchronize()
        w.state.copy_(S_save)
        if i:
            vt.append(ev[0].elapsed_time(ev[1]))
            ct.append(ev[1].elapsed_time(ev[2]))
    torch.cuda.synchronize()
    Ns = np.diff(w.node_offset.cpu().numpy())
    snap_bytes = int(Ns.sum()) * H * w.dv * w.dk * 4
    v_bytes = snap_bytes + verify_bytes(Ns, H) - int(Ns.sum()) * H * 516
    del snaps
    return {"verify_ms_per_layer": statistics.median(vt), "commit_ms_per_layer": statistics.median(ct),
            "snapshot_bytes_per_layer": snap_bytes, "verify_bytes_per_layer": v_bytes,
            "verify_gbs": v_bytes / (statistics.median(vt) * 1e-3) / 1e9,
            "state_blocks_per_request": "N+1 (treewy: 1)"}


# ---------------------------------------------------------------- studies

def _median_ms(fn, stream, reps, before=None):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        if before is not None:
            before()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def study_widths(args, local):
    """Verify and commit cost against tree width: full width trees of the
    shapes (w1, w2, w3), w in 1..3 (N = w1 + w1 w2 + w1 w2 w3), 256 requests x
    32 heads, dk = dv = 128, beside the storeall comparator on the same inputs.
    Every launch's inputs exceed L2; the state is restored before each commit."""
    from gdn_speculative_tree_gb300 import binding
    stream = torch.cuda.current_stream()
    peak, peak_kind = read_peaks()
    base = wl.CONFIGS[CONFIG_NAME].with_(tree="widths", accepted="uniform")
    rows = []
    shapes = sorted(((a, b, c) for a in (1, 2, 3) for b in (1, 2, 3) for c in (1, 2, 3)),
                    key=lambda s: (s[0] + s[0] * s[1] + s[0] * s[1] * s[2], s))
    for shape in shapes:
        cfg = base.with_(widths=shape)
        w = wl.generate(cfg, device=torch.device("cuda", local))
        tv = binding.TreeVerifier(w)
        S0 = w.state.clone()
        Ns, plen = tree_stats(w.trees, w.accepted.cpu().numpy())
        vb, cb = verify_bytes(Ns, w.H), commit_bytes(plen, w.H)
        for _ in range(args.warmup):
            tv.verify(stream)
        v_ms = _median_ms(lambda: tv.verify(stream), stream, 20)
        c_ms = _median_ms(lambda: tv.commit(None, stream), stream, 20,
                          before=lambda: w.state.copy_(S0))
        w.state.copy_(S0)
        if tv.status.any().item():
            raise SystemExit(f"device status bits set for widths {shape}")
        row = {"widths": list(shape), "N": int(Ns[0]), "depth": 3,
               "verify_us": v_ms * 1e3, "verify_gbs": vb / (v_ms * 1e-3) / 1e9,
               "verify_frac": vb / (v_ms * 1e-3) / 1e9 / peak,
               "verify_us_per_node": v_ms * 1e3 / int(Ns[0]),
               "commit_us": c_ms * 1e3, "commit_frac": cb / (c_ms * 1e-3) / 1e9 / peak}
        sa = run_storeall(tv, stream)
        if "verify_ms_per_layer" in sa:
            row["storeall_verify_us"] = sa["verify_ms_per_layer"] * 1e3
            row["storeall_commit_us"] = sa["commit_ms_per_layer"] * 1e3
            row["treewy_speedup_verify"] = sa["verify_ms_per_layer"] / v_ms
        rows.append(row)
        del tv, w, S0
        torch.cuda.empty_cache()
    print(json.dumps({"study": "verify cost vs tree width", "peak_gbs": peak,
                      "peak_kind": f"{peak_kind} hbm_gbs", "R": base.R, "H": base.H,
                      "rows": rows}), flush=True)


def study_fixed64(args, local):
    """The wide workload with every tree at the capacity, N = 64 (random
    trees of depth <= 8): verify, commit and the fused commit-into-verify
    per layer, median of 20 launches each (a layer's inputs exceed L2)."""
    from gdn_speculative_tree_gb300 import binding
    stream = torch.cuda.current_stream()
    peak, peak_kind = read_peaks()
    cfg = wl.CONFIGS[CONFIG_NAME].with_(tree="random64_d8")
    w = wl.generate(cfg, device=torch.device("cuda", local))
    tv = binding.TreeVerifier(w)
    S0 = w.state.clone()
    Ns, plen = tree_stats(w.trees, w.accepted.cpu().numpy())
    vb, cb = verify_bytes(Ns, w.H), commit_bytes(plen, w.H)
    fb = vb + cb - int(w.H * 65536 * int((plen > 0).sum()))
    for _ in range(args.warmup):
        tv.verify(stream)
    v_ms = _median_ms(lambda: tv.verify(stream), stream, 20)
    c_ms = _median_ms(lambda: tv.commit(None, stream), stream, 20, before=lambda: w.state.copy_(S0))
    f_ms = _median_ms(lambda: binding.treewy_commit_verify(tv.batch, w.accepted, tv.batch, stream),
                      stream, 20, before=lambda: w.state.copy_(S0))
    if tv.status.any().item():
        raise SystemExit("device status bits set in the N = 64 study")
    g = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    print(json.dumps({
        "study": "wide workload with N fixed at 64", "R": cfg.R, "H": cfg.H,
        "nodes_per_layer": int(Ns.sum()), "peak_gbs": peak, "peak_kind": f"{peak_kind} hbm_gbs",
        "verify": {"ms": v_ms, "algorithmic_bytes": vb, "gbs": g(vb, v_ms), "frac": g(vb, v_ms) / peak},
        "commit": {"ms": c_ms, "algorithmic_bytes": cb, "gbs": g(cb, c_ms), "frac": g(cb, c_ms) / peak},
        "fused": {"ms": f_ms, "algorithmic_bytes": fb, "gbs": g(fb, f_ms), "frac": g(fb, f_ms) / peak}}),
        flush=True)


def study_graph(args, local):
    """Launch overhead of 30 layers of verify + commit issued eagerly against
    the same calls captured once as a CUDA graph and replayed, on the chain
    workload (64 requests x 32 heads, chains of 4) and on the wide ragged
    tree workload (256 requests x 32 heads, N 16..64): the pages say the tree
    path could not be captured in their engine."""
    from gdn_speculative_tree_gb300 import binding
    dev = torch.device("cuda", local)
    layers = args.layers
    for name in ("chain", "wide"):
        cfg = wl.CONFIGS[name]
        work = [binding.TreeVerifier(wl.generate(cfg, layer=l, device=dev)) for l in range(layers)]
        stream = torch.cuda.Stream(device=dev)
        nodes = int(work[0].wl.node_offset[-1])

        def step():
            for tv in work:
                tv.verify(stream)
            for tv in work:
                tv.commit(None, stream)

        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                step()
        torch.cuda.synchronize()
        reps = max(args.steps, 20)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            eager_ms = _median_ms(step, stream, reps)
        host_eager = (time.perf_counter() - t0) / reps * 1e3
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                g.replay()
            torch.cuda.synchronize()
            graph_ms = _median_ms(g.replay, stream, reps)
        for tv in work:
            if tv.status.any().item():
                raise SystemExit("device status bits set in the graph study")
        print(json.dumps({"study": "CUDA-graph capture of batched tree verify+commit",
                          "workload": f"{name}: {cfg.R} requests x {cfg.H} heads, {layers} layers",
                          "launches_per_step": 2 * layers, "eager_ms_per_step": eager_ms,
                          "graph_ms_per_step": graph_ms, "eager_host_ms_per_step": host_eager,
                          "eager_nodes_per_s": nodes * 1e3 / eager_ms,
                          "graph_nodes_per_s": nodes * 1e3 / graph_ms,
                          "graph_speedup": eager_ms / graph_ms}), flush=True)
        del work, g
        torch.cuda.empty_cache()


def study_bf16state(args, local):
    """A bf16 state pool (32 KiB per head instead of 64 KiB), the serving
    dtype: 30 layers of verify + commit, and the fused commit-into-verify
    step, on the wide ragged workload (the benchmark), on the chain workload
    (multi-token-prediction chains, the pages' serving shape) and on the
    binary-tree workload; one JSON line each.  Each step cycles through 30 layers of distinct inputs,
    more than the 129 MB L2 holds."""
    from gdn_speculative_tree_gb300 import binding
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peak, peak_kind = read_peaks()
    layers = args.layers
    g = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    for name, label in ((CONFIG_NAME, "wide ragged trees, 256 req x 32 heads"),
                        ("chain", "MTP chains of 4, 64 req x 32 heads"),
                        ("binary", "complete binary trees of 15 nodes, 128 req x 32 heads")):
        cfg = wl.CONFIGS[name]
        work = [binding.TreeVerifier(wl.generate(cfg, layer=l, device=dev, state_dtype="bf16"))
                for l in range(layers)]
        Ns, plen = tree_stats(work[0].wl.trees, work[0].wl.accepted.cpu().numpy())
        H = cfg.H
        vb, cb = verify_bytes(Ns, H, 32768), commit_bytes(plen, H, 32768)
        fb = vb + cb - int(H * 32768 * int((plen > 0).sum()))
        nodes = int(Ns.sum())

        def timed(fn_layer):
            for _ in range(args.warmup):
                for tv in work:
                    fn_layer(tv)
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps * layers)]
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record(stream)
            i = 0
            for _ in range(args.steps):
                for tv in work:
                    ev[i][0].record(stream)
                    fn_layer(tv)
                    ev[i][1].record(stream)
                    i += 1
            end.record(stream)
            torch.cuda.synchronize()
            per = [a.elapsed_time(b) for a, b in ev]
            return start.elapsed_time(end) / args.steps, sum(per) / len(per)

        v_step, v_ms = timed(lambda tv: tv.verify(stream))
        c_step, c_ms = timed(lambda tv: tv.commit(None, stream))
        f_step, f_ms = timed(lambda tv: binding.treewy_commit_verify(tv.batch, tv.wl.accepted,
                                                                     tv.batch, stream))
        for tv in work:
            if tv.status.any().item():
                raise SystemExit(f"device status bits set in the bf16 state study ({name})")
        print(json.dumps({
            "study": "bf16 state pool", "config": name,
            "workload": f"{label}, {layers} layers, bf16 state", "peak_gbs": peak,
            "peak_kind": f"{peak_kind} hbm_gbs",
            "ms_per_step": v_step + c_step, "value": nodes / ((v_step + c_step) * 1e-3), "unit": UNIT,
            "verify": {"avg_launch_ms": v_ms, "algorithmic_bytes": vb, "gbs": g(vb, v_ms),
                       "frac": g(vb, v_ms) / peak},
            "commit": {"avg_launch_ms": c_ms, "algorithmic_bytes": cb, "gbs": g(cb, c_ms),
                       "frac": g(cb, c_ms) / peak},
            "fused": {"ms_per_step": f_step, "value": nodes / (f_step * 1e-3), "avg_launch_ms": f_ms,
                      "algorithmic_bytes": fb, "gbs": g(fb, f_ms), "frac": g(fb, f_ms) / peak}}),
            flush=True)
        del work
        torch.cuda.empty_cache()


def storeall_chunked(w, o, stream, reps=3, max_bytes=34e9):
    """The storeall comparator over a whole batch, verified and rolled back in
    request chunks whose snapshots fit in max_bytes; returns summed median
    times of the chunks and the snapshot bytes (the state is restored after
    every rollback, untimed)."""
    from gdn_speculative_tree_gb300 import binding
    node = w.node_offset.cpu().numpy().astype(np.int64)
    per_node = w.H * w.dv * w.dk * 4
    chunks, r0 = [], 0
    while r0 < w.R:
        r1 = r0 + 1
        while r1 < w.R and (node[r1 + 1] - node[r0]) * per_node <= max_bytes:
            r1 += 1
        chunks.append((r0, r1))
        r0 = r1
    most = max(int(node[b] - node[a]) for a, b in chunks)
    snaps = torch.empty(most, w.H, w.dv, w.dk, device=w.q.device, dtype=torch.float32)
    S_save = w.state.clone()
    status = torch.zeros(w.R, device=w.q.device, dtype=torch.int32)
    v_tot = c_tot = 0.0
    for a, b in chunks:
        bt = binding.make_batch(node_offset=w.node_offset[a:b + 1], parent=w.parent, q=w.q, k=w.k,
                                v=w.v, alpha=w.alpha, beta=w.beta, state=w.state,
                                state_slot=w.state_slot[a:b], o=o, U=o, status=status[a:b],
                                max_nodes=w.max_nodes, T=w.T)
        vt, ct = [], []
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for i in range(reps + 1):
            ev[0].record(stream)
            binding.treewy_storeall_verify(bt, snaps, stream)
            ev[1].record(stream)
            binding.treewy_storeall_commit(bt, snaps, w.accepted[a:b], stream)
            ev[2].record(stream)
            ev[2].synchronize()
            w.state.copy_(S_save)
            if i:
                vt.append(ev[0].elapsed_time(ev[1]))
                ct.append(ev[1].elapsed_time(ev[2]))
        v_tot += statistics.median(vt)
        c_tot += statistics.median(ct)
    torch.cuda.synchronize()
    if status.any().item():
        raise SystemExit("device status bits set in the storeall comparator")
    del snaps
    torch.cuda.empty_cache()
    return v_tot, c_tot, int(node[-1]) * per_node, len(chunks)


def study_configs(args, local, pool):
    """Every workload of the benchmark family, one JSON line each: verify,
    commit and the fused commit-into-verify per launch (median of 20 launches,
    L2 flushed before each, the state restored untimed before each commit),
    their algorithmic bytes, GB/s and fraction of the measured HBM peak, the
    node counters, the storeall comparator on the same inputs (in request
    chunks) and the oracle on a bounded sample on every host core."""
    from gdn_speculative_tree_gb300 import binding
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peak, peak_kind = read_peaks()
    # L2 flush before each timed launch: 256 MB written (twice the 129 MB L2),
    # then another 256 MB buffer read, so that the launch starts from a cold
    # L2 holding no dirty lines (otherwise the write-back of the flush's own
    # writes, up to the whole L2, would fall inside the timed launch)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.sum()
    g = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    specs = [("chain", wl.CONFIGS["chain"], 32),
             ("binary", wl.CONFIGS["binary"], 16),
             ("wide", wl.CONFIGS["wide"], 16),
             ("wide_fixed64", wl.CONFIGS["wide"].with_(tree="random64_d8"), 8),
             ("stress", wl.CONFIGS["stress"], 4)]
    only = set(args.configs.split(",")) if args.configs else None
    for name, cfg, n_oracle in specs:
        if only is not None and name not in only:
            continue
        w = wl.generate(cfg, device=dev)
        tv = binding.TreeVerifier(w)
        S0 = w.state.clone()
        Ns, plen = tree_stats(w.trees, w.accepted.cpu().numpy())
        H = w.H
        vb, cb = verify_bytes(Ns, H), commit_bytes(plen, H)
        fb = vb + cb - int(H * 65536 * int((plen > 0).sum()))
        nodes = int(Ns.sum())
        for _ in range(args.warmup):
            tv.verify(stream)

        def restore_flush():
            w.state.copy_(S0)
            flush()

        v_ms = _median_ms(lambda: tv.verify(stream), stream, 20, before=flush)
        c_ms = _median_ms(lambda: tv.commit(None, stream), stream, 20, before=restore_flush)
        f_ms = _median_ms(lambda: binding.treewy_commit_verify(tv.batch, w.accepted, tv.batch, stream),
                          stream, 20, before=restore_flush)
        w.state.copy_(S0)
        torch.cuda.synchronize()
        if tv.status.any().item():
            raise SystemExit(f"device status bits set in config {name}")
        line = {"study": "configs", "config": name, "R": w.R, "H": H, "nodes_per_layer": nodes,
                "N_mean": float(Ns.mean()), "N_max": int(Ns.max()),
                "peak_gbs": peak, "peak_kind": f"{peak_kind} hbm_gbs",
                "verify": {"ms": v_ms, "algorithmic_bytes": vb, "gbs": g(vb, v_ms),
                           "frac": g(vb, v_ms) / peak,
                           "tree_nodes_per_s": nodes / (v_ms * 1e-3),
                           "head_node_verifies_per_s": nodes * H / (v_ms * 1e-3),
                           "head_verifies_per_s": w.R * H / (v_ms * 1e-3)},
                "commit": {"ms": c_ms, "algorithmic_bytes": cb, "gbs": g(cb, c_ms),
                           "frac": g(cb, c_ms) / peak,
                           "committing_heads": int((plen > 0).sum()) * H},
                "fused": {"ms": f_ms, "algorithmic_bytes": fb, "gbs": g(fb, f_ms),
                          "frac": g(fb, f_ms) / peak,
                          "vs_separate": (v_ms + c_ms) / f_ms},
                "l2": "flushed before every timed launch: 256 MB written, then 256 MB of another buffer read (cold L2, no dirty lines)"}
        if not args.no_storeall:
            o = torch.empty_like(tv.o)
            sv, sc, sbytes, nch = storeall_chunked(w, o, stream)
            sv_bytes = sbytes + vb - nodes * H * 516
            line["storeall"] = {"verify_ms": sv, "commit_ms": sc, "snapshot_bytes": sbytes,
                                "verify_bytes": sv_bytes, "verify_gbs": g(sv_bytes, sv),
                                "verify_frac": g(sv_bytes, sv) / peak, "chunks": nch,
                                "treewy_verify_speedup": sv / v_ms,
                                "state_blocks_per_request": "N+1 (treewy: 1)"}
            del o
        if pool is not None:
            cnodes, dt = oracle_sample(pool, cfg, n_oracle, 1)
            line["oracle"] = {"requests": n_oracle, "nodes": cnodes, "wall_s": dt,
                              "nodes_per_s": cnodes / dt, "cores": pool.workers,
                              "gpu_speedup_verify_commit": (cnodes / dt) ** -1 * nodes /
                              ((v_ms + c_ms) * 1e-3)}
        print(json.dumps(line), flush=True)
        del tv, w, S0
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--cpu-requests", type=int, default=16,
                    help="requests of the oracle's CPU-baseline sample (0: skip it, and the "
                         "oracle samples of --study configs)")
    ap.add_argument("--ref-requests", type=int, default=8,
                    help="requests per step of the reference arm's sample")
    ap.add_argument("--no-storeall", action="store_true")
    ap.add_argument("--configs", default="",
                    help="--study configs: comma-separated subset of chain,binary,wide,"
                         "wide_fixed64,stress")
    ap.add_argument("--study", choices=["widths", "graph", "bf16state", "fixed64", "configs"],
                    help="print study lines instead of the benchmark line (1 GPU)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    # The oracle's worker pool is forked here, before this process makes any
    # GPU call (its workers only run numpy).
    pool = None
    wants_pool = args.impl == "reference" or (args.study in (None, "configs") and args.cpu_requests > 0)
    if wants_pool and rank == 0 and world == 1:
        from oracle.pool import OraclePool
        pool = OraclePool(method="fork")
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.study is not None:
            if rank == 0:
                from gdn_speculative_tree_gb300 import binding
                from gdn_speculative_tree_gb300 import build as _build
                torch.cuda.set_device(local)
                _build.build()
                binding.load()
                if args.study == "configs":
                    study_configs(args, local, pool)
                else:
                    {"widths": study_widths, "graph": study_graph, "bf16state": study_bf16state,
                     "fixed64": study_fixed64}[args.study](args, local)
        elif args.impl == "reference":
            if rank == 0 and pool is None:
                from oracle.pool import OraclePool
                pool = OraclePool(method="spawn")
            run_reference(args, world, rank, pool)
        else:
            run_ours(args, world, rank, local, pool)
    finally:
        if pool is not None:
            pool.close()
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
