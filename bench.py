"""Benchmark of the paged-KV hot path on GB300.

One step = the whole hot path over one batch: the fused kernel appends each
sequence's new token to the paged pool and runs the split-KV paged-attention
decode over every sequence (continuous-batching decode, 256 sequences,
context lengths lognormal with median 1024 and sigma 1.2 clipped to
[1, 8192], bf16, 14 query / 2 KV heads, head_dim 64, block_size 16).

Printed (rank 0, one JSON line):
  value      KV-read GB/s: K/V bytes of all contexts / device time per step
  e2e        the same metric through the public API with the step's inputs
             copied from pinned host memory and the output copied back
  roofline   the decode kernel's algorithmic bytes per launch / its average
             launch time (CUDA events on its stream) against measured HBM
             bandwidth
  cpu_baseline  the fp64 CPU oracle, timed on this host's cores on the same batch

``--impl reference`` times the fp64 CPU oracle instead (the reference arm:
there is no reference implementation to install, the pages hold no code).
Run under torchrun for N > 1: every rank runs an independent replica on its
own GPU (no collective on the data path), and rank 0 reports the total over
all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("paged decode attention: KV-read GB/s (% of GB300 HBM peak), "
          "µs per decode step")
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def reduce_max_sum(dist, elapsed: float, units: float, device=None):
    """Slowest rank's time and the units all ranks processed."""
    if dist is None:
        return elapsed, units
    import torch
    t = torch.tensor([elapsed], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------------------
# clocks sampled while the GPU works
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="ns_clocks_", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s, p in zip(sm, pw) if p is not None] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------

def make_workload(name: str):
    from paged_kv_decode_ns_gb300 import workloads as wl
    return wl.WORKLOADS[name]()


def workload_config(st, name, pools):
    return {"workload": f"{st.name}: {name}", "num_seqs": st.num_seqs,
            "context_tokens": int(st.context_lens.sum()),
            "max_context": int(st.context_lens.max()),
            "num_q_heads": st.num_q_heads, "num_kv_heads": st.num_kv_heads,
            "head_dim": st.head_dim, "block_size": st.block_size,
            "num_blocks": st.num_blocks, "step": "fused kv_append + split-KV paged decode",
            "l2": (f"inputs larger than L2: {pools} rotating pool copies of "
                   f"{2 * st.k_pool.nbytes / 1e6:.0f} MB each (L2 129 MB)")}


def run_cpu_oracle(st, num_threads: int, max_seqs: int | None = None):
    """Time the fp64 oracle on the first ``max_seqs`` sequences; return
    (seconds, kv_bytes, n_seqs, threads)."""
    import oracle
    orc = oracle.load()
    n = st.num_seqs if max_seqs is None else max(1, min(st.num_seqs, max_seqs))
    q = st.q[:n]
    t0 = time.perf_counter()
    orc.paged_attention(st.dtype, q, st.k_pool, st.v_pool, st.block_tables[:n],
                        st.context_lens[:n], st.scale, num_threads=num_threads)
    dt = time.perf_counter() - t0
    kv = int(st.context_lens[:n].astype(np.int64).sum()) * st.num_kv_heads * st.head_dim * 4
    return dt, kv, n, num_threads


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def bench_ours(args):
    import torch
    from paged_kv_decode_ns_gb300 import binding as nb

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    st = make_workload(args.workload)

    def dt_of(bits):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev)
        return t.view(torch.bfloat16 if st.dtype == "bf16" else torch.float16)

    def ints(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(dev)

    # device-resident state: the pool (rotated copies so that no step finds
    # its K/V in L2), the step's inputs, the output and the workspace
    pool_bytes = 2 * st.k_pool.nbytes
    npools = max(1, args.pools if args.pools else math.ceil(2 * L2_BYTES / max(pool_bytes, 1)))
    k0, v0 = dt_of(st.k_pool), dt_of(st.v_pool)
    pools = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(npools - 1)]
    q = dt_of(st.q)
    k_new, v_new = dt_of(st.k_new), dt_of(st.v_new)
    slots = ints(st.slot_mapping, np.int64)
    tables = ints(st.block_tables, np.int32)
    lens = ints(st.context_lens, np.int32)
    out = torch.empty_like(q)
    ws = nb.alloc_workspace(st.num_seqs, st.num_q_heads, st.num_kv_heads, st.head_dim, dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        kp, vp = pools[i % npools]
        nb.ns_kv_append_paged_attn_decode(q, k_new, v_new, slots, kp, vp, tables, lens,
                                          st.scale, out, ws, stream=stream)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    nb.raise_on_device_status()

    # ---- timed region: K steps, device time, max over ranks
    barrier(dist)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    elapsed_ms = e0.elapsed_time(e1)

    # ---- per-launch duration of the decode kernel (events on its stream)
    n_lat = min(args.steps, 200)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_lat)]
    for i, (a, b) in enumerate(evs):
        a.record(stream)
        step(i)
        b.record(stream)
    torch.cuda.synchronize(dev)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)

    # keep the GPU busy long enough for the clock sampler (untimed)
    t_end = time.time() + max(0.0, args.soak_s - elapsed_ms / 1e3)
    i = 0
    while time.time() < t_end:
        for _ in range(200):
            step(i)
            i += 1
        torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    nb.raise_on_device_status()

    # ---- end to end through the public API with host buffers
    def pinned(t):
        return torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
    h_in = [pinned(x) for x in (q, k_new, v_new, slots, tables, lens)]
    d_in = [q, k_new, v_new, slots, tables, lens]
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = h_out.numel() * h_out.element_size()
    n_e2e = max(1, min(args.steps, args.e2e_steps))
    for i in range(3):
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        step(i)
        h_out.copy_(out, non_blocking=True)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for i in range(n_e2e):
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        step(i)
        h_out.copy_(out, non_blocking=True)
    e3.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e2e_ms = e2.elapsed_time(e3)
    nb.raise_on_device_status()

    kv_bytes = st.kv_read_bytes()
    alg_bytes = st.algorithmic_bytes(with_append=True)
    t_max, units = reduce_max_sum(dist, elapsed_ms, kv_bytes * args.steps, dev)
    te2e_max, units_e2e = reduce_max_sum(dist, e2e_ms, kv_bytes * n_e2e, dev)
    if rank != 0:
        return None

    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
    value = units / (t_max * 1e-3) / 1e9
    cpu = None
    if args.cpu_baseline:
        cores = host_cores()
        secs, kvb, n, thr = run_cpu_oracle(st, cores)
        cpu = {"value": kvb / secs / 1e9, "unit": "GB/s", "cores": thr, "kind": "oracle",
               "sample": f"all {n} sequences of the batch, attention only, one pass, "
                         f"{secs:.2f} s (fp64 C oracle, OpenMP over (sequence, head))"}
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_max / args.steps, "us_per_step": 1e3 * t_max / args.steps,
        "hbm_peak_frac": value / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": st.dtype, "data": "synthetic (seeded; no dataset or weights involved)",
        "config": workload_config(st, args.workload, npools),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": args.traffic,
                     "kernel": "paged_decode_kernel (fused kv_append)",
                     "bytes_per_launch": alg_bytes, "launch_us": launch_ms * 1e3,
                     "peak_source": f"{peak_src} hbm_gbs"},
        "cpu_baseline": cpu,
        "e2e": {"value": units_e2e / (te2e_max * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": 1e3 * te2e_max / n_e2e, "steps": n_e2e},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle
# ---------------------------------------------------------------------------

def bench_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    st = make_workload(args.workload)
    cores = host_cores()
    budget = args.reference_budget_s
    # size the per-step sample so that warmup + steps fit the budget
    t1, _, _, _ = run_cpu_oracle(st, cores, max_seqs=8)
    per_seq = max(t1 / 8, 1e-6)
    n = int(max(1, min(st.num_seqs, budget / (args.steps + args.warmup) / per_seq)))
    for _ in range(args.warmup):
        run_cpu_oracle(st, cores, max_seqs=n)
    total_t, total_b = 0.0, 0
    for _ in range(args.steps):
        secs, kvb, n_done, thr = run_cpu_oracle(st, cores, max_seqs=n)
        total_t += secs
        total_b += kvb
    value = total_b / total_t / 1e9
    sample = (f"first {n} of {st.num_seqs} sequences per step "
              f"({int(st.context_lens[:n].sum())} context tokens), attention only")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": workload_config(st, args.workload, 1),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_b256")
    ap.add_argument("--pools", type=int, default=0, help="rotating pool copies (0 = enough to exceed 2x L2)")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--soak-s", type=float, default=1.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch from an ncu capture of the current kernel")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    res = bench_reference(args) if args.impl == "reference" else bench_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
