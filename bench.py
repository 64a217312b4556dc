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

# DRAM bytes per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture, keyed by workload and kernel,
# with a hash of the kernel's source files at capture time.  The bench reports
# the figure only while those sources are unchanged (else null).
KERNEL_SOURCES = {
    "paged_decode_kernel": ["paged_kv_decode_ns_gb300/csrc/paged_decode.cuh",
                            "paged_kv_decode_ns_gb300/csrc/paged_decode_launch.cuh",
                            "paged_kv_decode_ns_gb300/csrc/ns_common.cuh", "include/ns_paged.h"],
    "tc_prefill_kernel": ["paged_kv_decode_ns_gb300/csrc/tc_prefill.cu",
                          "paged_kv_decode_ns_gb300/csrc/ns_common.cuh",
                          "paged_kv_decode_ns_gb300/csrc/tcgen05.cuh", "include/ns_paged.h"],
}
PROFILED_TRAFFIC = {
    # ncu capture of the committed kernel (dram__bytes_read.sum + dram__bytes_write.sum
    # of one launch of the default command): 238.97 MB read + 3.02 MB written
    ("decode_b256", "paged_decode_kernel"): {
        "sources_sha256": "2b58c7c4cb7198c03f7ca272085777c9b661caccb0b7a272b9f5b5c754fc564d",
        "bytes": 241993216},
    # ncu capture of the committed kernel: 4.73 MB read, 0 written
    ("mixed_chunked_prefill", "tc_prefill_kernel"): {
        "sources_sha256": "dc7e7767b5ed32791155281aabc498f1bf5ef60ab74f169a39dd48bfaaf84944",
        "bytes": 4729088},
}


def strip_comments(src: str) -> str:
    """C/C++ source with comments removed and blank lines dropped, so that a
    comment edit does not count as a change to the kernel."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # string or character literal: copy it whole
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    lines = (ln.rstrip() for ln in "".join(out).splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_sources_sha(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(rel.encode())
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()


def traffic_source(args, traffic):
    """Where the roofline's traffic figure comes from (it is not measured in this run)."""
    if args.traffic is not None:
        return "--traffic on the command line"
    if traffic is None:
        return None
    return ("ncu capture (dram__bytes_read.sum + dram__bytes_write.sum, one launch) of the same "
            "kernel sources, matched by their sha256 in bench.py")


def profiled_traffic(workload: str, kernel: str):
    rec = PROFILED_TRAFFIC.get((workload, kernel))
    if rec is None or rec["sources_sha256"] != kernel_sources_sha(kernel):
        return None
    return rec["bytes"]
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


def decode_policy(args):
    """The forced decode policy the command line asks for, or None (automatic)."""
    p = {}
    if getattr(args, "whole_sequences", False):
        p["whole_sequences"] = 1
    if getattr(args, "min_blocks_per_cta", 0):
        p["min_blocks_per_cta"] = args.min_blocks_per_cta
    if getattr(args, "num_ctas", 0):
        p["num_ctas"] = args.num_ctas
    if getattr(args, "merge_levels", 0):
        p["merge_levels"] = args.merge_levels
    return p or None


def workload_config(st, name, pools, layers=1, kv="native", policy=None):
    step = ("fused kv_append + split-KV paged decode" if st.is_decode
            else "kv_append + chunked prefill (tensor-core spans, decode-walk rows)")
    if layers > 1:
        step = (f"{layers} attention layers (Qwen2.5-0.5B stack), each a fused kv_append + "
                f"split-KV paged decode over its own pool; tables, lengths and slots shared")
        l2 = (f"inputs larger than L2: {layers} layer pools of "
              f"{2 * st.k_pool.nbytes / 1e6:.0f} MB each (L2 129 MB)")
    else:
        pool_mb = 2 * st.k_pool.size * st.kv_row_bytes(kv) // st.head_dim / 1e6
        l2 = (f"inputs larger than L2: {pools} rotating pool copies of "
              f"{pool_mb:.0f} MB each (L2 129 MB)")
    return {"workload": f"{st.name}: {name}" + (f" x {layers} layers" if layers > 1 else ""),
            "layers": layers, "num_seqs": st.num_seqs,
            "context_tokens": int(st.context_lens.sum()),
            "max_context": int(st.context_lens.max()),
            "num_q_heads": st.num_q_heads, "num_kv_heads": st.num_kv_heads,
            "head_dim": st.head_dim, "block_size": st.block_size,
            "num_blocks": st.num_blocks, "step": step, "query_tokens": st.num_tokens,
            "kv_cache": "q8_0 (int8 codes, fp16 scale per 32 elements)" if kv == "q8_0" else st.dtype,
            "decode_policy": dict(policy) if policy else "auto",
            "l2": l2}


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

def prefill_flops(st) -> int:
    """Tensor-core flops of the spans of 2+ rows: 4*D*Hq per (row, key it sees)."""
    f = 0
    for s in range(st.num_seqs):
        n, L = int(st.query_lens[s]), int(st.context_lens[s])
        if n >= 2:
            keys = n * (L - n) + n * (n + 1) // 2
            f += 4 * st.head_dim * st.num_q_heads * keys
    return f


class Step:
    """Device-resident state of one workload and the public-API call of one step.

    Decode workloads: one fused call (append the new token of every sequence
    and run the split-KV decode).  The mixed workload: ns_kv_append of all new
    tokens, then ns_paged_attn_prefill over every span.  With ``layers`` > 1
    (decode only) a step is that many fused calls, one per attention layer,
    each over its own pool, q and new K/V (drawn on the device from a seeded
    generator); block tables, lengths and slots are shared.
    """

    def __init__(self, st, dev, npools, layers=1, overlap=False, kv="native", policy=None):
        import torch
        from paged_kv_decode_ns_gb300 import binding as nb
        self.nb, self.torch, self.st, self.dev = nb, torch, st, dev
        self.kv = kv

        def dt_of(bits):
            t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev)
            return t.view(torch.bfloat16 if st.dtype == "bf16" else torch.float16)

        def ints(a, dt):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(dev)

        k0, v0 = dt_of(st.k_pool), dt_of(st.v_pool)
        self.pools = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(npools - 1)]
        self.npools = npools
        self.q = dt_of(st.q)
        self.k_new, self.v_new = dt_of(st.k_new), dt_of(st.v_new)
        self.slots = ints(st.slot_mapping, np.int64)
        self.tables = ints(st.block_tables, np.int32)
        self.lens = ints(st.context_lens, np.int32)
        self.qsl = ints(st.query_start_loc, np.int32)
        self.out = torch.empty_like(self.q)
        self.ws = nb.alloc_workspace(st.num_tokens, st.num_q_heads, st.num_kv_heads,
                                     st.head_dim, dev)
        self.decode = st.is_decode
        self.inputs = [self.q, self.k_new, self.v_new, self.slots, self.tables, self.lens]
        if not self.decode:
            self.inputs.append(self.qsl)
        # kernels per step: fused decode = 1; append + span rows + walk + tensor-core = 4
        self.launches = 1 if self.decode else 4
        self.layers = layers
        self.config = None
        if overlap or policy:
            self.config = nb.DecodeConfig()
        if overlap:  # programmatic dependent launches (see ns_decode_config.overlap_prologue)
            self.config.overlap_prologue = 1
        for k, v in (policy or {}).items():  # a forced split policy (decode workloads)
            setattr(self.config, k, v)
        self.layer_io = []
        self.q8pools = []
        self.stage, self.calls = 0, {}  # prepared calls by (buffer set, call)
        if kv == "q8_0":
            if not self.decode or layers > 1:
                raise ValueError("--kv q8_0 applies to single-layer decode workloads")
            # each pool copy quantised on the device by the library's own append
            # (every pool slot is a token), then the 16-bit copies are dropped
            self.q8pools = [self.quantize_pool(kp, vp) for kp, vp in self.pools]
            self.pools = [self.pools[0]]
        if layers > 1:
            if not self.decode:
                raise ValueError("layers > 1 applies to decode workloads")
            gen = torch.Generator(device=dev)
            gen.manual_seed(7000)

            def rnd(t):
                return torch.randn(t.shape, generator=gen, device=dev, dtype=torch.float32).to(t.dtype)
            self.layer_io.append((k0, v0, self.q, self.k_new, self.v_new, self.out))
            for _ in range(1, layers):
                self.layer_io.append((rnd(k0), rnd(v0), rnd(self.q), rnd(self.k_new), rnd(self.v_new),
                                      torch.empty_like(self.q)))
            self.inputs = ([t for io in self.layer_io for t in io[2:5]]
                           + [self.slots, self.tables, self.lens])
            self.out = self.layer_io[-1][5]  # read back end to end: the last layer's output
            self.launches = layers

    def quantize_pool(self, kp, vp):
        torch, nb = self.torch, self.nb
        NB, Hkv, bs, D = kp.shape
        kc = torch.empty((NB, Hkv, bs, D), dtype=torch.int8, device=self.dev)
        vc = torch.empty_like(kc)
        ks = torch.empty((NB, Hkv, bs, D // 32), dtype=torch.float16, device=self.dev)
        vs = torch.empty_like(ks)
        rows_k = kp.permute(0, 2, 1, 3).contiguous().view(NB * bs, Hkv, D)
        rows_v = vp.permute(0, 2, 1, 3).contiguous().view(NB * bs, Hkv, D)
        slots = torch.arange(NB * bs, dtype=torch.int64, device=self.dev)
        nb.ns_kv_append_q8_0(rows_k, rows_v, slots, kc, ks, vc, vs)
        return kc, ks, vc, vs

    def prepared(self, key, make):
        """The step's calls are prepared once per set of buffers (the binding's
        prepared calls: arguments checked and marshalled once), as a serving
        loop that repeats a step does; ``stage`` names the buffer set in use."""
        c = self.calls.get((self.stage,) + key)
        if c is None:
            c = self.calls[(self.stage,) + key] = make()
        return c

    def run_layer(self, layer, stream=None):
        nb = self.nb

        def make():
            kp, vp, q, kn, vn, out = self.layer_io[layer]
            return nb.prepare(nb.ns_kv_append_paged_attn_decode, q, kn, vn, self.slots, kp, vp,
                              self.tables, self.lens, self.st.scale, out, self.ws, config=self.config)
        self.prepared(("layer", layer), make)(stream)

    def run(self, i, stream=None):
        nb = self.nb
        if self.layers > 1:
            for layer in range(self.layers):
                self.run_layer(layer, stream)
            return
        if self.q8pools:
            p = i % len(self.q8pools)

            def make_q8():
                kc, ks, vc, vs = self.q8pools[p]
                return nb.prepare(nb.ns_kv_append_paged_attn_decode_q8_0, self.q, self.k_new, self.v_new,
                                  self.slots, kc, ks, vc, vs, self.tables, self.lens, self.st.scale,
                                  self.out, self.ws)
            self.prepared(("q8", p), make_q8)(stream)
            return
        p = i % self.npools
        kp, vp = self.pools[p]
        if self.decode:
            self.prepared(("decode", p), lambda: nb.prepare(
                nb.ns_kv_append_paged_attn_decode, self.q, self.k_new, self.v_new, self.slots, kp, vp,
                self.tables, self.lens, self.st.scale, self.out, self.ws, config=self.config))(stream)
        else:
            self.prepared(("append", p), lambda: nb.prepare(
                nb.ns_kv_append, self.k_new, self.v_new, self.slots, kp, vp))(stream)
            self.prepared(("prefill", p), lambda: nb.prepare(
                nb.ns_paged_attn_prefill, self.q, self.qsl, kp, vp, self.tables, self.lens,
                self.st.scale, self.out, self.ws))(stream)

    def run_dominant(self, i, stream=None):
        """The dominant kernel alone: the fused decode (one layer's), or the tensor-core prefill."""
        if self.layers > 1:
            return self.run_layer(i % self.layers, stream)
        if self.decode:
            return self.run(i, stream)
        nb = self.nb
        p = i % self.npools

        def make():
            kp, vp = self.pools[p]
            cfg = nb.PrefillConfig()
            cfg.phases = nb.NS_PREFILL_TENSOR_CORE
            return nb.prepare(nb.ns_paged_attn_prefill, self.q, self.qsl, kp, vp, self.tables, self.lens,
                              self.st.scale, self.out, self.ws, config=cfg)
        self.prepared(("tensor_core", p), make)(stream)


def stage_inputs(step, torch, dev):
    """Move the step's per-step inputs into one device buffer (their slices
    become the tensors the step uses) with a pinned host copy beside it, so
    that a step's inputs reach the device in one copy, as a serving loop
    stages its per-step metadata.  Returns (device buffer, host buffer)."""
    align = 256
    offs, total = [], 0
    for t in step.inputs:
        offs.append(total)
        total += (t.numel() * t.element_size() + align - 1) // align * align
    d_all = torch.empty(total, dtype=torch.uint8, device=dev)
    h_all = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    remap = {}
    for t, off in zip(step.inputs, offs):
        n = t.numel() * t.element_size()
        view = d_all[off:off + n].view(t.dtype).view(t.shape)
        view.copy_(t)
        h_all[off:off + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        remap[id(t)] = view

    def sub(x):
        return remap.get(id(x), x) if isinstance(x, torch.Tensor) else x
    for name, val in list(vars(step).items()):
        if isinstance(val, torch.Tensor):
            setattr(step, name, sub(val))
    step.layer_io = [tuple(sub(x) for x in io) for io in step.layer_io]
    step.inputs = [remap[id(t)] for t in step.inputs]
    step.stage, step.calls = 0, {}  # the staged views replace the buffers the calls were prepared on
    return d_all, h_all


def second_stage(step, d_all, torch):
    """A second set of the step's staged inputs and of its outputs, for a
    double-buffered end-to-end loop.  Returns (device buffer 2, use, outs):
    use(b) points the step at set b (0: the first staging, 1: the second) and
    outs[b] is the output that set's step reads back."""
    d_all2 = torch.empty_like(d_all)
    base, end = d_all.data_ptr(), d_all.data_ptr() + d_all.numel()

    def twin(t):
        if not isinstance(t, torch.Tensor) or not (base <= t.data_ptr() < end):
            return t
        off = t.data_ptr() - base
        n = t.numel() * t.element_size()
        return d_all2[off:off + n].view(t.dtype).view(t.shape)
    names = [k for k, v in vars(step).items() if isinstance(v, torch.Tensor) and twin(v) is not v]
    sets = [{k: getattr(step, k) for k in names}, {k: twin(getattr(step, k)) for k in names}]
    ios = [step.layer_io, [tuple(twin(x) for x in io) for io in step.layer_io]]
    if ios[1]:  # each layer's output (the last of its tensors) gets a twin too
        ios[1] = [io1[:-1] + (torch.empty_like(io0[-1]),) for io0, io1 in zip(ios[0], ios[1])]
        outs = [step.out, ios[1][-1][-1]]
    else:
        outs = [step.out, torch.empty_like(step.out)]

    def use(b):
        for k, v in sets[b].items():
            setattr(step, k, v)
        step.out = outs[b]
        step.layer_io = ios[b]
        step.stage = b
    return d_all2, use, outs


def hold_stream(torch, stream, calls):
    """Hold the stream with a device-side sleep long enough for the host to
    enqueue `calls` calls behind it, so that the device never waits for the
    host inside a timed region (a call's host side can take longer than its
    kernel)."""
    if hasattr(torch.cuda, "_sleep"):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(200_000 * calls))  # ~100 us of clock cycles per call


def time_events(torch, stream, fn, n):
    """Mean device time of fn(i) over n back-to-back calls between two events
    on the launch stream (ms), queued behind a hold of the stream."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(torch, stream, n)
    a.record(stream)
    for i in range(n):
        fn(i)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def bench_ours(args):
    import torch
    from paged_kv_decode_ns_gb300 import binding as nb

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    st = make_workload(args.workload)
    pool_bytes = 2 * st.k_pool.size * st.kv_row_bytes(args.kv) // st.head_dim
    npools = max(1, args.pools if args.pools else math.ceil(2 * L2_BYTES / max(pool_bytes, 1)))
    if args.layers > 1:
        npools = 1  # the layers' pools are the rotation
    step = Step(st, dev, npools, layers=args.layers, overlap=args.overlap, kv=args.kv, policy=decode_policy(args))
    stream = torch.cuda.current_stream(dev)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    for i in range(args.warmup):
        step.run(i)
    torch.cuda.synchronize(dev)
    nb.raise_on_device_status()

    # ---- timed region: K steps, device time, max over ranks
    barrier(dist)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(torch, stream, min(args.steps, 4000))
    e0.record(stream)
    for i in range(args.steps):
        step.run(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    elapsed_ms = e0.elapsed_time(e1)

    # ---- the same steps launched as programmatic dependents (opt-in in the
    # API: each launch's prologue may overlap the previous kernel's tail)
    overlap_us = None
    if step.decode and not args.overlap and args.steps >= 10 and args.kv == "native":
        plain_cfg, step.config = step.config, nb.DecodeConfig()
        step.config.overlap_prologue = 1
        n_ov = min(args.steps, 2000)
        for i in range(20):
            step.run(i)
        torch.cuda.synchronize(dev)
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        o0.record(stream)
        for i in range(n_ov):
            step.run(i)
        o1.record(stream)
        torch.cuda.synchronize(dev)
        overlap_us = 1e3 * o0.elapsed_time(o1) / n_ov
        step.config = plain_cfg

    # ---- the dominant kernel per launch (events on its stream)
    n_lat = max(3, min(args.steps, 200))
    launch_ms = time_events(torch, stream, step.run_dominant, n_lat)

    # ---- CUDA-graph replay of the same steps (launch overhead removed)
    graph_us = None
    if args.graph:
        per_graph = 2 * npools
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream(dev)
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            for i in range(per_graph):          # warm the capture stream's path
                step.run(i)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g):
            for i in range(per_graph):
                step.run(i)
        reps = max(3, args.steps // per_graph)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        graph_us = 1e3 * g0.elapsed_time(g1) / (reps * per_graph)
        del g

    # keep the GPU busy long enough for the clock sampler (untimed)
    t_end = time.time() + max(0.0, args.soak_s - elapsed_ms / 1e3)
    i = 0
    while time.time() < t_end:
        for _ in range(200):
            step.run(i)
            i += 1
        torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    nb.raise_on_device_status()

    # ---- end to end through the public API with host buffers: every step
    # copies its inputs from pinned host memory (one staged copy) and reads
    # its result back
    d_all, h_all = stage_inputs(step, torch, dev)
    h_out = torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True)
    h2d = h_all.numel()
    d2h = h_out.numel() * h_out.element_size()
    n_e2e = max(1, min(args.steps, args.e2e_steps))

    def e2e_step(i):
        d_all.copy_(h_all, non_blocking=True)
        step.run(i)
        h_out.copy_(step.out, non_blocking=True)
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for i in range(n_e2e):
        e2e_step(i)
    e3.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e2e_ms = e2.elapsed_time(e3)
    nb.raise_on_device_status()

    # ---- the same, double-buffered as a serving loop overlaps them: step
    # i+1's inputs upload, and step i's output is read back, on a copy stream
    # while the next step computes.  Every step still moves its own inputs and
    # its own output; the timed region ends when the last output is on the host.
    # Reported beside the serial loop: its host work per step is larger, so
    # small steps are bound by the host here.
    d_all2, use, out_bufs = second_stage(step, d_all, torch)
    d_bufs = [d_all, d_all2]
    h_outs = [h_out, torch.empty_like(h_out, pin_memory=True)]
    cs = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_pipelined(n, start_ev=None):
        with torch.cuda.stream(cs):
            if start_ev is not None:
                cs.wait_event(start_ev)
            d_bufs[0].copy_(h_all, non_blocking=True)
            ev_in[0].record(cs)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                nx = (i + 1) % 2
                with torch.cuda.stream(cs):
                    if i >= 1:
                        cs.wait_event(ev_done[nx])  # the step before read that buffer
                    d_bufs[nx].copy_(h_all, non_blocking=True)
                    ev_in[nx].record(cs)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # that output buffer is on the host
            use(b)
            step.run(i)
            ev_done[b].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_done[b])
                h_outs[b].copy_(out_bufs[b], non_blocking=True)
                ev_out[b].record(cs)
        stream.wait_event(ev_out[(n - 1) % 2])
    e2e_pipelined(4)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e4.record(stream)
    e2e_pipelined(n_e2e, e4)
    e5.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    use(0)
    e2e_ms_pipelined = e4.elapsed_time(e5)
    nb.raise_on_device_status()

    kv_bytes = st.kv_read_bytes(args.kv) * args.layers
    alg_bytes = st.algorithmic_bytes(with_append=True, kv=args.kv)  # one launch: one layer
    t_max, units = reduce_max_sum(dist, elapsed_ms, kv_bytes * args.steps, dev)
    te2e_max, units_e2e = reduce_max_sum(dist, e2e_ms, kv_bytes * n_e2e, dev)
    te2e_pipe_max, _ = reduce_max_sum(dist, e2e_ms_pipelined, kv_bytes * n_e2e, dev)
    if rank != 0:
        return None

    peaks, peak_src = measured_peaks()
    value = units / (t_max * 1e-3) / 1e9
    if step.decode:
        peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
        achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
        traffic = args.traffic if args.traffic is not None else (
            profiled_traffic(args.workload, "paged_decode_kernel") if args.kv == "native" else None)
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "traffic_source": traffic_source(args, traffic),
                    "kernel": "paged_decode_kernel (fused kv_append + split-KV decode"
                              + (", q8_0 pools)" if args.kv == "q8_0" else ")"),
                    "bytes_per_launch": alg_bytes, "launch_us": launch_ms * 1e3,
                    "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
    else:
        # fp16 and bf16 share the nominal dense tensor rate: bf16 peak x 1.0
        peak = float(peaks.get("bf16_tflops", 1900.0))
        flops = prefill_flops(st)
        achieved = flops / (launch_ms * 1e-3) / 1e12
        traffic = args.traffic if args.traffic is not None else profiled_traffic(args.workload,
                                                                                  "tc_prefill_kernel")
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "traffic_source": traffic_source(args, traffic),
                    "kernel": "tc_prefill_kernel (tcgen05, spans of 2+ rows)",
                    "flops_per_launch": flops, "launch_us": launch_ms * 1e3,
                    "peak_source": f"{peak_src} bf16_tflops (burst) x nominal fp16/bf16 ratio 1.0"}
    cpu = None
    if args.cpu_baseline:
        cores = host_cores()
        max_seqs = None if step.decode else 16
        secs, kvb, n, thr = run_cpu_oracle(st, cores, max_seqs=max_seqs)
        # one thread on a bounded sample (the first 32 sequences)
        secs1, kvb1, n1, _ = run_cpu_oracle(st, 1, max_seqs=32 if max_seqs is None else min(32, max_seqs))
        cpu = {"value": kvb / secs / 1e9, "unit": "GB/s", "cores": thr, "kind": "oracle",
               "sample": f"{'all' if n == st.num_seqs else 'first'} {n} sequences of the "
                         f"batch (decode rows), attention only, one pass, {secs:.2f} s "
                         f"(fp64 C oracle, OpenMP over (row, head))",
               "value_1thread": kvb1 / secs1 / 1e9,
               "sample_1thread": f"first {n1} sequences, one thread, {secs1:.2f} s"}
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_max / args.steps, "us_per_step": 1e3 * t_max / args.steps,
        "graph_us_per_step": graph_us, "hbm_peak_frac": value / float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS)),
        "overlap_us_per_step": overlap_us,
        "layer_us": ({"eager": 1e3 * t_max / args.steps / args.layers,
                      "graph": graph_us / args.layers if graph_us else None}
                     if args.layers > 1 else None),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": st.dtype, "data": "synthetic (seeded; no dataset or weights involved)",
        "config": dict(workload_config(st, args.workload, npools, args.layers, args.kv, decode_policy(args)),
                       overlap_prologue=bool(args.overlap)),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": units_e2e / (te2e_max * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": 1e3 * te2e_max / n_e2e, "steps": n_e2e,
                "loop": "serial: upload, call, read-back on one stream",
                "pipelined_us_per_step": 1e3 * te2e_pipe_max / n_e2e},
        "gpu_launches": args.steps * step.launches,
        "clocks": clocks,
        # the device's record of the last call's split (decode workloads)
        "plan": nb.ns_read_decode_plan(step.ws) if st.is_decode and args.layers == 1 else None,
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
    ap.add_argument("--overlap", action="store_true",
                    help="decode launches as programmatic dependents (a prologue may overlap the "
                         "previous kernel's tail); off for the default line")
    ap.add_argument("--kv", choices=["native", "q8_0"], default="native",
                    help="KV pool format: the workload's 16-bit type, or the 8-bit q8_0 cache")
    ap.add_argument("--layers", type=int, default=1,
                    help="attention layers per step (decode workloads; 24 = the Qwen2.5-0.5B stack)")
    ap.add_argument("--pools", type=int, default=0, help="rotating pool copies (0 = enough to exceed 2x L2)")
    ap.add_argument("--whole-sequences", action="store_true",
                    help="force whole (sequence, kv head) pairs per worker (no split, no merge)")
    ap.add_argument("--min-blocks-per-cta", type=int, default=0,
                    help="force the split's minimum KV blocks per CTA (0 = automatic)")
    ap.add_argument("--num-ctas", type=int, default=0, help="force the decode grid (0 = one CTA per SM)")
    ap.add_argument("--merge-levels", type=int, default=0, choices=[0, 1, 2],
                    help="force one- or two-level merges of cut pairs (0 = automatic)")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--soak-s", type=float, default=1.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch from an ncu capture of the current kernel")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    res = bench_reference(args) if args.impl == "reference" else bench_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
