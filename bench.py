"""Benchmark: one decode step of paged attention on GB300.

A step is the whole hot path on one batch: reshape_and_cache of the batch's
new tokens, then decode over every sequence's paged K/V history.  The default
workload is the LLaMA-7B-shaped layer (64 sequences, 32 heads, head_dim 128,
16-token blocks, contexts uniform in [128, 2048], shuffled block placement,
64 new tokens), with seeded synthetic fp16 N(0, 1) inputs.

Prints one JSON line.  `value` is KV GB/s of the step (algorithmic bytes: K
and V of every context token, q, the output, the table entries used, the
context lengths and the new tokens' K/V in and out, divided by the step time,
device-timed with inputs resident in HBM).  The `roofline` object covers the
dominant kernel (decode) against the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "pa_decode KV GB/s and % of GB300 HBM peak; decode tokens/s (seq·layer/s)"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ("paged_kv_cache_269_gb300/csrc/pa_decode.cu",
                  "paged_kv_cache_269_gb300/csrc/pa_device.cuh")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--op", choices=["step", "copy_blocks", "swap_out", "swap_in", "prefill",
                                    "shared_prefix", "variants"],
                   default="step",
                   help="step: reshape_and_cache + decode (the hot path); the others time "
                        "pa_copy_blocks on a 4096-block pool, 2048 random pairs")
    p.add_argument("--workload", default="llama7b_b64",
                   choices=workloads.WORKLOADS + workloads.PREFILL_WORKLOADS)
    p.add_argument("--partition-tokens", type=int, default=0)
    p.add_argument("--dtype", choices=["f16", "bf16"], default="f16",
                   help="element type of q, the caches and the output")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="CPU work the oracle baseline leg runs for (bounded sample)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--ref-seconds", type=float, default=120.0,
                   help="--impl reference: oracle time the whole run is sized for")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other workloads' decode (and shared-prefix call) timings "
                        "that the step line carries under \"workloads\"")
    p.add_argument("--flush-l2", action="store_true",
                   help="write a 256 MiB buffer, then read another, before every step so "
                        "shared blocks start cold and L2 holds no dirty lines; "
                        "step time then sums per-step events and excludes the flush")
    return p.parse_args()


def step_bytes(case):
    return workloads.decode_algorithmic_bytes(case) + workloads.reshape_algorithmic_bytes(case)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def decode_source_hash():
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ("paged_kv_cache_269_gb300/csrc/pa_prefill.cu",)


def recorded_prefill_traffic(workload):
    """DRAM bytes (read + write) per prefill launch from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"pa_prefill_{workload.replace('prefill_', '')}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path, encoding="utf-8"):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    h = hashlib.sha256()
    for rel in PREFILL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if vals.get("kernel_source_sha256_16") != h.hexdigest()[:16]:
        return None
    try:
        return int(float(vals["dram_bytes_read"]) + float(vals["dram_bytes_write"]))
    except (KeyError, ValueError):
        return None


SHARED_SOURCES = DECODE_SOURCES + PREFILL_SOURCES


def recorded_shared_traffic(workload):
    """DRAM bytes (read + write) of one shared-prefix call (the prefix kernel
    plus the suffix decode) on a workload from the committed ncu summary, if
    it was taken on the current sources of both kernels; else None."""
    path = os.path.join(ROOT, "profiles", f"pa_shared_prefix_call_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path, encoding="utf-8"):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    h = hashlib.sha256()
    for rel in SHARED_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if vals.get("kernel_source_sha256_16") != h.hexdigest()[:16]:
        return None
    try:
        return int(float(vals["dram_bytes_per_call"]))
    except (KeyError, ValueError):
        return None


def recorded_traffic(workload):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"pa_decode_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path, encoding="utf-8"):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != decode_source_hash():
        return None
    try:
        return int(float(vals["dram_bytes_per_launch_full_size"]))
    except (KeyError, ValueError):
        return None


class L2Flush:
    """Evicts L2 before a timed call: a 256 MiB write (twice L2) replaces
    every cached input line, then a 256 MiB read of a second buffer replaces
    the write's dirty lines with clean ones.  Without the read, the timed
    call pays for writing those 128 MB back to HBM as it evicts them (16 us
    on a 100 us HBM-bound decode); with it, the call starts with neither its
    inputs nor dirty lines in L2."""

    def __init__(self, torch, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.int32, device=dev)

    def __call__(self, torch, stream):
        with torch.cuda.stream(stream):
            self.w.fill_(1)
            self.r.sum()


class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms; summary() keeps the
    samples whose nvidia-smi timestamp falls inside a time window."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.samples = []
        self.thread = None

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.samples.append((time.time(), line))

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1, window="timed region"):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        import datetime
        for arrival, l in self.samples:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                t = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = arrival
            if not (t0 <= t <= t1):
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


# ----------------------------------------------------------------------------
# oracle (CPU) legs
# ----------------------------------------------------------------------------

def subset_case(case, idx):
    """The decode case restricted to sequences idx (their new tokens with
    them), sharing the caches."""
    import dataclasses
    idx = np.asarray(idx)
    sub = dataclasses.replace(case, context_lens=case.context_lens[idx],
                              block_tables=case.block_tables[idx], q=case.q[idx])
    if case.num_new_tokens:
        # one new token per sequence with ctx > 0, in sequence order
        has = case.context_lens > 0
        tok = np.cumsum(has) - 1
        t = tok[idx[has[idx]]]
        sub.k_new, sub.v_new, sub.slot_mapping = case.k_new[t], case.v_new[t], case.slot_mapping[t]
    return sub


def oracle_pass(case, kc, vc, lib):
    """One pass of the oracle over the case: reshape_and_cache into the given
    caches (in place), then decode.  Returns the seconds it took."""
    import oracle
    t0 = time.perf_counter()
    if case.num_new_tokens:
        oracle.reshape_and_cache_into(case.k_new, case.v_new, kc, vc, case.slot_mapping, lib=lib)
    oracle.decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale, lib=lib,
                  dtype=case.dtype)
    return time.perf_counter() - t0


def oracle_sample(case, seconds):
    """Time the oracle, as it stands, on the whole workload (repeated until
    `seconds` of CPU work have run, at least once).  The caches are copied
    once, outside the timing."""
    import oracle
    lib = oracle.load()
    kc = np.array(case.k_cache, copy=True, order="C")
    vc = np.array(case.v_cache, copy=True, order="C")
    runs, el = 0, 0.0
    while True:
        el += oracle_pass(case, kc, vc, lib)
        runs += 1
        if el >= seconds:
            break
    return el / runs, runs, oracle.num_threads(lib)


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    lib = oracle.load()
    case = workloads.make_workload(args.workload, dtype=args.dtype)
    S = case.num_seqs
    kc = np.array(case.k_cache, copy=True, order="C")
    vc = np.array(case.v_cache, copy=True, order="C")
    # Each step is a bounded sample of the workload: a rotating window of n
    # sequences, n chosen from one full pass so that the whole run takes about
    # --ref-seconds (every sequence when the full pass fits).
    full = oracle_pass(case, kc, vc, lib)
    per_step = args.ref_seconds / max(1, args.warmup + args.steps)
    n = S if full <= per_step else max(1, int(S * per_step / full))
    secs, nbytes = 0.0, 0
    for i in range(args.warmup + args.steps):
        idx = (np.arange(n) + i * n) % S
        sub = case if n == S else subset_case(case, idx)
        t = oracle_pass(sub, kc, vc, lib)
        if i >= args.warmup:
            secs += t
            nbytes += step_bytes(sub)
    value = nbytes / secs / 1e9
    ms_step = secs / args.steps * 1e3
    sample = (f"each step: the fp64 C oracle (OpenMP) over reshape_and_cache + decode of "
              + ("the whole workload" if n == S else
                 f"a rotating window of {n} of the {S} sequences (bytes counted for those)"))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(case, args),
        "tokens_per_s": round(n * args.steps / secs, 2),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.num_threads(lib),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def max_over_ranks(values, dist, device):
    """Element-wise maximum of `values` over all ranks (a list of floats; the
    same list on one rank)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_value(world, bytes_per_step_per_rank, step_ms):
    """Whole-job GB/s: every rank moves its bytes in each step; the step time
    is the slowest rank's."""
    return world * bytes_per_step_per_rank / (step_ms * 1e-3) / 1e9


def config_of(case, args):
    return {"workload": args.workload, "num_seqs": case.num_seqs, "num_heads": case.num_heads,
            "head_dim": case.head_dim, "block_size": case.block_size,
            "num_blocks": case.num_blocks, "max_blocks_per_seq": case.max_blocks_per_seq,
            "total_context_tokens": int(case.context_lens.sum()),
            "new_tokens": case.num_new_tokens,
            "l2": ("flushed before every step (256 MiB write, then 256 MiB read of another "
                          "buffer; excluded from the step time)"
                   if getattr(args, "flush_l2", False) else
                   "inputs larger than L2 (no flush)" if 2 * case.k_cache.nbytes > L2_BYTES
                   else "inputs smaller than L2"),
            "parallelism": f"dp{args.gpus} (replicas)", "seed": case.seed,
            "launch": ("eager, events around every step" if getattr(args, "flush_l2", False) else
                       f"timed steps replayed from CUDA graphs of up to {STEP_GRAPH} steps, "
                       "captured and uploaded during the warm-up")}


# ----------------------------------------------------------------------------
# native leg
# ----------------------------------------------------------------------------

STEP_GRAPH = 64                 # timed steps per captured CUDA graph


def upload_graphs(graphs, stream):
    """Upload captured graphs to the device (cuGraphUpload) ahead of their
    first replay, so that the timed region does not pay for it; nothing runs.
    Skipped where this torch does not expose the executable graph."""
    import ctypes
    try:
        cuda = ctypes.CDLL("libcuda.so.1")
        execs = [g.raw_cuda_graph_exec() for g in graphs]
    except (OSError, AttributeError, RuntimeError):
        return False
    cuda.cuGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    cuda.cuGraphUpload.restype = ctypes.c_int
    ok = all(cuda.cuGraphUpload(ctypes.c_void_p(e), ctypes.c_void_p(stream.cuda_stream)) == 0
             for e in execs)
    stream.synchronize()
    return ok
ROOFLINE_MIN_LAUNCHES = 200     # decode-only launches timed for the roofline
ROOFLINE_MIN_SECONDS = 0.5      # ... and at least this long, so the clock sampler sees it


SIDE_WORKLOADS = ("tiny", "llama7b_b64", "cb_mix", "shared_prefix", "long_ctx", "cb_mix_1k",
                  "cb_mix_4k")
SIDE_SHARED = ("shared_prefix", "shared_prefix_4k")
SIDE_MIN_SECONDS = 0.25
SIDE_GRAPH = 20                 # decode launches per captured graph


def side_workloads(args, dev):
    """The other decode workloads, timed in the same run as the step line:
    each workload's decode alone (its block tables and lengths, q and caches
    drawn on the device), back to back between two events from a replayed
    CUDA graph of SIDE_GRAPH launches, at least ROOFLINE_MIN_LAUNCHES
    launches and SIDE_MIN_SECONDS; then the
    shared-prefix call against pa_decode on each shared-prefix batch, one call
    per L2 flush.  Fractions are of the measured HBM copy rate."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    peak, _ = measured_peaks()
    et = torch.bfloat16 if args.dtype == "bf16" else torch.float16
    dt = 1 if args.dtype == "bf16" else 0
    stream = torch.cuda.Stream(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)

    def on_device(case):
        t = {k: torch.from_numpy(np.ascontiguousarray(getattr(case, k))).to(dev)
             for k in ("block_tables", "context_lens")}
        for k in ("q", "k_cache", "v_cache"):
            t[k] = torch.randn(getattr(case, k).shape, generator=gen, device=dev, dtype=et)
        return t

    def decode_fn(case, d):
        ws = torch.empty(max(16, pa.decode_workspace_bytes(
            case.num_seqs, case.num_heads, case.head_dim, case.block_size, case.num_blocks,
            case.max_blocks_per_seq, args.partition_tokens, dtype=dt)), dtype=torch.uint8,
            device=dev)
        ctr = torch.zeros(pa.decode_counters_bytes(case.num_seqs, case.num_heads) // 4,
                          dtype=torch.int32, device=dev)
        out = torch.empty(case.q.shape, dtype=et, device=dev)
        return lambda: pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                 d["context_lens"], case.scale,
                                 partition_tokens=args.partition_tokens, workspace=ws,
                                 counters=ctr, stream=stream)

    res = {}
    sampler = ClockSampler(dev.index or 0) if not args.no_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_begin = time.time()
    for w in SIDE_WORKLOADS:
        if w == args.workload:
            continue
        case = workloads.make_workload(w, values=False, dtype=args.dtype)
        d = on_device(case)
        fn = decode_fn(case, d)
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        # SIDE_GRAPH launches captured once and replayed, so that the host's
        # per-call cost does not pace small batches
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(SIDE_GRAPH):
                fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            graph.replay()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        est = e0.elapsed_time(e1) / SIDE_GRAPH
        n = max(ROOFLINE_MIN_LAUNCHES, int(SIDE_MIN_SECONDS * 1e3 / max(est, 1e-3)) + 1)
        reps = min(20000, (n + SIDE_GRAPH - 1) // SIDE_GRAPH)
        n = reps * SIDE_GRAPH
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / n
        del graph
        if pa.device_errors(stream=stream):
            raise RuntimeError(f"device error in the {w} decode")
        alg = workloads.decode_algorithmic_bytes(case)
        uq = workloads.decode_unique_bytes(case)
        res[w] = {"decode_ms": round(ms, 4), "gbs": round(alg / (ms * 1e-3) / 1e9, 2),
                  "frac": round(alg / (ms * 1e-3) / 1e9 / peak, 4),
                  "unique_gbs": round(uq / (ms * 1e-3) / 1e9, 2),
                  "unique_frac": round(uq / (ms * 1e-3) / 1e9 / peak, 4),
                  "num_seqs": case.num_seqs, "num_heads": case.num_heads, "launches": n}
        del d, fn
        torch.cuda.empty_cache()
    flush = L2Flush(torch, dev)
    for w in SIDE_SHARED:
        case = workloads.make_workload(w, values=False, dtype=args.dtype)
        d = on_device(case)
        S = case.num_seqs
        gs = torch.tensor([0, S], dtype=torch.int32, device=dev)
        gp = torch.tensor([case.shared_prefix_blocks], dtype=torch.int32, device=dev)
        ws = torch.empty(pa.decode_shared_prefix_workspace_bytes(
            S, case.num_heads, case.head_dim, case.block_size, case.num_blocks,
            case.max_blocks_per_seq, args.partition_tokens, dtype=dt), dtype=torch.uint8,
            device=dev)
        ctr = torch.zeros(pa.decode_shared_prefix_counters_bytes(
            S, case.num_heads, case.head_dim, case.block_size, case.num_blocks) // 4,
            dtype=torch.int32, device=dev)
        out = torch.empty(case.q.shape, dtype=et, device=dev)

        def shared():
            pa.decode_shared_prefix(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                    d["context_lens"], case.scale, gs, gp, max_group_size=S,
                                    partition_tokens=args.partition_tokens, counters=ctr,
                                    workspace=ws, stream=stream)

        plain = decode_fn(case, d)

        def per_call(fn, calls):
            for _ in range(3):
                fn()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(calls)]
            for a0, a1 in evs:
                flush(torch, stream)
                a0.record(stream)
                fn()
                a1.record(stream)
            torch.cuda.synchronize(dev)
            return sum(a0.elapsed_time(a1) for a0, a1 in evs) / calls

        calls = 100 if S <= 256 else 20
        ms_s, ms_p = per_call(shared, calls), per_call(plain, calls)
        if pa.device_errors(stream=stream):
            raise RuntimeError(f"device error in the {w} shared-prefix call")
        uq = workloads.decode_unique_bytes(case)
        res[w + "_shared_call"] = {
            "ms": round(ms_s, 4), "unique_gbs": round(uq / (ms_s * 1e-3) / 1e9, 2),
            "unique_frac": round(uq / (ms_s * 1e-3) / 1e9 / peak, 4),
            "plain_decode_ms": round(ms_p, 4), "speedup_vs_plain": round(ms_p / ms_s, 3),
            "num_seqs": S, "num_heads": case.num_heads, "calls": calls}
        del d
        torch.cuda.empty_cache()
    t_end = time.time()
    if sampler:
        time.sleep(0.1)
        sampler.stop()
    return {"method": "decode alone: back-to-back launches between two events, replayed from "
                      f"a CUDA graph of {SIDE_GRAPH} launches (at least {ROOFLINE_MIN_LAUNCHES} "
                      f"launches and {SIDE_MIN_SECONDS} s), inputs larger than L2 except tiny; "
                      "shared-prefix call and pa_decode on its batch: one call per "
                      "L2 flush (256 MiB write, then 256 MiB read), mean over the calls; q and "
                      "caches drawn on the device; fractions of the measured HBM copy rate",
            "dtype": args.dtype, "results": res,
            "clocks": sampler.summary(t_begin, t_end, "these timings") if sampler else None}


def run_native(args, rank, world, local_rank):
    import torch
    import paged_kv_cache_269_gb300 as pa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pa.lib()
    case = workloads.make_workload(args.workload, new_tokens=True, dtype=args.dtype)
    et = torch.bfloat16 if args.dtype == "bf16" else torch.float16

    def t(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:  # bf16 bit patterns
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    d = dict(q=t(case.q), k_cache=t(case.k_cache), v_cache=t(case.v_cache),
             block_tables=t(case.block_tables), context_lens=t(case.context_lens),
             k_new=t(case.k_new), v_new=t(case.v_new), slot_mapping=t(case.slot_mapping))
    out = torch.empty(case.q.shape, dtype=et, device=dev)
    stream = torch.cuda.Stream(dev)
    nws = pa.decode_workspace_bytes(case.num_seqs, case.num_heads, case.head_dim,
                                    case.block_size, case.num_blocks, case.max_blocks_per_seq,
                                    args.partition_tokens, dtype=1 if args.dtype == "bf16" else 0)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    ctr = torch.zeros(pa.decode_counters_bytes(case.num_seqs, case.num_heads) // 4,
                      dtype=torch.int32, device=dev)
    torch.cuda.synchronize(dev)

    flush = L2Flush(torch, dev) if args.flush_l2 else None

    def decode_only(ins):
        pa.decode(out, ins["q"], d["k_cache"], d["v_cache"], ins["block_tables"],
                  ins["context_lens"], case.scale, partition_tokens=args.partition_tokens,
                  workspace=ws, counters=ctr, stream=stream)

    def step(ins, ev=None):
        if flush is not None:
            flush(torch, stream)
        if ev is not None:
            ev[2].record(stream)
        pa.reshape_and_cache(ins["k_new"], ins["v_new"], d["k_cache"], d["v_cache"],
                             ins["slot_mapping"], stream=stream)
        if ev is not None:
            ev[0].record(stream)
        decode_only(ins)
        if ev is not None:
            ev[1].record(stream)

    dist = None
    if world > 1:
        import torch.distributed as dist

    # The clock sampler starts before the warm-up, so that its start-up pause
    # never leaves the GPU idle between the warm-up and the timed steps.
    sampler = ClockSampler(local_rank) if not args.no_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # The first warm-up step runs the library's per-device set-up outside any
    # capture; the timed steps' graphs are captured and uploaded (nothing
    # runs) after it, so that the remaining warm-up steps lead straight into
    # the timed region with no idle GPU in between.
    step(d)
    torch.cuda.synchronize(dev)
    graphs = []
    if not args.flush_l2:
        left = args.steps
        while left > 0:
            n = min(left, STEP_GRAPH)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(n):
                    step(d)
            graphs.append(g)
            left -= n
        upload_graphs(graphs, stream)
    for _ in range(max(3, args.warmup) - 1):
        step(d)
    torch.cuda.synchronize(dev)
    if pa.device_errors(stream=stream):
        raise RuntimeError("device error during warm-up")

    # With --flush-l2 every step carries events around its kernels (the step
    # time is built from them, flush excluded).  Otherwise the K steps are
    # replayed from the CUDA graphs captured above (up to STEP_GRAPH steps
    # each), with no event between their kernels, so each decode may launch
    # early behind its reshape_and_cache and one host call submits many steps.
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
           for _ in range(args.steps)] if args.flush_l2 else [None] * args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_begin = time.time()
    start.record(stream)
    if graphs:
        with torch.cuda.stream(stream):
            for g in graphs:
                g.replay()
    else:
        for i in range(args.steps):
            step(d, evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    del graphs
    step_ms = start.elapsed_time(end) / args.steps
    if args.flush_l2:  # per-step events around reshape + decode, flush excluded
        step_ms = sum(e[2].elapsed_time(e[1]) for e in evs) / args.steps
    if pa.device_errors(stream=stream):
        raise RuntimeError("device error during the timed steps")

    # The decode kernel's own duration, for the roofline: right after the
    # steps, back-to-back decode launches between two events on the launching
    # stream, at least ROOFLINE_MIN_LAUNCHES of them and at least
    # ROOFLINE_MIN_SECONDS.  With --flush-l2, every decode of the timed steps
    # was bracketed by events after a flush; their mean is used instead.
    if args.flush_l2:
        decode_ms_each = [e[0].elapsed_time(e[1]) for e in evs]
        decode_ms = sum(decode_ms_each) / len(decode_ms_each)
        n_roof = len(decode_ms_each)
        sampling = (f"CUDA events around the decode of each of the {n_roof} timed steps, "
                    f"L2 flushed before each step")
    else:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(20):
            decode_only(d)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        est_ms = e0.elapsed_time(e1) / 20
        n_roof = max(ROOFLINE_MIN_LAUNCHES, int(ROOFLINE_MIN_SECONDS * 1e3 / max(est_ms, 1e-3)) + 1)
        n_roof = min(n_roof, 200000)
        e0.record(stream)
        for _ in range(n_roof):
            decode_only(d)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        decode_ms = e0.elapsed_time(e1) / n_roof
        decode_ms_each = [decode_ms]
        sampling = (f"{n_roof} back-to-back decode launches between two CUDA events on the "
                    f"launching stream, right after the timed steps "
                    f"({decode_ms * n_roof / 1e3:.2f} s)")
    t_end = time.time()
    if dist:
        dist.barrier()
    if sampler:
        time.sleep(0.1)
        sampler.stop()
    if pa.device_errors(stream=stream):
        raise RuntimeError("device error during the roofline launches")

    # e2e: per-step inputs from pinned host memory, result read back every step
    e2e = None
    if not args.no_e2e:
        # The step's inputs packed into one pinned host buffer (256-byte
        # aligned fields) so that a step makes one host-to-device copy.
        names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
        arrays = {k: np.ascontiguousarray(getattr(case, k)) for k in names}
        offsets, total = {}, 0
        for k in names:
            offsets[k] = total
            total += (arrays[k].nbytes + 255) // 256 * 256
        host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        hb = host_buf.numpy()
        for k in names:
            hb[offsets[k]:offsets[k] + arrays[k].nbytes] = arrays[k].view(np.uint8).reshape(-1)
        dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
        tdt = {np.dtype(np.float16): torch.float16, np.dtype(np.int32): torch.int32,
               np.dtype(np.uint16): torch.bfloat16}
        dev_in = {k: dev_buf[offsets[k]:offsets[k] + arrays[k].nbytes].view(
            tdt[arrays[k].dtype]).view(arrays[k].shape) for k in names}
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = total
        d2h = out_host.numel() * out_host.element_size()

        def e2e_step():
            with torch.cuda.stream(stream):
                dev_buf.copy_(host_buf, non_blocking=True)
            step(dev_in)
            with torch.cuda.stream(stream):
                out_host.copy_(out, non_blocking=True)
            stream.synchronize()

        def timed(fn):
            for _ in range(3):
                fn()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            for _ in range(args.steps):
                fn()
            return (time.perf_counter() - t0) / args.steps

        eager_s = timed(e2e_step)
        # the same step through the package's graph-replayed step runner: one
        # graph launch per step holds the host-to-device copy of the packed
        # inputs, reshape_and_cache, decode and the copy of the output into
        # pinned host memory
        from paged_kv_cache_269_gb300.step import DecodeStep
        runner = DecodeStep(d["k_cache"], d["v_cache"], case.num_seqs, case.max_blocks_per_seq,
                            case.scale, use_graph=True, partition_tokens=args.partition_tokens,
                            stream=stream, host_out=True)
        runner.prepare(case.q, case.k_new, case.v_new, case.slot_mapping, case.block_tables,
                       case.context_lens)

        def graph_step():   # one graph launch: H2D, reshape_and_cache, decode, D2H
            runner.launch()
            stream.synchronize()

        graph_s = timed(graph_step)

        # pipelined: two staging slots in turn; step k + 1's packed inputs are
        # copied to the device on a copy stream while step k's graph runs, and
        # the host takes step k's output (written into pinned host memory by
        # the decode) once step k + 1 is launched.  Every step still makes its
        # host-to-device copy and returns its output to the host inside the
        # timed region; the last step is waited for before the clock stops.
        from paged_kv_cache_269_gb300.step import PipelinedDecodeStep
        pipe = PipelinedDecodeStep(d["k_cache"], d["v_cache"], case.num_seqs,
                                   case.max_blocks_per_seq, case.scale, use_graph=True,
                                   partition_tokens=args.partition_tokens, stream=stream,
                                   host_out=True)
        for _ in range(2):
            pipe.prepare(case.q, case.k_new, case.v_new, case.slot_mapping, case.block_tables,
                         case.context_lens)
            pipe.result(pipe.launch())

        def pipelined_run(n):
            prev = None
            for _ in range(n):
                t = pipe.launch()
                if prev is not None:
                    pipe.result(prev)
                prev = t
            pipe.result(prev)

        pipelined_run(3)
        if dist:
            dist.barrier()
        t0 = time.perf_counter()
        pipelined_run(args.steps)
        pipe_s = (time.perf_counter() - t0) / args.steps
        e2e_s = min(eager_s, graph_s, pipe_s)
        e2e_s = max_over_ranks([e2e_s], dist, dev)[0]
        e2e = {"value": round(job_value(world, step_bytes(case), e2e_s * 1e3), 3), "unit": UNIT,
               "ms_per_step": round(e2e_s * 1e3, 4),
               "ms_per_step_eager": round(eager_s * 1e3, 4),
               "ms_per_step_graph": round(graph_s * 1e3, 4),
               "ms_per_step_pipelined": round(pipe_s * 1e3, 4),
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    step_ms, decode_ms = max_over_ranks([step_ms, decode_ms], dist, dev)

    if rank != 0:
        return
    # the other workloads, timed in this run (one GPU runs them; at N > 1 the
    # ranks would only repeat them)
    side = side_workloads(args, dev) if world == 1 and not args.no_workloads else None
    peak, peak_kind = measured_peaks()
    dec_bytes = workloads.decode_algorithmic_bytes(case)
    uniq_bytes = workloads.decode_unique_bytes(case)
    achieved = dec_bytes / (decode_ms * 1e-3) / 1e9
    value = job_value(world, step_bytes(case), step_ms)
    cpu = None
    if not args.no_cpu_baseline:
        sec, runs, cores = oracle_sample(case, args.cpu_seconds)
        cpu = {"value": round(step_bytes(case) / sec / 1e9, 4), "unit": UNIT, "cores": cores,
               "kind": "oracle",
               "sample": f"full {args.workload} step (reshape_and_cache + decode), "
                         f"{runs} run(s), {sec:.2f} s each"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic", "config": config_of(case, args),
        "tokens_per_s": round(world * case.num_seqs / (step_ms * 1e-3), 1),
        "pct_of_peak": round(100 * value / peak, 2),
        "decode_ms": round(decode_ms, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": "pa_decode",
                     "duration_sampling": sampling,
                     "launches_timed": int(n_roof),
                     "algorithmic_bytes_per_launch": int(dec_bytes),
                     "unique_bytes_per_launch": int(uniq_bytes),
                     "achieved_unique": round(uniq_bytes / (decode_ms * 1e-3) / 1e9, 2),
                     "traffic": recorded_traffic(args.workload)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(t_begin, t_end, "timed steps and the decode launches timed "
                                  "for the roofline") if sampler else None,
        "workloads": side,
    }
    print(json.dumps(line))


def run_copy_op(args, local_rank):
    """Time pa_copy_blocks: device -> device (copy-on-write), device -> pinned
    host (swap out) or pinned host -> device (swap in)."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    N, H, B, D, n = 4096, 32, 16, 128, 2048
    g = torch.Generator(device=dev).manual_seed(11)
    kc = torch.randn((N, H, B, D), generator=g, device=dev).half()
    vc = torch.randn((N, H, B, D), generator=g, device=dev).half()
    src = torch.randperm(N, device=dev, generator=g)[:n]
    block_bytes = H * B * D * 2
    if args.op == "copy_blocks":
        dk, dv = torch.empty_like(kc), torch.empty_like(vc)
        pairs = torch.stack([src, torch.randperm(N, device=dev, generator=g)[:n]], 1)
        a_k, a_v, b_k, b_v = kc, vc, dk, dv
    elif args.op == "swap_out":
        b_k = torch.empty((n, H, B, D), dtype=torch.float16).pin_memory()
        b_v = torch.empty_like(b_k).pin_memory()
        pairs = torch.stack([src, torch.arange(n, device=dev)], 1)
        a_k, a_v = kc, vc
    else:  # swap_in
        a_k = torch.randn((n, H, B, D)).half().pin_memory()
        a_v = torch.randn((n, H, B, D)).half().pin_memory()
        pairs = torch.stack([torch.arange(n, device=dev), src], 1)
        b_k, b_v = kc, vc
    pairs = pairs.to(torch.int32).contiguous()
    stream = torch.cuda.Stream(dev)
    call = lambda: pa.copy_blocks(a_k, a_v, b_k, b_v, pairs, stream=stream)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize(dev)
    assert pa.device_errors(stream=stream) == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    moved = 2 * n * block_bytes                   # K and V, one direction
    if args.op == "copy_blocks":
        alg, peak, src_note = 2 * moved, measured_peaks()[0], "MEASURED_PEAKS.json hbm_gbs"
    else:
        # the link ceiling measured here: one contiguous cudaMemcpyAsync of
        # the same byte count in the same direction
        host = torch.empty(moved // 2, dtype=torch.float16).pin_memory()
        devbuf = torch.empty(moved // 2, dtype=torch.float16, device=dev)
        cp = (lambda: host.copy_(devbuf, non_blocking=True)) if args.op == "swap_out" else \
             (lambda: devbuf.copy_(host, non_blocking=True))
        with torch.cuda.stream(stream):
            for _ in range(3):
                cp()
            e0.record(stream)
            for _ in range(args.steps):
                cp()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        alg = moved
        peak = moved / (e0.elapsed_time(e1) / args.steps * 1e-3) / 1e9
        src_note = "contiguous cudaMemcpyAsync of the same bytes, measured in this run"
    achieved = alg / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": f"pa_copy_blocks {args.op} GB/s", "value": round(achieved, 2), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "f16",
        "data": "synthetic",
        "config": {"op": args.op, "pool_blocks": N, "pairs": n, "num_heads": H, "block_size": B,
                   "head_dim": D, "block_bytes_k_plus_v": 2 * block_bytes},
        "roofline": {"bound": "hbm" if args.op == "copy_blocks" else "host link",
                     "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": src_note,
                     "algorithmic_bytes_per_launch": int(alg)},
        "gpu_launches": args.steps}))


def run_prefill_op(args, local_rank):
    """Time pa_prefill on a prefill workload (tensor-core bound)."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = args.workload if args.workload in workloads.PREFILL_WORKLOADS else "prefill_llama7b"
    case = workloads.make_prefill_workload(wl, dtype=args.dtype)

    def t(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    q, kc, vc = t(case.q), t(case.k_cache), t(case.v_cache)
    bt, cl, qs = t(case.block_tables), t(case.context_lens), t(case.query_start)
    out = torch.empty_like(q)
    max_q = int((case.query_start[1:] - case.query_start[:-1]).max())
    stream = torch.cuda.Stream(dev)
    call = lambda: pa.prefill(out, q, kc, vc, bt, cl, qs, case.scale, max_query_len=max_q,
                              stream=stream)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize(dev)
    assert pa.device_errors(stream=stream) == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    flops = workloads.prefill_algorithmic_flops(case)
    tflops = flops / (ms * 1e-3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, src = float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        peak, src = 1900.0, "fallback 1.9 PFLOP/s"
    print(json.dumps({
        "metric": "pa_prefill TFLOP/s", "value": round(tflops, 2), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 4),
        "higher_is_better": True, "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": wl, "num_seqs": case.num_seqs, "num_heads": case.num_heads,
                   "head_dim": case.head_dim, "query_tokens": int(case.query_start[-1]),
                   "context_tokens": int(case.context_lens.sum())},
        "tokens_per_s": round(int(case.query_start[-1]) / (ms * 1e-3), 1),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "peak_source": src,
                     "algorithmic_flops_per_launch": int(flops),
                     "traffic": recorded_prefill_traffic(wl), "traffic_unit": "DRAM bytes per launch",
                     "note": "algorithmic flops: 4*D per causal (query, key) pair per head; "
                             "the kernel issues 1.5x (P V runs for P_hi and P_lo)"},
        "gpu_launches": args.steps}))


def run_shared_prefix_op(args, local_rank):
    """Time pa_decode_shared_prefix (the tensor-core prefix kernel, then the
    suffix decode) against pa_decode on the same batch sharing a 512-token
    prompt (the shared_prefix workload, or shared_prefix_4k with
    --workload), with L2 flushed before every call (so the prefix comes from
    HBM once per call, not from the last call's L2 lines)."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pa.lib()
    wl = args.workload if args.workload in ("shared_prefix", "shared_prefix_4k") else "shared_prefix"
    case = workloads.make_workload(wl, dtype=args.dtype)
    et = torch.bfloat16 if args.dtype == "bf16" else torch.float16

    def t(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    q, kc, vc = t(case.q), t(case.k_cache), t(case.v_cache)
    bt, cl = t(case.block_tables), t(case.context_lens)
    S = case.num_seqs
    gs = torch.tensor([0, S], dtype=torch.int32, device=dev)
    gp = torch.tensor([case.shared_prefix_blocks], dtype=torch.int32, device=dev)
    out_s = torch.empty(case.q.shape, dtype=et, device=dev)
    out_p = torch.empty_like(out_s)
    stream = torch.cuda.Stream(dev)
    dt = 1 if args.dtype == "bf16" else 0
    dims = pa.Dims(S, case.num_heads, case.head_dim, case.block_size, case.num_blocks, dt)
    import ctypes
    l = pa.lib()
    ws = torch.empty(l.pa_decode_shared_prefix_workspace_bytes(ctypes.byref(dims),
                                                               case.max_blocks_per_seq,
                                                               args.partition_tokens),
                     dtype=torch.uint8, device=dev)
    ctr = torch.zeros(l.pa_decode_shared_prefix_counters_bytes(ctypes.byref(dims)) // 4,
                      dtype=torch.int32, device=dev)
    ws_p = torch.empty(max(16, pa.decode_workspace_bytes(S, case.num_heads, case.head_dim,
                                                         case.block_size, case.num_blocks,
                                                         case.max_blocks_per_seq,
                                                         args.partition_tokens, dtype=dt)),
                       dtype=torch.uint8, device=dev)
    ctr_p = torch.zeros(pa.decode_counters_bytes(S, case.num_heads) // 4, dtype=torch.int32,
                        device=dev)
    flush = L2Flush(torch, dev)

    def shared():
        pa.decode_shared_prefix(out_s, q, kc, vc, bt, cl, case.scale, gs, gp, max_group_size=S,
                                partition_tokens=args.partition_tokens, counters=ctr,
                                workspace=ws, stream=stream)

    def plain():
        pa.decode(out_p, q, kc, vc, bt, cl, case.scale, partition_tokens=args.partition_tokens,
                  workspace=ws_p, counters=ctr_p, stream=stream)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for e0, e1 in evs:
            flush(torch, stream)
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    sampler = ClockSampler(local_rank) if not args.no_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_begin = time.time()
    ms_s = timed(shared)
    ms_p = timed(plain)
    t_end = time.time()
    if sampler:
        time.sleep(0.1)
        sampler.stop()
    if pa.device_errors(stream=stream):
        raise RuntimeError("device error during the timed calls")
    # two correct answers (within the decode tolerance of the oracle, which the
    # tests check): here only that they agree with each other
    diff = float((out_s.float() - out_p.float()).abs().max())
    if not diff <= 4e-3:
        raise RuntimeError(f"shared-prefix and plain decode disagree by {diff}")
    shared_ms = sum(ms_s) / len(ms_s)
    plain_ms = sum(ms_p) / len(ms_p)
    uniq = workloads.decode_unique_bytes(case)
    logical = workloads.decode_algorithmic_bytes(case)
    peak, peak_kind = measured_peaks()
    achieved = uniq / (shared_ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "shared-prefix decode GB/s (unique bytes)", "value": round(achieved, 2),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(shared_ms, 4), "higher_is_better": True, "dtype": args.dtype,
        "data": "synthetic",
        "config": {"workload": wl, "num_seqs": S, "num_heads": case.num_heads,
                   "head_dim": case.head_dim, "prefix_blocks": case.shared_prefix_blocks,
                   "total_context_tokens": int(case.context_lens.sum()),
                   "partition_tokens": args.partition_tokens or 512,
                   "l2": "flushed before every call (256 MiB write, then 256 MiB read of another "
                         "buffer, outside the events)"},
        "ms_median": round(statistics.median(ms_s), 4),
        "plain_decode_ms": round(plain_ms, 4),
        "plain_decode_unique_gbs": round(uniq / (plain_ms * 1e-3) / 1e9, 2),
        "speedup_vs_plain": round(plain_ms / shared_ms, 3),
        "logical_gbs": round(logical / (shared_ms * 1e-3) / 1e9, 2),
        "tokens_per_s": round(S / (shared_ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": "prefix kernel + suffix decode (two launches)",
                     "unique_bytes_per_call": int(uniq), "logical_bytes_per_call": int(logical),
                     "traffic": recorded_shared_traffic(wl),
                     "traffic_unit": "DRAM bytes per call (both kernels)"},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(t_begin, t_end) if sampler else None}))


def run_variants_op(args, local_rank):
    """Decode GB/s of every built (dtype, head_dim, block_size) variant on a
    LLaMA-shaped batch with the same bytes per token (64 sequences, contexts
    U[128, 2048], H x D = 4096): decode only, --steps launches between two
    events, against the measured copy rate.  One JSON line."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pa.lib()
    peak, peak_kind = measured_peaks()
    rng = np.random.default_rng(11)
    ctx = rng.integers(128, 2049, size=64)
    steps = max(1, args.steps)
    results = []
    for dt in ("f16", "bf16"):
        for D in (64, 128, 256):
            for B in (8, 16, 32):
                H = 4096 // D
                case = workloads.build_case(f"v{D}_{B}", ctx, num_heads=H, head_dim=D,
                                            block_size=B, seed=31, dtype=dt)

                def t(a):
                    a = np.ascontiguousarray(a)
                    if a.dtype == np.uint16:
                        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
                    return torch.from_numpy(a).to(dev)

                q, kc, vc, bt, cl = map(t, (case.q, case.k_cache, case.v_cache, case.block_tables,
                                            case.context_lens))
                out = torch.empty_like(q)
                stream = torch.cuda.Stream(dev)
                for _ in range(max(3, args.warmup)):
                    pa.decode(out, q, kc, vc, bt, cl, case.scale, stream=stream)
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(steps):
                    pa.decode(out, q, kc, vc, bt, cl, case.scale, stream=stream)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                if pa.device_errors(stream=stream):
                    raise RuntimeError(f"device error in variant {dt} {D}x{B}")
                us = e0.elapsed_time(e1) / steps * 1e3
                gbs = workloads.decode_algorithmic_bytes(case) / us / 1e3
                results.append({"dtype": dt, "head_dim": D, "block_size": B, "num_heads": H,
                                "decode_us": round(us, 2), "GB/s": round(gbs, 1),
                                "frac": round(gbs / peak, 4)})
                del q, kc, vc, bt, cl, out, case
                torch.cuda.empty_cache()
    print(json.dumps({"metric": "pa_decode GB/s per variant", "unit": "GB/s",
                      "steps": steps, "warmup": max(3, args.warmup), "data": "synthetic",
                      "config": {"num_seqs": 64, "context": "U[128, 2048]", "heads_x_dim": 4096,
                                 "launches": "decode only, between two events"},
                      "peak": peak, "peak_source": peak_kind, "variants": results}))


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.op == "prefill":
        if rank == 0:
            run_prefill_op(args, local_rank)
        return
    if args.op == "shared_prefix":
        if rank == 0:
            run_shared_prefix_op(args, local_rank)
        return
    if args.op == "variants":
        if rank == 0:
            run_variants_op(args, local_rank)
        return
    if args.op != "step":
        if rank == 0:
            run_copy_op(args, local_rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_native(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
