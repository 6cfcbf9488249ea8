"""Benchmark of the DSA indexer fused Q/K prepare-and-store on GB300.

One step = one fused call over the prefill workload (T = 8192 tokens of one
sequence, H = 64 indexer heads, D = 128, rope_dim = 64 NeoX, slots contiguous
in 128 pages of 64): the whole hot path (RoPE on q and k, LayerNorm on k,
e4m3 + ue8m0 quantisation, gate-weight fold, index-K cache store) in one
kernel launch.  Prints ONE JSON line (rank 0):

  value      tokens/s over all ranks, inputs resident in HBM (two alternating
             input sets of 2 x 210 MB, so no step reads the previous one's data
             from the 129 MB L2)
  e2e        the same through the public Python API with pinned host buffers:
             host->device copy of q, k|w, positions and slots, the call, and
             device->host copy of (q_fp8, weights), all inside the timed region;
             steps alternate between two streams so one step's device->host
             copy overlaps the next one's host->device copy (the one-stream
             figure is reported beside it)
  roofline   algorithmic bytes per launch / launch time vs the measured HBM
             copy bandwidth; traffic = DRAM bytes per launch from the committed
             ncu summary when it was taken on the current kernel source
  decode     us per call at the decode shapes (T = 64, H = 64, GPT-J; and
             T in {1, 8, 32, 64, 256}, H = 32, NeoX): one decode step of 21
             indexer layers (shared positions / slots / rope cache, per-layer
             q, k|w, outputs and index-K cache) captured as a CUDA graph and
             replayed after an L2 flush -- plain, with PDL, and with PDL plus
             early rope reads -- plus a single-call graph, eager calls through
             the binding, and eager calls through the C ABI with pre-bound
             arguments (eager_abi_us, with their host time host_abi_us)
  prefill_few_heads  prefill (T = 8192) with H = 32 and H = 16 heads
  hadamard   the Hadamard-rotated variant (q and k times H_128 / sqrt(128)
             after RoPE) on the prefill inputs and in the decode step
  unfused    the same call as four launches with bf16 intermediates (the
             pages' pre-fusion chain) on the prefill inputs and in the decode
             step, for the 4 -> 1 launch comparison
  stress     the heavy-tailed 65,536-token workload (1.7 GB per call) in
             both pairings: us/call and HBM GB/s
  k_only     the k-only call (index-K store) on 65,536 heavy-tailed keys in
             both pairings, cycling input sets larger than L2
  mqa_logits the indexer's fp8 paged MQA logits (the consumer of the index-K
             cache) on the tcgen05 tensor cores at the 16K-context decode step
  cpu_baseline  the oracle (plain C) on a bounded sample, one spawned process
             per host core over disjoint token ranges; the one-core figure
             sits inside it, and so do one-core us/call figures for the
             tiny, decode and sweep workloads

``--impl reference`` times the oracle instead (the CPU statement of the path),
on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s + achieved HBM GB/s (% of peak) prefill; µs/call at decode T=1..64"
WORKLOAD = "prefill T=8192 H=64 D=128 rope_dim=64 NeoX, 128 pages x 64 (contiguous slots)"
# DRAM traffic of the kernels, per launch, from ncu (written by --traffic-from)
TRAFFIC_JSON = {"prefill": os.path.join(ROOT, "profiles", "traffic_prefill_T8192_H64.json"),
                "decode": os.path.join(ROOT, "profiles", "traffic_decode_T64_H64.json"),
                "k_only": os.path.join(ROOT, "profiles", "traffic_k_only_T65536.json")}
TRAFFIC_KERNEL = {"prefill": "dsa_pipeline_kernel", "decode": "dsa_direct_kernel",
                  "k_only": "dsa_kstream_kernel"}
# The decode probe repeats one small input set, which stays in L2 between
# launches; its capture flushes the caches before each launch instead, so
# the inputs come from DRAM (and the outputs stay in L2 within the window).
TRAFFIC_CACHE = {"prefill": "none", "decode": "all", "k_only": "none"}
TRAFFIC_METRICS = ("dram__bytes_read.sum,dram__bytes_write.sum,lts__t_sectors_op_write.sum,"
                   "lts__t_sectors_op_read.sum,gpu__time_duration.sum")
KERNEL_SRCS = [os.path.join(ROOT, "prep_token_gb300", "csrc", f)
               for f in ("dsa_prep.cu", "dsa_prep_kernels.cuh", "dsa_common.cuh")]
L2_FLUSH_BYTES = 256 << 20
GRAPH_STEPS = 50


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def max_over_ranks(value: float, device="cpu") -> float:
    """The largest `value` over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_source_hash(files=None):
    """sha256 over the sources a kernel is compiled from (the prefill kernel's
    by default), with comments and whitespace removed, so that a comment edit
    does not orphan the committed profile."""
    h = hashlib.sha256()
    for f in files or KERNEL_SRCS:
        src = open(f).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()


def profile_traffic(which="prefill"):
    """DRAM bytes per launch (read + write) from the committed traffic summary
    of that kernel, or None when its sources have changed since the capture."""
    path = TRAFFIC_JSON[which]
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return float(rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"])


def write_traffic_json(csv_path, which):
    """Turn an ncu --csv launch list of the TRAFFIC_METRICS (two back-to-back
    launches of one kernel) into the committed summary: the figures of the
    last launch.  With --cache-control none (prefill, k-only: inputs larger
    than L2) that launch also drains what the one before left dirty in L2,
    so its DRAM writes are those of a launch in a stream; the decode capture
    flushes the caches before each launch (TRAFFIC_CACHE)."""
    import csv
    launches = {}
    name = None
    with open(csv_path) as f:
        rows = list(csv.reader(f))
    hdr = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    cols = rows[hdr]
    for r in rows[hdr + 1:]:
        if len(r) != len(cols):
            continue
        d = dict(zip(cols, r))
        name = d["Kernel Name"]
        launches.setdefault(int(d["ID"]), {})[d["Metric Name"]] = float(d["Metric Value"].replace(",", ""))
    last = launches[max(launches)]
    probe = {"prefill": "prefill", "decode": "decode", "k_only": "k_only"}[which]
    rec = {
        "kernel": name,
        "workload": {"prefill": "prefill T=8192 H=64 NeoX (synth.make_prefill(seed=3))",
                     "decode": "decode T=64 H=64 GPT-J (synth.make_decode(seed=1))",
                     "k_only": "k-only T=65536 (synth.make_k_bulk, four input sets cycled)"}[which],
        "command": (f"ncu --metrics {TRAFFIC_METRICS} --cache-control {TRAFFIC_CACHE[which]} "
                    f"--clock-control none "
                    f"-k regex:{TRAFFIC_KERNEL[which]} -s 2 -c 2 --csv --log-file traffic.csv "
                    f"python bench.py --probe {probe}"),
        "launches_captured": len(launches),
        "dram_bytes_read_per_launch": last["dram__bytes_read.sum"],
        "dram_bytes_write_per_launch": last["dram__bytes_write.sum"],
        "lts_read_sector_bytes": last["lts__t_sectors_op_read.sum"] * 32,
        "lts_write_sector_bytes": last["lts__t_sectors_op_write.sum"] * 32,
        "duration_ns_under_ncu": last["gpu__time_duration.sum"],
        "kernel_source_sha256": kernel_source_hash(),
    }
    with open(TRAFFIC_JSON[which], "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling around a timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.out):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.out):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.out)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        num = lambda v: float(v) if re.match(r"^[0-9.]+$", v) else None
        sm = [num(r[1]) for r in rows]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows]
        pmax = max([p for p in pw if p is not None], default=None)
        # "under load": samples drawing at least half the peak power seen
        loaded = [s for s, p in zip(sm, pw)
                  if s is not None and p is not None and pmax and p >= 0.5 * pmax]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": pmax, "samples": len(rows), "samples_under_load": len(loaded),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- our arm

def _dev_inputs(inp, dev):
    import torch

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    kw = bf16(inp.kw)
    d = dict(q=bf16(inp.q), kw=kw, k=kw[:, :128], w=kw[:, 128:128 + inp.H])
    for n, key in (("positions", "positions"), ("slots", "slots"), ("cos", "cos"),
                   ("sin", "sin"), ("gamma", "gamma"), ("beta", "beta")):
        d[key] = torch.from_numpy(getattr(inp, n)).to(dev)
    d["cache"] = torch.zeros(inp.cache_bytes, dtype=torch.uint8, device=dev)
    d["q_out"] = torch.empty((inp.T, inp.H, 128), dtype=torch.float8_e4m3fn, device=dev)
    d["w_out"] = torch.empty((inp.T, inp.H), dtype=torch.float32, device=dev)
    return d


def _add_workspace(dp, torch, inp, d, dev):
    d["ws"] = torch.empty(dp.dsa_unfused_workspace_bytes(inp.T, inp.H), dtype=torch.uint8,
                          device=dev)


def _call(dp, inp, d, stream, T=None, k_only=False, pdl=False, unfused=False, hadamard=False):
    if unfused:
        dp.dsa_indexer_qk_prepare_store_unfused(
            d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
            d["beta"], inp.eps, inp.softmax_scale, d["cache"], inp.page_size, inp.rope_dim,
            inp.style, q_fp8_out=d["q_out"], weights_out=d["w_out"], workspace=d["ws"],
            max_position=inp.max_position, stream=stream, num_tokens=T, pdl=bool(pdl))
        return
    if k_only:
        dp.dsa_indexer_k_prepare_store(
            d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"],
            inp.eps, d["cache"], inp.page_size, inp.rope_dim, inp.style,
            max_position=inp.max_position, stream=stream, num_tokens=T, pdl=pdl,
            hadamard=hadamard)
        return
    dp.dsa_indexer_qk_prepare_store(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, d["cache"], inp.page_size, inp.rope_dim,
        inp.style, q_fp8_out=d["q_out"], weights_out=d["w_out"],
        max_position=inp.max_position, stream=stream, num_tokens=T, pdl=pdl, hadamard=hadamard)


def _prepared(dp, inp, d, stream, k_only=False, hadamard=False):
    """The decode call checked and bound once (dp.PreparedCall): each call is
    then one ctypes call into the C ABI with pre-built arguments."""
    if k_only:
        return dp.prepare_k_prepare_store(
            d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"],
            inp.eps, d["cache"], inp.page_size, inp.rope_dim, inp.style,
            max_position=inp.max_position, stream=stream, hadamard=hadamard)
    return dp.prepare_qk_prepare_store(
        d["q"], d["k"], d["w"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"],
        d["beta"], inp.eps, inp.softmax_scale, d["cache"], inp.page_size, inp.rope_dim,
        inp.style, q_fp8_out=d["q_out"], weights_out=d["w_out"],
        max_position=inp.max_position, stream=stream, hadamard=hadamard)


def _prefill_graph_us(torch, sets, stream, call, steps):
    """us per call of `call(inp, d)` on the alternating prefill sets: a graph
    of 10 calls replayed up to 100 times (after 3 eager warm-up calls)."""
    with torch.cuda.stream(stream):
        for i in range(3):
            call(*sets[i & 1])
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(10):
            call(*sets[i & 1])
    reps = max(1, min(100, steps // 10))
    with torch.cuda.stream(stream):
        g.replay()
        u0 = torch.cuda.Event(enable_timing=True)
        u1 = torch.cuda.Event(enable_timing=True)
        u0.record(stream)
        for _ in range(reps):
            g.replay()
        u1.record(stream)
    stream.synchronize()
    del g
    return u0.elapsed_time(u1) * 1000.0 / (10 * reps), 10 * reps


def _decode_timings(dp, torch, dev, make, reps=30, layers=21, k_only_too=False,
                    unfused_too=False, hadamard=False):
    """us per call for one decode step of `layers` indexer layers: the layers
    share the step's positions, slots and rope cache (as in a model) and each
    has its own q, k|w, outputs and index-K cache.  Timed as a graph of the
    `layers` sequential calls replayed `reps` times with an L2 flush before
    each replay (only the replay is timed) -- plain, with programmatic
    dependent launch, and with PDL plus early reads of positions / cos / sin --
    and as a single-call graph and back-to-back eager calls."""
    base = make(0)
    shared = None
    sets = []
    for i in range(layers):
        inp = base if i == 0 else make(i)
        d = _dev_inputs(inp, dev)
        if shared is None:
            shared = {k: d[k] for k in ("positions", "slots", "cos", "sin")}
        d.update(shared)
        inp.positions, inp.slots, inp.cos, inp.sin = base.positions, base.slots, base.cos, base.sin
        inp.max_position = base.max_position
        sets.append((inp, d))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    out = {"T": base.T, "H": base.H, "style": "gptj" if base.style else "neox"}
    modes = [("qk", False, False)] + ([("k_only", True, False)] if k_only_too else []) + \
        ([("unfused_qk", False, True)] if unfused_too else [])
    if unfused_too:
        for inp, d in sets:
            _add_workspace(dp, torch, inp, d, dev)
    for name, k_only, unfused in modes:
        with torch.cuda.stream(stream):
            for inp, d in sets:          # warm-up outside capture
                _call(dp, inp, d, stream, k_only=k_only, unfused=unfused, hadamard=hadamard)
        stream.synchronize()
        res = {"launches_per_call": 4 if unfused else 1}
        variants = ((layers, False, f"graph{layers}_us"), (layers, True, f"graph{layers}_pdl_us"))
        if not unfused:
            variants += ((layers, "early", f"graph{layers}_pdl_early_us"), (1, False, "graph1_us"))
        for n_layers, pdl, key in variants:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for inp, d in sets[:n_layers]:
                    _call(dp, inp, d, stream, k_only=k_only, pdl=pdl, unfused=unfused,
                          hadamard=hadamard)
            times = []
            for _ in range(reps):
                with torch.cuda.stream(stream):
                    flush.fill_(1)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                stream.synchronize()
                times.append(e0.elapsed_time(e1) * 1000.0 / n_layers)
            res[key] = {"median": statistics.median(times), "best": min(times)}
            del g
        # eager: back-to-back calls through the Python binding
        times = []
        with torch.cuda.stream(stream):
            for _ in range(5):
                flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for inp, d in sets:
                    _call(dp, inp, d, stream, k_only=k_only, unfused=unfused, hadamard=hadamard)
                e1.record(stream)
                stream.synchronize()
                times.append(e0.elapsed_time(e1) * 1000.0 / len(sets))
        res["eager_us"] = {"median": statistics.median(times), "best": min(times)}
        if not unfused:
            # eager through the C ABI with pre-bound arguments (no binding checks):
            # device time per call and host time per call
            calls = [_prepared(dp, inp, d, stream, k_only=k_only, hadamard=hadamard)
                     for inp, d in sets]
            times, host = [], []
            with torch.cuda.stream(stream):
                for _ in range(5):
                    flush.fill_(1)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    h0 = time.perf_counter()
                    for c in calls:
                        c()
                    host.append((time.perf_counter() - h0) * 1e6 / len(calls))
                    e1.record(stream)
                    stream.synchronize()
                    times.append(e0.elapsed_time(e1) * 1000.0 / len(calls))
            res["eager_abi_us"] = {"median": statistics.median(times), "best": min(times)}
            res["host_abi_us"] = {"median": statistics.median(host), "best": min(host)}
        out[name] = res
    return out


def _k_dev_inputs(inp, dev):
    """Device buffers of a k-only call: the k|w rows, indices, rope table,
    LayerNorm parameters and a zeroed index-K cache."""
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    kw = t(inp.kw.view(np.int16)).view(torch.bfloat16)
    return dict(k=kw[:, :128], positions=t(inp.positions), slots=t(inp.slots), cos=t(inp.cos),
                sin=t(inp.sin), gamma=t(inp.gamma), beta=t(inp.beta),
                cache=torch.zeros(inp.cache_bytes, dtype=torch.uint8, device=dev))


def _k_bulk_timing(dp, torch, dev, peaks, reps=20, n_sets=4):
    """The k-only call at prefill size (65,536 keys, 8 sequences of 8192),
    both pairings: us per call over a graph of 8 calls that cycles through
    `n_sets` input sets (k|w rows, slots and caches; 4 x 43 MB, more than the
    129 MB L2), so every call reads its keys from HBM.  Plain launches, PDL
    launches, and PDL with the positions and cos/sin read before the wait
    (pdl="early": the k rows come from the previous kernel, the rest not)."""
    import synth
    out = {}
    kbytes = None
    for style, name in ((synth.NEOX, "neox"), (synth.GPTJ, "gptj")):
        sets = []
        for i in range(n_sets):
            inp = synth.make_k_bulk(seed=6 + i, style=style)
            sets.append((inp, _k_dev_inputs(inp, dev)))
        stream = torch.cuda.Stream(device=dev)
        T = sets[0][0].T
        kbytes = synth.algorithmic_bytes(T, 0, with_q=False)

        def call(inp, d, pdl):
            dp.dsa_indexer_k_prepare_store(
                d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"],
                inp.eps, d["cache"], inp.page_size, inp.rope_dim, inp.style,
                max_position=inp.max_position, pdl=pdl, stream=stream)

        def timed(pdl, rounds=3):
            """median (and best) over `rounds` timings of `reps` graph replays"""
            with torch.cuda.stream(stream):
                for inp, d in sets:
                    call(inp, d, pdl)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(8):
                    call(*sets[i % n_sets], pdl)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
            times = []
            for _ in range(rounds):
                with torch.cuda.stream(stream):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(reps):
                        g.replay()
                    e1.record(stream)
                stream.synchronize()
                times.append(e0.elapsed_time(e1) * 1000.0 / (8 * reps))
            del g
            us = statistics.median(times)
            gbs = kbytes / (us * 1e-6) / 1e9
            return {"us_per_call": us, "us_best": min(times), "calls": 8 * reps * rounds,
                    "gb_per_s": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
                    "keys_per_s": T / (us * 1e-6)}

        out[name] = timed(False)
        out[name]["pdl"] = timed(True)
        out[name]["pdl_early"] = timed("early")
        out["workload"] = (f"k-only T={T} (8 x 8192 tokens) rope_dim=64, 2048 shuffled pages, "
                           f"{n_sets} input sets cycled (larger than L2)")
        del sets
    out["algorithmic_bytes"] = kbytes
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import prep_token_gb300 as dp
    import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dp.library()
    peaks, peak_kind = measured_peaks()

    # two input sets, alternated, so consecutive steps never share L2 lines
    sets = []
    for i in range(2):
        inp = synth.make_prefill(seed=3 + 1000 * rank + i)
        sets.append((inp, _dev_inputs(inp, dev)))
    T, H = sets[0][0].T, sets[0][0].H
    algo_bytes = synth.algorithmic_bytes(T, H)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        inp, d = sets[i & 1]
        _call(dp, inp, d, stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    # The K timed steps are replayed from CUDA graphs (GRAPH_STEPS launches per
    # graph, plus one graph for the remainder) so the host's per-call Python
    # cost never gaps the device; every step is still one full launch.
    per_graph = min(GRAPH_STEPS, args.steps)
    n_rep, rem = divmod(args.steps, per_graph)
    graphs = []
    for n, reps in ((per_graph, n_rep), (rem, 1)):
        if n and reps:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    step(i)
            graphs.append((g, reps))
    with torch.cuda.stream(stream):
        for g, _ in graphs:
            g.replay()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for g, reps in graphs:
                for _ in range(reps):
                    g.replay()
            e1.record(stream)
        stream.synchronize()
    del graphs
    torch.cuda.synchronize(dev)
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    if world > 1:
        torch.distributed.barrier()
    ms_per_step = elapsed_ms / args.steps
    value = world * T * args.steps / (elapsed_ms / 1000.0)
    launch_us = ms_per_step * 1000.0
    achieved = algo_bytes / (launch_us * 1e-6) / 1e9

    # end to end through the public API, host buffers, copies inside the region.
    # Steps alternate between two streams, each with its own device buffers
    # and pinned host outputs, so one step's device->host copy overlaps the
    # next step's host->device copy (the two directions of the host link).
    inp0 = sets[0][0]
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_q = pin(inp0.q.view(np.int16)).view(torch.bfloat16)
    h_kw = pin(inp0.kw.view(np.int16)).view(torch.bfloat16)
    h_pos, h_slots = pin(inp0.positions), pin(inp0.slots)
    h_out = [(torch.empty((T, H, 128), dtype=torch.uint8).pin_memory(),
              torch.empty((T, H), dtype=torch.float32).pin_memory()) for _ in range(2)]
    lanes = [(torch.cuda.Stream(device=dev), sets[j][1], h_out[j]) for j in range(2)]
    e2e_steps = max(4, min(50, args.steps))

    def e2e_step(i, lane=None):
        s, d, (h_qo, h_wo) = lanes[i & 1] if lane is None else lanes[lane]
        with torch.cuda.stream(s):
            d["q"].copy_(h_q, non_blocking=True)
            d["kw"].copy_(h_kw, non_blocking=True)
            d["positions"].copy_(h_pos, non_blocking=True)
            d["slots"].copy_(h_slots, non_blocking=True)
            _call(dp, inp0, d, s)
            h_qo.copy_(d["q_out"].view(torch.uint8), non_blocking=True)
            h_wo.copy_(d["w_out"], non_blocking=True)

    def e2e_region(serial):
        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        s0 = lanes[0][0]
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(s0)
        lanes[1][0].wait_event(f0)
        for i in range(e2e_steps):
            e2e_step(i, 0 if serial else None)
        done = torch.cuda.Event()
        done.record(lanes[1][0])
        s0.wait_event(done)
        f1.record(s0)
        torch.cuda.synchronize(dev)
        return max_over_ranks(f0.elapsed_time(f1), dev)

    e2e_serial_ms = e2e_region(serial=True)
    e2e_ms = e2e_region(serial=False)
    h2d = h_q.numel() * 2 + h_kw.numel() * 2 + h_pos.numel() * 8 + h_slots.numel() * 8
    d2h = h_out[0][0].numel() + h_out[0][1].numel() * 4

    # the unfused four-launch chain on the same prefill inputs (baseline)
    unfused = None
    if not args.no_unfused:
        for inp, d in sets:
            _add_workspace(dp, torch, inp, d, dev)
        uus, ucalls = _prefill_graph_us(
            torch, sets, stream, lambda inp, d: _call(dp, inp, d, stream, unfused=True),
            args.steps)
        for _, d in sets:
            del d["ws"]
        unfused = {"prefill_us": uus, "launches_per_call": 4, "calls": ucalls,
                   "fused_speedup": uus / launch_us,
                   "hbm_bytes_per_call": synth.algorithmic_bytes(T, H)
                   + T * (H + 1) * 128 * 2 * 2 + T * 128 * 2 * 2}

    # the same launches under programmatic dependent launch: a launch's CTAs
    # start on SMs the previous one has left and wait there for it to finish
    pdl_us, pdl_calls = _prefill_graph_us(
        torch, sets, stream, lambda inp, d: _call(dp, inp, d, stream, pdl=True), args.steps)
    prefill_pdl = {"us_per_call": pdl_us, "calls": pdl_calls,
                   "gb_per_s": algo_bytes / (pdl_us * 1e-6) / 1e9,
                   "hbm_frac": algo_bytes / (pdl_us * 1e-6) / 1e9 / peaks["hbm_gbs"]}

    # prefill with fewer heads (units of 64 / H tokens): T = 8192, H = 32 and 16
    few_heads = {}
    for Hf in (32, 16):
        fsets = []
        for i in range(2):
            finp = synth.make_prefill(seed=3 + Hf + 1000 * rank + i, H=Hf)
            fsets.append((finp, _dev_inputs(finp, dev)))
        fus, fcalls = _prefill_graph_us(
            torch, fsets, stream, lambda inp, d: _call(dp, inp, d, stream), args.steps)
        fbytes = synth.algorithmic_bytes(T, Hf)
        fgb = fbytes / (fus * 1e-6) / 1e9
        few_heads[f"prefill_T{T}_H{Hf}"] = {
            "us_per_call": fus, "calls": fcalls, "gb_per_s": fgb, "hbm_frac": fgb / peaks["hbm_gbs"],
            "tokens_per_s": T / (fus * 1e-6), "algorithmic_bytes": fbytes}
        del fsets

    # the Hadamard-rotated variant: same bytes, more arithmetic per vector
    hadamard = None
    if not args.no_hadamard:
        hus, hcalls = _prefill_graph_us(
            torch, sets, stream, lambda inp, d: _call(dp, inp, d, stream, hadamard=True),
            args.steps)
        hgb = algo_bytes / (hus * 1e-6) / 1e9
        hadamard = {"prefill_us": hus, "calls": hcalls, "gb_per_s": hgb,
                    "hbm_frac": hgb / peaks["hbm_gbs"], "tokens_per_s": T / (hus * 1e-6),
                    "vs_plain": hus / launch_us, "launches_per_call": 1}
        if rank == 0 and not args.no_decode:
            hadamard["c2_decode_T64_H64_gptj"] = _decode_timings(
                dp, torch, dev, lambda i: synth.make_decode(seed=1 + 100 * i), hadamard=True)

    # the heavy-tailed stress workload at full size: 8 sequences x 8192 tokens,
    # 1.7 GB per call (far larger than L2), in both pairings
    stress = None
    if not args.no_stress:
        sinp = synth.make_stress(seed=4 + 1000 * rank)
        sd = _dev_inputs(sinp, dev)
        sbytes = synth.algorithmic_bytes(sinp.T, sinp.H)
        stress = {"workload": f"T={sinp.T} H={sinp.H} (8 x 8192 tokens) rope_dim=64, "
                              f"2048 shuffled pages", "algorithmic_bytes": sbytes}
        for style, name in ((synth.NEOX, "neox"), (synth.GPTJ, "gptj")):
            sinp.style = style
            us, calls = _prefill_graph_us(torch, [(sinp, sd), (sinp, sd)], stream,
                                          lambda inp, d: _call(dp, inp, d, stream),
                                          min(args.steps, 200))
            gbs = sbytes / (us * 1e-6) / 1e9
            stress[name] = {"us_per_call": us, "calls": calls, "gb_per_s": gbs,
                            "hbm_frac": gbs / peaks["hbm_gbs"],
                            "tokens_per_s": sinp.T / (us * 1e-6)}
        # the k-only call at the same size: its own section, on input sets larger than L2
        del sd

    k_only = None
    if not args.no_stress:
        k_only = _k_bulk_timing(dp, torch, dev, peaks)

    logits = None
    if rank == 0 and not args.no_logits:
        logits = _logits_timing(dp, torch, dev, peaks)

    decode = None
    if rank == 0 and not args.no_decode:
        decode = {"c2_decode_T64_H64_gptj": _decode_timings(
            dp, torch, dev, lambda i: synth.make_decode(seed=1 + 100 * i), k_only_too=True,
            unfused_too=True)}
        for Tn in (1, 8, 32, 64, 256):
            decode[f"sweep_T{Tn}_H32"] = _decode_timings(
                dp, torch, dev, lambda i, Tn=Tn: synth.make_sweep(Tn, seed=2 + 100 * i))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(sets[0][0], budget_s=args.cpu_seconds)
        cpu = cpu_baseline_parallel(sets[0][0], cpu, budget_s=args.cpu_seconds)
        cpu["other_workloads"] = cpu_baseline_configs()

    if rank != 0:
        return None
    return {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "io_dtype": "bf16 in; e4m3 codes + fp32 ue8m0 scales + fp32 weights out",
        "data": "synthetic (seeded N(0,1) bf16, positions 0..8191, contiguous slots)",
        "config": {"workload": WORKLOAD, "T": T, "H": H, "head_dim": 128, "rope_dim": 64,
                   "rope_style": "neox", "page_size": 64, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: two alternating input sets of "
                         f"{algo_bytes / 1e6:.0f} MB per call"},
        "gb_per_s": achieved,
        "hbm_frac": achieved / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_kind": f"{peak_kind} (torch bf16 copy, read+write)",
                     "algorithmic_bytes_per_launch": algo_bytes,
                     "launch_us": launch_us,
                     "traffic": profile_traffic(),
                     "nominal_frac_8tbs": achieved / 8000.0},
        "e2e": {"value": world * T * e2e_steps / (e2e_ms / 1000.0), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
                "streams": 2, "serial_ms_per_step": e2e_serial_ms / e2e_steps,
                "host_link_gb_per_s": (h2d + d2h) / (e2e_ms / e2e_steps) / 1e6},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
        "decode": decode,
        "unfused": unfused,
        "hadamard": hadamard,
        "prefill_pdl": prefill_pdl,
        "prefill_few_heads": few_heads,
        "stress": stress,
        "k_only": k_only,
        "mqa_logits": logits,
        "cpu_baseline": cpu,
    }


# ----------------------------------------------------------------- oracle

def _oracle_call(inp, lo, hi, cache, q_fp8, weights):
    import oracle
    kw = inp.kw[lo:hi]
    return oracle.qk_prepare_store(
        np.ascontiguousarray(inp.q[lo:hi]).reshape(-1), inp.q_stride_t, inp.q_stride_h,
        np.ascontiguousarray(kw).reshape(-1), inp.k_stride_t,
        np.ascontiguousarray(kw).reshape(-1)[128:], inp.w_stride_t,
        np.ascontiguousarray(inp.positions[lo:hi]), np.ascontiguousarray(inp.slots[lo:hi]),
        inp.cos, inp.sin, inp.cs_stride, inp.max_position, inp.gamma, inp.beta, inp.eps,
        inp.softmax_scale, q_fp8, weights, cache, inp.num_pages, inp.page_size, inp.H,
        inp.rope_dim, inp.style)


_WORKER = {}


def _pool_init(seed, barrier):
    """Spawned oracle worker: build the seeded prefill inputs once, then wait
    until every worker is ready."""
    import oracle
    import synth
    oracle.build()
    inp = synth.make_prefill(seed=seed)
    _WORKER["inp"] = inp
    _WORKER["cache"] = np.zeros(inp.cache_bytes, np.uint8)
    barrier.wait()


def _pool_job(job):
    """The oracle over tokens [lo, hi) of the worker's prefill inputs, `reps`
    times.  Returns (tokens, seconds)."""
    lo, hi, reps = job
    inp = _WORKER["inp"]
    q_fp8 = np.zeros((hi - lo, inp.H, 128), np.uint8)
    weights = np.zeros((hi - lo, inp.H), np.float32)
    t0 = time.perf_counter()
    for _ in range(reps):
        _oracle_call(inp, lo, hi, _WORKER["cache"], q_fp8, weights)
    return (hi - lo) * reps, time.perf_counter() - t0


class OraclePool:
    """One spawned process per host core this process may use, each holding
    the seeded prefill inputs.  The oracle is single-threaded, so the cores
    split the tokens: run() hands every worker its own contiguous range."""

    def __init__(self, seed=3):
        import multiprocessing as mp
        import oracle
        oracle.build()
        self.cores = len(os.sched_getaffinity(0))
        ctx = mp.get_context("spawn")
        barrier = ctx.Barrier(self.cores + 1)
        self.pool = ctx.Pool(self.cores, initializer=_pool_init, initargs=(seed, barrier))
        barrier.wait(timeout=900)

    def run(self, first, span, T, reps=1):
        """Worker c takes tokens [first + c*span, +span) mod T; returns
        (tokens, wall seconds)."""
        jobs = []
        for c in range(self.cores):
            lo = (first + c * span) % T
            jobs.append((lo, min(T, lo + span), reps))
        t0 = time.perf_counter()
        res = self.pool.map(_pool_job, jobs, chunksize=1)
        return sum(r[0] for r in res), time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline_configs(budget_s=0.5):
    """The oracle on one host core for each of the other workloads (tiny,
    the decode step, the decode sweep): us per call, each timed over about
    `budget_s` of repeated calls."""
    import synth
    import oracle
    oracle.build()
    cases = [("tiny_T4_H8", synth.make_tiny(seed=0, fused_kw=True)),
             ("c2_decode_T64_H64_gptj", synth.make_decode(seed=1))]
    cases += [(f"sweep_T{n}_H32", synth.make_sweep(n, seed=2)) for n in (1, 8, 32, 64, 256)]
    out = {}
    for name, inp in cases:
        cache = np.zeros(inp.cache_bytes, np.uint8)
        q_fp8 = np.zeros((inp.T, inp.H, 128), np.uint8)
        weights = np.zeros((inp.T, inp.H), np.float32)
        calls, t0 = 0, time.perf_counter()
        while calls == 0 or time.perf_counter() - t0 < budget_s:
            _oracle_call(inp, 0, inp.T, cache, q_fp8, weights)
            calls += 1
        us = (time.perf_counter() - t0) / calls * 1e6
        out[name] = {"us_per_call": us, "tokens_per_s": inp.T / (us * 1e-6), "calls": calls,
                     "cores": 1}
    return out


def cpu_baseline_parallel(inp, single, budget_s=10.0):
    """The same oracle on every host core (OraclePool), over the prefill
    tokens; pool start-up is outside the timed region."""
    pool = OraclePool(seed=3)
    try:
        per_core = max(1, int(single["value"] * budget_s / 2))
        span = max(1, min(inp.T // pool.cores, per_core))
        reps = max(1, per_core // span)
        toks, dt = pool.run(0, span, inp.T, reps)
    finally:
        pool.close()
    return {"value": toks / dt, "unit": "tokens/s", "cores": pool.cores, "kind": "oracle",
            "sample": f"{toks} tokens of the prefill workload ({pool.cores} spawned processes, "
                      f"{span} consecutive tokens x {reps} each), {dt:.1f} s wall",
            "single_core": single}


def cpu_baseline(inp, budget_s=10.0):
    """The oracle, as it stands, on one host core, over consecutive chunks of
    the prefill workload until `budget_s` of CPU time has been spent."""
    import oracle
    oracle.build()
    chunk = 256
    cache = np.zeros(inp.cache_bytes, np.uint8)
    q_fp8 = np.zeros((chunk, inp.H, 128), np.uint8)
    weights = np.zeros((chunk, inp.H), np.float32)
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        lo = done % inp.T
        hi = min(inp.T, lo + chunk)
        _oracle_call(inp, lo, hi, cache, q_fp8, weights)
        done += hi - lo
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} tokens of the prefill workload (chunks of {chunk}), "
                      f"{dt:.1f} s on one host core"}


def run_reference(args, rank, world):
    """The oracle as it stands, timed on every host core (OraclePool): each
    step is one bounded sample of the prefill workload, split over the cores."""
    if rank != 0:
        return None
    import synth
    import oracle
    oracle.build()
    inp = synth.make_prefill(seed=3)
    cache = np.zeros(inp.cache_bytes, np.uint8)
    # calibrate on one core, then size each step's sample so the run stays ~2 minutes
    q_fp8 = np.zeros((32, inp.H, 128), np.uint8)
    weights = np.zeros((32, inp.H), np.float32)
    t0 = time.perf_counter()
    _oracle_call(inp, 0, 32, cache, q_fp8, weights)
    per_tok = (time.perf_counter() - t0) / 32
    pool = OraclePool(seed=3)
    try:
        total_steps = args.steps + args.warmup
        # at least 16 tokens per core per step, so the pool's messaging stays
        # small next to the oracle's own work
        span = int(max(16, min(inp.T // pool.cores, 100.0 / max(total_steps, 1) / per_tok)))
        for i in range(args.warmup):
            pool.run(i * span * pool.cores, span, inp.T)
        toks, dt = 0, 0.0
        for i in range(args.steps):
            n, s = pool.run((args.warmup + i) * span * pool.cores, span, inp.T)
            toks += n
            dt += s
    finally:
        pool.close()
    value = toks / dt
    sample = (f"{span * pool.cores} tokens of the prefill workload per step "
              f"({span} consecutive tokens on each of {pool.cores} spawned processes)")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1000 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "T": inp.T, "H": inp.H},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": pool.cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def _logits_inputs(torch, dev, synth, T=64, H=64, context=16384):
    li = synth.make_logits(seed=5, T=T, H=H, context=context)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return li, dict(q=d(li.q_fp8), w=d(li.weights), cache=d(li.cache), bt=d(li.block_table),
                    lens=d(li.context_lens),
                    out=torch.empty((T, li.max_context), dtype=torch.float32, device=dev))


def _logits_call(dp, li, t, stream, pdl=False):
    dp.dsa_indexer_mqa_logits(t["q"], t["w"], t["cache"], li.page_size, t["bt"], t["lens"],
                              li.max_context, logits=t["out"], stream=stream, pdl=pdl)


def _logits_timing(dp, torch, dev, peaks, calls=10, reps=20):
    """The indexer's fp8 paged MQA logits on the tensor cores, at the decode
    step of the pages' serving bench (64 sequences, 16K context, 64 heads):
    us per call, HBM GB/s and fp8 tensor TFLOP/s.  The 138 MB index-K cache is
    larger than L2, so consecutive calls re-read it from HBM."""
    import synth
    li, t = _logits_inputs(torch, dev, synth)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            _logits_call(dp, li, t, stream)
    stream.synchronize()

    def timed(pdl):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(calls):
                _logits_call(dp, li, t, stream, pdl=pdl)
        with torch.cuda.stream(stream):
            g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / (calls * reps)

    us = timed(False)
    us_pdl = timed(True)
    us_pdl_early = timed("early")
    T, H, L = li.T, li.H, int(li.context_lens[0])
    nbytes = T * (L * (128 + 4 + 4) + (L // 64) * 4 + H * (128 + 4) + 4)
    flops = 2.0 * T * L * H * 128
    fp8_peak = 2.0 * peaks.get("bf16_tflops", 1900.0)
    return {"workload": f"T={T} H={H} context={L} page_size=64", "us_per_call": us,
            "us_per_call_pdl": us_pdl, "us_per_call_pdl_early": us_pdl_early,
            "gb_per_s": nbytes / us / 1e3, "hbm_frac": nbytes / us / 1e3 / peaks["hbm_gbs"],
            "tflops": flops / us / 1e6, "fp8_peak_tflops": fp8_peak,
            "fp8_frac": flops / us / 1e6 / fp8_peak,
            "peak_note": "fp8 peak = measured bf16 cuBLAS peak x 2 (the nominal fp8/bf16 ratio)",
            "algorithmic_bytes": nbytes, "flops": flops, "calls": calls * reps,
            "gpu_launches": calls * reps}


def probe_workload(which):
    """The inputs and the Hadamard switch of a q+k probe: prefill, prefill_h32,
    prefill_h16, decode, prefill_hadamard or decode_hadamard."""
    import synth
    had = which.endswith("_hadamard")
    base = which[:-len("_hadamard")] if had else which
    if base == "decode":
        return synth.make_decode(seed=1), had
    if base == "prefill":
        return synth.make_prefill(seed=3), had
    if base.startswith("prefill_h") and base[len("prefill_h"):].isdigit():
        return synth.make_prefill(seed=3, H=int(base[len("prefill_h"):])), had
    raise ValueError(f"no probe workload {which!r}")


def run_probe(which, local_rank):
    """A few eager calls on one workload, for ncu captures (no timing, no JSON)."""
    import torch
    import prep_token_gb300 as dp
    import synth
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if which == "logits":
        li, t = _logits_inputs(torch, dev, synth)
        for _ in range(6):
            _logits_call(dp, li, t, torch.cuda.current_stream())
        torch.cuda.synchronize(dev)
        print(f"probe logits: 6 calls (T={li.T}, H={li.H}, context={li.max_context})")
        return
    if which == "k_only":
        sets = [synth.make_k_bulk(seed=6 + i) for i in range(4)]
        sets = [(inp, _k_dev_inputs(inp, dev)) for inp in sets]
        for i in range(6):  # cycling four sets (170 MB, more than L2), as the bench does
            inp, d = sets[i % 4]
            dp.dsa_indexer_k_prepare_store(
                d["k"], d["positions"], d["slots"], d["cos"], d["sin"], d["gamma"], d["beta"],
                inp.eps, d["cache"], inp.page_size, inp.rope_dim, inp.style,
                max_position=inp.max_position)
        torch.cuda.synchronize(dev)
        print(f"probe k_only: 6 calls (T={inp.T}, four input sets)")
        return
    inp, had = probe_workload(which)
    d = _dev_inputs(inp, dev)
    stream = torch.cuda.current_stream()
    for _ in range(6):
        _call(dp, inp, d, stream, hadamard=had)
    torch.cuda.synchronize(dev)
    print(f"probe {which}: 6 calls (T={inp.T}, H={inp.H})")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-unfused", action="store_true")
    ap.add_argument("--no-logits", action="store_true")
    ap.add_argument("--no-hadamard", action="store_true")
    ap.add_argument("--no-stress", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--probe", choices=("prefill", "decode", "logits", "prefill_hadamard",
                                        "decode_hadamard", "k_only", "prefill_h32",
                                        "prefill_h16"),
                    help="make 6 eager calls on that workload and exit (for profilers)")
    ap.add_argument("--traffic-from", nargs=2, metavar=("CSV", "WHICH"),
                    help="write the traffic summary of WHICH (prefill | decode | k_only) "
                         "from an ncu launch-list CSV of the traffic metrics, and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)
    if args.traffic_from:
        print(json.dumps(write_traffic_json(*args.traffic_from)))
        return
    if args.probe:
        run_probe(args.probe, local_rank)
        return
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
