#!/usr/bin/env python3
"""Benchmark of the HashEvict decode step (hash + evict + attend) on B300.

One layer-step = one `he_step` call for one attention layer over the whole
batch: code the query heads and the new key, score every cached slot by
group-summed Hamming distance, evict the most dissimilar slot, write the new
token into it, and attend over the retained cache.  A bf16 layer-step is three
kernel launches (cache-streaming attention, codes and eviction, merge and
overwrite).

Headline workload: the 32-layer Llama-3-8B-shaped decode loop (batch 16,
32 query / 8 KV heads, head_dim 128, bf16, 32-bit codes, budget 9728 of a
32768-token prompt, 32 independent layer caches, 20 GB of cache).  One decode
step is one token through all 32 layers: 32 layer-steps.  The timed region
replays a CUDA graph of captured he_step calls (64 tokens per layer, round robin
over the layers, as a serving loop issues them), at least 0.5 s of it however
few steps are asked for.  `per_config` repeats the measurement on the other
workloads (the Llama-3-8B layer at batch 8, the 128K-token sequence, batch 64,
and the 32-layer loop at code lengths 8, 16 and 64), each with its own clock
record; the smaller ones rotate over several layer caches so that every step
reads a cache that is not in L2 (126 MB).

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle (the
reported baseline) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "HashEvict decode steps/s (hash+evict+attend); achieved HBM GB/s vs B300 peak"
DEFAULT_WORKLOAD = "llama8b_32layer"
FALLBACK_HBM_GBS = 6400.0
NOMINAL_HBM_GBS = 8000.0  # B300 HBM3e, nominal (NVIDIA's figure is about 8 TB/s)
# the other workloads measured by a default run: (workload, code length or None, layers rotated)
PER_CONFIG = [("llama8b_b8", None, 4), ("long_128k", None, 4), ("serving_b64", None, 2),
              ("llama8b_32layer", 8, 32), ("llama8b_32layer", 16, 32),
              ("llama8b_32layer", 64, 32)]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64,
                    help="decode steps to time at least (the timed region also lasts at least "
                         "--min-seconds)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--bits", type=int, default=None, help="override the code length")
    ap.add_argument("--budget", type=int, default=None,
                    help="override the cache budget (e.g. a multiple of --chunk)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer caches (default: the workload's own layer count if above 1, "
                         "else 4)")
    ap.add_argument("--min-seconds", type=float, default=0.5,
                    help="shortest timed region of the headline workload")
    ap.add_argument("--config-seconds", type=float, default=0.3,
                    help="shortest timed region of each per_config workload")
    ap.add_argument("--threshold", type=float, default=0.0,
                    help="binarisation threshold tau (0: the sign test of the method)")
    ap.add_argument("--tau-mode", choices=["fixed", "median"], default="fixed",
                    help="median: one threshold per bit and (batch, KV head), the lower "
                         "median of the filled keys' projections (--threshold unused)")
    ap.add_argument("--decay", type=float, default=0.0,
                    help="score memory gamma (0: the step's own distances, the method)")
    ap.add_argument("--v-format", choices=["elem", "int8", "fp8"], default="elem",
                    help="value cache rows: bf16 (elem), or int8 / fp8 (E4M3) bytes with one "
                         "scale per slot (keys stay bf16)")
    ap.add_argument("--chunk", type=int, default=1,
                    help="chunk eviction: chunks of this many slots (1: the method)")
    ap.add_argument("--engine", choices=["pipeline", "fused"], default="pipeline",
                    help="bf16 step engine: three kernels (default) or one kernel")
    ap.add_argument("--graph-ring", type=int, default=64,
                    help="tokens per layer in the captured step graph (even)")
    ap.add_argument("--e2e-steps", type=int, default=8, help="decode steps of the e2e pass")
    ap.add_argument("--eager-steps", type=int, default=8,
                    help="decode steps of the eager (one call per layer-step) pass")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU work of the headline's all-core oracle sample")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="target wall time of the timed oracle steps of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha() -> str:
    """Hash of the kernel sources with comments and whitespace removed: an edit
    of the code (not of its comments) invalidates a committed ncu summary."""
    csrc = os.path.join(ROOT, "lsh_pre_attention_decode_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                src = fh.read()
            src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
            src = re.sub(r"//[^\n]*", " ", src)
            h.update(f.encode())
            h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the cache-streaming kernel from the committed ncu
    summary of this workload, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"stream_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_sha or not m_tr or m_sha.group(1) != kernel_source_sha():
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _query(self):
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                 timeout=5).stdout.strip()
            f = [x.strip() for x in out.split(",")]
            if len(f) >= 9:
                self.samples.append(f)
        except Exception:
            pass

    def _run(self):
        while not self._stop.is_set():
            self._query()
            self._stop.wait(0.05)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=10)
        if not self.samples:
            self._query()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        pw = [float(s[3]) for s in self.samples if s[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in self.samples for n, v in zip(names, s[5:9])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(self.samples)}


def make_workload(name: str, bits=None, budget=None) -> synth.Workload:
    w = synth.WORKLOADS[name]
    if bits:
        w = w.with_(bits=bits)
    if budget:
        w = w.with_(budget=budget, prompt=max(w.prompt, budget + 64))
    return w


def step_unit(w: synth.Workload) -> str:
    return ("one decode token through all %d attention layers (%d he_step calls)"
            % (w.layers, w.layers) if w.layers > 1 else
            "one he_step call (one attention layer, the whole batch)")


def config_of(w: synth.Workload, opts: dict, extra=None):
    chunk = opts.get("chunk", 1)
    c = {"workload": f"{w.name}: {w.description}" + (
            f"; threshold {opts.get('threshold')}, score memory {opts.get('decay')}"
            if (opts.get("threshold") or opts.get("decay")) else "") + (
            "; per-bit median thresholds" if opts.get("tau_mode") == "median" else "") + (
            f"; {opts.get('v_format')} value cache"
            if opts.get("v_format", "elem") != "elem" else "") + (
            f"; chunk eviction, chunks of {chunk} slots" if chunk > 1 else "") + (
            "; single-kernel engine" if opts.get("engine") == "fused" else "") + (
            f"; code length {w.bits}" if w.bits != synth.WORKLOADS[w.name].bits else "") + (
            f"; budget set to {w.budget}" if w.budget != synth.WORKLOADS[w.name].budget else ""),
         "batch": w.batch, "heads": w.heads, "kv_heads": w.kv_heads, "head_dim": w.head_dim,
         "bits": w.bits, "budget": w.budget, "prompt": w.prompt, "dtype": w.dtype,
         "layers": w.layers, "step": step_unit(w),
         "cache_fill": "first `budget` prompt tokens; timed steps are streamed tokens " + (
             "(eviction on every step)" if chunk <= 1 else
             f"(one chunk eviction every {chunk} steps, tokens staged between)")}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline; test infrastructure, never on the product path)
# ---------------------------------------------------------------------------

def run_cpu_baseline(w: synth.Workload, target_s: float, steps: int | None = None,
                     threads: int | None = None, threshold: float = 0.0, decay: float = 0.0,
                     tau_mode: str = "fixed",
                     v_format: str = "elem", chunk: int = 1):
    """Times the CPU oracle, as it stands, on a bounded sample of the workload.

    The unit of work is a unit-step: one streamed token through one (batch, KV
    head) unit of layer 0 with a full cache (hash, evict, overwrite, fp64
    attention).  A layer-step of the workload is batch * kv_heads unit-steps and
    a decode step is `layers` layer-steps, so the throughput is reported as
    unit-steps / (batch * kv_heads * layers) / second: an extrapolation from the
    sample (every unit and layer costs the same).  With `steps` = K each timed
    step is a sample of s units (s sized so that the K steps take about
    target_s of wall time); without it the sample is up to every unit for about
    target_s.  `threads` host threads, one unit each (default: every core; the
    oracle releases the GIL).
    Returns (decode steps per second, threads used, sample description, seconds)."""
    import concurrent.futures as cf
    import oracle
    o = oracle.load()
    cores = threads or os.cpu_count() or 1
    all_units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    U = len(all_units)
    W = o.projection(w.projection_seed(0), w.head_dim, w.bits, w.dtype)

    def prep(u):
        b, j = u
        K0 = synth.host_unit_kv(w, "key", b, j, 0, w.budget)
        V0 = synth.host_unit_kv(w, "value", b, j, 0, w.budget)
        median = tau_mode == "median"
        if chunk > 1:
            return o.unit_fill_chunk(W, w.budget, chunk, K0, V0, tau=threshold, median=median)
        return o.unit_fill(W, w.budget, K0, V0, tau=threshold, memory=decay > 0.0,
                           vq=False if v_format == "elem" else v_format, median=median)

    def run(u, st, t0, n):
        b, j = u
        q = synth.host_unit_queries(w, b, j, w.budget + t0, n)
        k = synth.host_unit_kv(w, "key", b, j, w.budget + t0, n)
        v = synth.host_unit_kv(w, "value", b, j, w.budget + t0, n)
        t = time.perf_counter()
        o.unit_stream(st, q, k, v, decay=decay)
        return time.perf_counter() - t

    # calibrate: one token through min(U, cores) units in parallel
    cal = all_units[:min(U, cores)]
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        cal_states = list(ex.map(prep, cal))
        t = time.perf_counter()
        list(ex.map(lambda a: run(*a, 0, 1), zip(cal, cal_states)))
        per_wave = time.perf_counter() - t
    par_unit_s = per_wave / len(cal)  # wall time per unit-step with the threads busy
    budget_unit_steps = max(1, int(target_s / max(par_unit_s, 1e-9)))
    if steps:
        per_step = max(1, min(U, budget_unit_steps // steps))
        total = steps * per_step
    else:
        per_step = None
        total = max(min(U, cores), budget_unit_steps)
    # (enough units to keep the threads busy; more would only add set-up time)
    n_units = min(U, total, 2 * cores if cores > 1 else 4)
    units = all_units[:n_units]
    toks = [total // n_units + (1 if i < total % n_units else 0) for i in range(n_units)]
    toks = [max(1, min(x, w.streamed - 2)) for x in toks]
    done = sum(toks)
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        states = list(ex.map(prep, units))
        t = time.perf_counter()
        list(ex.map(lambda a: run(a[0], a[1], 1, a[2]), zip(units, states, toks)))
        el = time.perf_counter() - t
    per_model_step = U * w.layers
    how = (f"{steps} steps x {per_step} unit(s) per step" if steps else
           f"{done} unit-steps over {n_units} units")
    full = n_units == U and w.layers == 1
    sample = (f"{w.name}, layer 0: {how} = {done} unit-steps (one streamed token through one "
              f"(batch, KV head) unit with a full cache: hash, evict, overwrite, fp64 attention), "
              f"{n_units} of {U} units, {min(cores, n_units)} thread(s); throughput scaled to "
              f"decode steps as unit-steps / {per_model_step} ({U} units x {w.layers} layer(s))"
              + ("" if full else ", extrapolated from the sampled units") +
              "; input generation excluded")
    return done / per_model_step / el, min(cores, n_units), sample, el


def cpu_baselines(w: synth.Workload, target_s: float, **opts) -> dict:
    """The oracle on every host core and on one thread, each a bounded sample."""
    val, cores, sample, _ = run_cpu_baseline(w, target_s, **opts)
    v1, _, sample1, _ = run_cpu_baseline(w, target_s / 3, threads=1, **opts)
    return {"value": val, "unit": "steps/s", "cores": cores, "kind": "oracle", "sample": sample,
            "extrapolated": "every unit and layer is taken to cost what the sampled ones did",
            "single_thread": {"value": v1, "unit": "steps/s", "cores": 1, "sample": sample1}}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def measure(w: synth.Workload, opts: dict, L: int, min_s: float, min_steps: int, warmup: int,
            graph_ring: int, rank: int, world: int, dist_on: bool, eager_steps: int = 0,
            e2e_steps: int = 0) -> dict:
    """Times `w` with L layer caches (this rank's shard), as a CUDA graph of
    captured he_step calls replayed back to back.  Returns the measurement."""
    import ctypes
    import torch
    import lsh_pre_attention_decode_b300 as hepkg
    from lsh_pre_attention_decode_b300 import HashEvict, layer_shard, max_over_ranks
    from lsh_pre_attention_decode_b300._binding import HashEvictError

    chunk = opts.get("chunk", 1)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    period = 2 * chunk // math.gcd(2, chunk) if chunk > 1 else 2
    Rg = min(graph_ring, 512)
    Rg -= Rg % period
    if Rg == 0:
        raise SystemExit(f"--graph-ring must hold at least {period} tokens per layer")
    R = Rg  # distinct inputs per layer: the captured ones
    layers = layer_shard(rank, world, L)
    handles, inputs = [], []
    for layer in layers:
        he = HashEvict(w.batch, w.heads, w.kv_heads, w.head_dim, w.bits, w.budget, w.dtype,
                       seed=w.projection_seed(layer), threshold=opts.get("threshold", 0.0),
                       decay=opts.get("decay", 0.0), v_format=opts.get("v_format", "elem"),
                       chunk=chunk, engine=opts.get("engine", "pipeline"),
                       tau_mode=opts.get("tau_mode", "fixed"))
        K = synth.gpu_kv(w, "key", 0, w.budget, layer)
        V = synth.gpu_kv(w, "value", 0, w.budget, layer)
        he.fill(K, V)
        del K, V
        q = synth.gpu_queries(w, w.budget, R, layer)
        k = synth.gpu_kv(w, "key", w.budget, R, layer, token_major=True)
        v = synth.gpu_kv(w, "value", w.budget, R, layer, token_major=True)
        out = torch.empty((w.batch, w.heads, w.head_dim), dtype=torch.float32, device=dev)
        handles.append(he)
        inputs.append((q, k, v, out))
    torch.cuda.synchronize()

    # raw entry-point calls with the input addresses taken once (the Python
    # wrapper's per-call conversions cost more host time than a step takes)
    he_step_raw = hepkg.lib().he_step
    hs = [he.h for he in handles]
    qp = [[x[0][t].data_ptr() for t in range(R)] for x in inputs]
    kp = [[x[1][t].data_ptr() for t in range(R)] for x in inputs]
    vp = [[x[2][t].data_ptr() for t in range(R)] for x in inputs]
    op = [x[3].data_ptr() for x in inputs]
    Ln = len(hs)
    # layer-steps per reported step: every layer of a multi-layer workload (one
    # decode token through the model), else one he_step call
    per = Ln if w.layers > 1 else 1

    def issue(i, sp):
        li, t = i % Ln, (i // Ln) % R
        rc = he_step_raw(hs[li], qp[li][t], kp[li][t], vp[li][t], op[li], sp)
        if rc:
            raise HashEvictError("he_step", rc)

    # warm-up decode steps (every layer once per decode step), eager
    n_warm = max(warmup, 3) * Ln
    for i in range(n_warm):
        issue(i, stream.cuda_stream)
    torch.cuda.synchronize()
    res = {}
    if eager_steps > 0:
        # one he_step call per layer-step from this thread, no graph
        n_eager = Ln * max(eager_steps, period)
        n_eager -= n_eager % (Ln * period)
        ee0 = torch.cuda.Event(enable_timing=True)
        ee1 = torch.cuda.Event(enable_timing=True)
        ee0.record(stream)
        th0 = time.perf_counter()
        for i in range(n_eager):
            issue(i, stream.cuda_stream)
        host_s = time.perf_counter() - th0
        ee1.record(stream)
        torch.cuda.synchronize()
        eager_ms = ee0.elapsed_time(ee1)
        res["eager"] = {"value": n_eager / per * world / (eager_ms / 1e3), "unit": "steps/s",
                        "layer_steps": n_eager, "ms_per_step": eager_ms / (n_eager / per),
                        "host_ms_per_layer_step": host_s * 1e3 / n_eager,
                        "note": "one he_step call per layer-step from Python (ctypes), no graph"}

    # the timed region replays a CUDA graph of GS layer-steps (Rg tokens per
    # layer, round robin; an even count per cache, and with chunk eviction a
    # whole number of staging cycles, so that every replay starts from the state
    # the capture started from)
    GS = Ln * Rg
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream().cuda_stream
        for i in range(GS):
            issue(i, cap)
    graph.replay()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    replay_s = g0.elapsed_time(g1) / 1e3
    replays = max(1, math.ceil(min_steps * Ln / GS), math.ceil(min_s / max(replay_s, 1e-6)))
    replays = int(max_over_ranks(replays, dev))
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0.record(stream)
        for _ in range(replays):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    del graph
    layer_steps = replays * GS

    # per-kernel durations: a separate pass in the library's kernel timing mode
    # (CUDA events on the launching stream before the cache-streaming kernel and
    # after each kernel of the step; the events serialise the three kernels)
    nk = min(layer_steps, max(256, 8 * Ln))
    nk = max(Ln * period, nk - nk % (Ln * period))  # whole cycles, at least one
    for he in handles:
        he.profile_start(nk // Ln + 1)
    for i in range(nk):
        issue(i, stream.cuda_stream)
    prof = {"stream_ms": 0.0, "prep_ms": 0.0, "merge_ms": 0.0, "step_ms": 0.0, "steps": 0}
    for he in handles:
        r = he.profile_stop()
        for key in prof:
            prof[key] += r[key]
    n_prof = prof["steps"]

    # chunk eviction: the same timing mode step by step on layer 0's cache,
    # split into evicting steps (the stage is full) and staging steps
    by_type = None
    if chunk > 1:
        he0 = handles[0]
        acc = {"evict": [0.0, 0.0, 0.0, 0], "stage": [0.0, 0.0, 0.0, 0]}
        for t in range(8 * chunk):
            kind = "evict" if he0.occupancy == he0.rows else "stage"
            he0.profile_start(1)
            rc = he_step_raw(hs[0], qp[0][t % R], kp[0][t % R], vp[0][t % R], op[0],
                             stream.cuda_stream)
            if rc:
                raise HashEvictError("he_step", rc)
            r = he0.profile_stop()
            a = acc[kind]
            a[0] += r["stream_ms"]
            a[1] += r["prep_ms"]
            a[2] += r["merge_ms"]
            a[3] += 1
        by_type = {k: {"steps": a[3], "stream_ms": a[0] / a[3], "prep_ms": a[1] / a[3],
                       "merge_ms": a[2] / a[3]} for k, a in acc.items() if a[3]}

    step_bytes = handles[0].step_bytes
    info = handles[0].launch_info()

    e2e = None
    if e2e_steps > 0:
        # end to end through the host-buffer entry point he_step_host: per
        # layer-step the H2D of q, k, v from pinned host memory, the step, the
        # D2H of out and a stream synchronisation, all inside the call
        x0 = inputs[0]
        qh = torch.empty((R,) + tuple(x0[0].shape[1:]), dtype=x0[0].dtype).pin_memory()
        kh = torch.empty((R,) + tuple(x0[1].shape[1:]), dtype=x0[1].dtype).pin_memory()
        vh = torch.empty_like(kh).pin_memory()
        qh.copy_(x0[0].cpu())
        kh.copy_(x0[1].cpu())
        vh.copy_(x0[2].cpu())
        oh = torch.empty(tuple(x0[3].shape), dtype=torch.float32).pin_memory()
        step_host_raw = hepkg.lib().he_step_host
        qhp = [qh[t].data_ptr() for t in range(R)]
        khp = [kh[t].data_ptr() for t in range(R)]
        vhp = [vh[t].data_ptr() for t in range(R)]
        ohp, sh = oh.data_ptr(), stream.cuda_stream
        n_e2e = e2e_steps * Ln
        n_e2e -= n_e2e % (Ln * period)
        n_e2e = max(n_e2e, Ln * period)

        def host_step(i):
            li, t = i % Ln, (i // Ln) % R
            rc = step_host_raw(hs[li], qhp[t], khp[t], vhp[t], ohp, sh)
            if rc:
                raise HashEvictError("he_step_host", rc)
        for i in range(Ln * period):
            host_step(i)
        if dist_on:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            host_step(i)
        e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
        h2d = qh[0].numel() * qh.element_size() + 2 * kh[0].numel() * kh.element_size()
        d2h = oh.numel() * oh.element_size()
        e2e = {"value": n_e2e / per / e2e_s * world, "unit": "steps/s",
               "h2d_bytes_per_step": h2d * per, "d2h_bytes_per_step": d2h * per,
               "api": "he_step_host, the C entry point (host buffers; per layer-step the H2D of "
                      "q, k, v, the step, the D2H of out and a stream synchronisation inside "
                      "the call; the host addresses taken once, as a C caller holds them)"}

    for he in handles:
        he.close()
    del inputs
    torch.cuda.synchronize()

    peak, peak_kind = measured_peaks()
    eb = 2 if w.dtype == "bf16" else 4
    occ = w.budget + (chunk - 1) / 2  # resident rows (chunk eviction: a cycle's mean)
    U = w.batch * w.kv_heads
    # K and V rows of every resident slot (byte value rows and their scales with
    # a quantised value cache)
    vq = opts.get("v_format", "elem") != "elem"
    stream_bytes = int(U * occ * (w.head_dim * eb + (w.head_dim + 4 if vq
                                                       else w.head_dim * eb)))
    stream_ms = prof["stream_ms"] / n_prof
    achieved = stream_bytes / (stream_ms / 1e3) / 1e9
    ms_per_layer_step = elapsed_ms / layer_steps
    step_gbs = step_bytes / (ms_per_layer_step / 1e3) / 1e9
    decode_steps = layer_steps / per
    value = decode_steps * world / (elapsed_ms / 1e3)
    res.update({
        "value": value, "unit": "steps/s", "steps": int(decode_steps), "layer_steps": layer_steps,
        "layer_steps_per_s": layer_steps * world / (elapsed_ms / 1e3),
        "tokens_per_s": value * w.batch, "ms_per_step": elapsed_ms / decode_steps,
        "timed_s": elapsed_ms / 1e3,
        "timed_region": f"{replays} replays of a CUDA graph of {GS} he_step calls ({Rg} tokens "
                        f"per layer, round robin over {Ln} layer caches), {elapsed_ms:.0f} ms",
        "l2": f"inputs larger than L2: steps rotate over {Ln} layer caches of "
              f"{step_bytes / 2**20:.0f} MiB each",
        "launch": info,
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak,
            "peak_source": (f"{peak_kind}: MEASURED_PEAKS.json hbm_gbs (of measured)"
                            if peak_kind == "measured" else "fallback 6.4 TB/s (of fallback)"),
            "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
            # (the committed summaries are of the method's three-kernel stream kernel)
            "traffic": profiled_traffic(w.name) if w.bits == synth.WORKLOADS[w.name].bits
            and is_method(opts) and opts.get("engine", "pipeline") == "pipeline" else None,
            "kernel": "he::stream_kernel (cache-streaming attention partials)",
            "algorithmic_bytes_per_launch": stream_bytes,
            "kernel_ms": stream_ms,
            "timing": f"CUDA events on the launching stream around each launch, mean over "
                      f"{n_prof} launches in a pass after the timed region",
            "other_kernels_ms": {"prep (codes + eviction)": prof["prep_ms"] / n_prof,
                                 "merge (LSE merge + overwrite)": prof["merge_ms"] / n_prof,
                                 "serialised step": prof["step_ms"] / n_prof},
            "by_step_type": by_type,
            "step": {"algorithmic_bytes_per_layer_step": step_bytes, "achieved": step_gbs,
                     "frac": step_gbs / peak, "frac_of_nominal_8tbs": step_gbs / NOMINAL_HBM_GBS,
                     "note": "he_step_bytes / time per layer-step of the timed region "
                             "(pipelined: prep overlaps the stream kernel)"}},
        "gpu_launches": (3 if w.dtype == "bf16" else 1) * layer_steps,
        "clocks": clk.summary(),
    })
    if e2e:
        res["e2e"] = e2e
    return res


def is_method(opts: dict) -> bool:
    """The options are those of the method as the pages describe it."""
    return (not opts.get("threshold") and not opts.get("decay") and opts.get("chunk", 1) <= 1
            and opts.get("tau_mode", "fixed") == "fixed"
            and opts.get("v_format", "elem") == "elem")


def run_ours(args, rank: int, world: int, dist_on: bool):
    w = make_workload(args.workload, args.bits, args.budget)
    opts = {"threshold": args.threshold, "decay": args.decay, "v_format": args.v_format,
            "tau_mode": args.tau_mode,
            "chunk": args.chunk, "engine": args.engine}
    L = args.layers if args.layers else (w.layers if w.layers > 1 else 4)
    if w.layers > 1 and L != w.layers:
        w = w.with_(layers=L)
    head = measure(w, opts, L, args.min_seconds, args.steps, args.warmup, args.graph_ring, rank,
                   world, dist_on, eager_steps=args.eager_steps, e2e_steps=args.e2e_steps)
    res = {"metric": METRIC, "value": head.pop("value"), "unit": "steps/s", "n_gpus": world,
           "steps": head.pop("steps"), "steps_requested": args.steps,
           "warmup": max(args.warmup, 3), "ms_per_step": head.pop("ms_per_step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
           "data": "synthetic (seeded generator, the pages' workload shapes; no model weights)"}
    res["tokens_per_s"] = head.pop("tokens_per_s")
    res["layer_steps_per_s"] = head.pop("layer_steps_per_s")
    res["config"] = config_of(w, opts, {
        "layers_per_rank": L, "timed_region": head.pop("timed_region"), "l2": head.pop("l2"),
        "parallelism": f"{world} independent replica(s), layers sharded by rank, no collective",
        "launch": head.pop("launch")})
    for key in ("roofline", "e2e", "gpu_launches", "clocks", "eager", "layer_steps", "timed_s"):
        if key in head:
            res[key] = head.pop(key)
    per_meta = []
    if not args.no_per_config and world == 1:
        per = {}
        for name, bits, layers in PER_CONFIG:
            wc = make_workload(name, bits)
            copts = {"engine": args.engine}
            if (wc.name, wc.bits) == (w.name, w.bits) and is_method(opts):
                continue
            key = name if bits is None else f"{name}_b{bits}"
            r = measure(wc, copts, layers, args.config_seconds, 0, args.warmup, args.graph_ring, rank,
                        world, dist_on)
            per[key] = {"config": config_of(wc, copts, {"layers_rotated": layers,
                                                     "timed_region": r.pop("timed_region")}),
                        **{k: r[k] for k in ("value", "unit", "ms_per_step", "layer_steps_per_s",
                                             "tokens_per_s", "steps", "timed_s", "roofline",
                                             "clocks", "gpu_launches")}}
            per_meta.append((key, wc))
        res["per_config"] = per
    return res, w, opts, per_meta


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    opts = {"threshold": args.threshold, "decay": args.decay, "v_format": args.v_format,
            "tau_mode": args.tau_mode,
            "chunk": args.chunk}

    if args.impl == "reference":
        if rank != 0:
            return 0
        w = make_workload(args.workload, args.bits, args.budget)
        val, cores, sample, el = run_cpu_baseline(w, args.ref_seconds, steps=args.steps, **opts)
        res = {
            "metric": METRIC, "impl": "reference", "value": val, "unit": "steps/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / val,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator, the pages' workload shapes; no model weights)",
            "config": config_of(w, opts),
            "cpu_baseline": {"value": val, "unit": "steps/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(res))
        return 0

    import torch
    dist_on = world > 1
    if dist_on:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import lsh_pre_attention_decode_b300 as hepkg
    hepkg.lib()
    res, w, opts, per_meta = run_ours(args, rank, world, dist_on)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baselines(
                w, args.cpu_seconds, **{k: v for k, v in opts.items() if k != "engine"})
            for key, wc in per_meta:
                res["per_config"][key]["cpu_baseline"] = cpu_baselines(wc, 3.0)
        print(json.dumps(res))
    if dist_on:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
