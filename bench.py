#!/usr/bin/env python3
"""Benchmark of the HashEvict decode step (hash + evict + attend) on B300.

One step = one `he_step` call for one attention layer over the whole batch:
code the query heads and the new key, score every cached slot by group-summed
Hamming distance, evict the most dissimilar slot, write the new token into it,
and attend over the retained cache.  A bf16 step is three kernel launches
(cache-streaming attention, codes and eviction, merge and overwrite).

Default workload: the Llama-3-8B-shaped layer (batch 8, 32 query / 8 KV heads,
head_dim 128, bf16, 32-bit codes, budget 4096 of an 8192-token prompt).  The
cache of a layer (129 MiB) is about the size of L2 (126 MB), so the timed steps
rotate over several independent layers (4 by default, 516 MiB): every step
reads a cache that the previous steps evicted from L2.

The timed region replays a CUDA graph of captured he_step calls (the three
launches per step issued once, then replayed), so the number is the device's
step rate; the same steps issued one call at a time from Python are reported
beside it ("eager"), and "e2e" goes through the host-buffer entry point.

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

DEFAULT_WORKLOAD = "llama8b_b8"
FALLBACK_HBM_GBS = 6400.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "stream_kernel_llama8b_b8.md")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--bits", type=int, default=None, help="override the code length")
    ap.add_argument("--budget", type=int, default=None,
                    help="override the cache budget (e.g. a multiple of --chunk)")
    ap.add_argument("--layers", type=int, default=None,
                    help="independent layer caches rotated (default: the workload's own "
                         "layer count if above 1, else 4)")
    ap.add_argument("--ring", type=int, default=512, help="distinct step inputs per layer")
    ap.add_argument("--threshold", type=float, default=0.0,
                    help="binarisation threshold tau (0: the sign test of the method)")
    ap.add_argument("--decay", type=float, default=0.0,
                    help="score memory gamma (0: the step's own distances, the method)")
    ap.add_argument("--v-int8", action="store_true",
                    help="int8 value cache with one scale per slot (keys stay bf16)")
    ap.add_argument("--chunk", type=int, default=1,
                    help="chunk eviction: chunks of this many slots (1: the method)")
    ap.add_argument("--graph-ring", type=int, default=64,
                    help="tokens per layer in the captured step graph (even)")
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU work of the oracle baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="target wall time of the timed oracle steps of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


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


def profiled_traffic():
    """DRAM bytes per launch of the cache-streaming kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    txt = open(PROFILE_SUMMARY).read()
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
            self._stop.wait(0.1)

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
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in self.samples for n, v in zip(names, s[5:9])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


def workload_from(args) -> synth.Workload:
    w = synth.WORKLOADS[args.workload]
    if args.bits:
        w = w.with_(bits=args.bits)
    if args.budget:
        w = w.with_(budget=args.budget, prompt=max(w.prompt, args.budget + 64))
    return w


def config_of(w: synth.Workload, args, extra=None):
    c = {"workload": f"{w.name}: {w.description}" + (
            f"; threshold {args.threshold}, score memory {args.decay}"
            if (args.threshold or args.decay) else "") + (
            "; int8 value cache" if args.v_int8 else "") + (
            f"; chunk eviction, chunks of {args.chunk} slots" if args.chunk > 1 else "") + (
            f"; budget set to {w.budget}" if args.budget else ""),
         "batch": w.batch, "heads": w.heads,
         "kv_heads": w.kv_heads, "head_dim": w.head_dim, "bits": w.bits, "budget": w.budget,
         "prompt": w.prompt, "dtype": w.dtype,
         "cache_fill": "first `budget` prompt tokens; timed steps are streamed tokens " + (
             "(eviction on every step)" if args.chunk <= 1 else
             f"(one chunk eviction every {args.chunk} steps, tokens staged between)")}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline; test infrastructure, never on the product path)
# ---------------------------------------------------------------------------

def run_cpu_baseline(w: synth.Workload, target_s: float, steps: int | None = None,
                     threshold: float = 0.0, decay: float = 0.0, v_int8: bool = False,
                     chunk: int = 1):
    """Times the CPU oracle, as it stands, on a bounded sample of the workload.

    The unit of work is a unit-step: one streamed token through one (batch, KV
    head) unit of layer 0 with a full cache (hash, evict, overwrite, fp64
    attention).  A full step of the workload is batch * kv_heads unit-steps, so
    the throughput is reported as unit-steps / (batch * kv_heads) / second.
    With `steps` = K each timed step is a sample of s units (s sized so that
    the K steps take about target_s of wall time, 1 <= s <= batch * kv_heads);
    without it the sample is every unit for about target_s.  One thread per
    unit on all host cores (the oracle releases the GIL).
    Returns (full steps per second, cores, sample description, seconds)."""
    import concurrent.futures as cf
    import oracle
    o = oracle.load()
    cores = os.cpu_count() or 1
    all_units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    U = len(all_units)
    W = o.projection(w.projection_seed(0), w.head_dim, w.bits, w.dtype)

    def prep(u):
        b, j = u
        K0 = synth.host_unit_kv(w, "key", b, j, 0, w.budget)
        V0 = synth.host_unit_kv(w, "value", b, j, 0, w.budget)
        if chunk > 1:
            return o.unit_fill_chunk(W, w.budget, chunk, K0, V0, tau=threshold)
        return o.unit_fill(W, w.budget, K0, V0, tau=threshold, memory=decay > 0.0, vq=v_int8)

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
    par_unit_s = per_wave / len(cal)  # wall time per unit-step with all cores busy
    budget_unit_steps = max(1, int(target_s / max(par_unit_s, 1e-9)))
    if steps:
        per_step = max(1, min(U, budget_unit_steps // steps))
        total = steps * per_step
    else:
        per_step = None
        total = max(U, budget_unit_steps)
    n_units = min(U, total)
    units = all_units[:n_units]
    toks = [total // n_units + (1 if i < total % n_units else 0) for i in range(n_units)]
    toks = [min(x, w.streamed - 2) for x in toks]
    done = sum(toks)
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        states = list(ex.map(prep, units))
        t = time.perf_counter()
        list(ex.map(lambda a: run(a[0], a[1], 1, a[2]), zip(units, states, toks)))
        el = time.perf_counter() - t
    how = (f"{steps} steps x {per_step} unit(s) per step" if steps else
           f"{done} unit-steps over {n_units} units")
    sample = (f"{w.name}, layer 0: {how} = {done} unit-steps (one streamed token through one "
              f"(batch, KV head) unit with a full cache: hash, evict, overwrite, fp64 attention), "
              f"{n_units} of {U} units, {min(cores, n_units)} threads; throughput scaled to full "
              f"steps as unit-steps / {U}; input generation excluded")
    return done / U / el, min(cores, n_units), sample, el


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, rank: int, world: int, dist_on: bool):
    import torch
    import lsh_pre_attention_decode_b300 as hepkg
    from lsh_pre_attention_decode_b300 import HashEvict, he_step, he_step_host, layer_shard, \
        max_over_ranks

    w = workload_from(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    L = args.layers if args.layers else (w.layers if w.layers > 1 else 4)
    R = args.ring
    # independent shards: rank r takes layers r*L .. r*L+L-1 (weak scaling, no collective)
    layers = layer_shard(rank, world, L)
    handles, inputs = [], []
    for layer in layers:
        he = HashEvict(w.batch, w.heads, w.kv_heads, w.head_dim, w.bits, w.budget, w.dtype,
                       seed=w.projection_seed(layer), threshold=args.threshold,
                       decay=args.decay, v_int8=args.v_int8, chunk=args.chunk)
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
    from lsh_pre_attention_decode_b300._binding import HashEvictError
    he_step_raw = hepkg.lib().he_step
    hs = [he.h for he in handles]
    qp = [[x[0][t].data_ptr() for t in range(R)] for x in inputs]
    kp = [[x[1][t].data_ptr() for t in range(R)] for x in inputs]
    vp = [[x[2][t].data_ptr() for t in range(R)] for x in inputs]
    op = [x[3].data_ptr() for x in inputs]
    cursor = [0]

    def step(sp=None):
        i = cursor[0]
        li = i % L
        t = (i // L) % R
        rc = he_step_raw(hs[li], qp[li][t], kp[li][t], vp[li][t], op[li],
                         stream.cuda_stream if sp is None else sp)
        if rc:
            raise HashEvictError("he_step", rc)
        cursor[0] += 1

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # eager: one he_step call per step from this thread
    n_eager = min(args.steps, 4000)
    ee0 = torch.cuda.Event(enable_timing=True)
    ee1 = torch.cuda.Event(enable_timing=True)
    ee0.record(stream)
    th0 = time.perf_counter()
    for _ in range(n_eager):
        step()
    host_s = time.perf_counter() - th0
    ee1.record(stream)
    torch.cuda.synchronize()
    eager_ms = ee0.elapsed_time(ee1)

    # the timed region replays a CUDA graph of GS steps (graph_ring tokens per
    # layer, in the same round-robin order; an even count per cache keeps the
    # library's per-step double buffering in phase): the host issues one launch
    # per GS steps instead of three per step
    # (with chunk eviction a whole number of staging cycles per cache too, so
    # that every replay starts from the state the capture started from)
    period = 2 * args.chunk // math.gcd(2, args.chunk) if args.chunk > 1 else 2
    Rg = min(args.graph_ring, R)
    Rg -= Rg % period
    if Rg == 0:
        raise SystemExit(f"--graph-ring must hold at least {period} tokens per layer")
    GS = L * Rg
    cursor[0] = 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream().cuda_stream
        for _ in range(GS):
            i = cursor[0]
            li, t = i % L, (i // L) % Rg
            rc = he_step_raw(hs[li], qp[li][t], kp[li][t], vp[li][t], op[li], cap)
            if rc:
                raise HashEvictError("he_step (capture)", rc)
            cursor[0] += 1
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    replays = max(1, (args.steps + GS - 1) // GS)
    K = replays * GS
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
    cursor[0] = 0

    # per-kernel durations: a separate pass in the library's kernel timing mode
    # (CUDA events on the launching stream before the cache-streaming kernel and
    # after each kernel of the step; the events serialise the three kernels)
    nk = min(K, 2000)
    for he in handles:
        he.profile_start(nk // L + 1)
    for _ in range(nk):
        step()
    prof = {"stream_ms": 0.0, "prep_ms": 0.0, "merge_ms": 0.0, "step_ms": 0.0, "steps": 0}
    for he in handles:
        r = he.profile_stop()
        for key in prof:
            prof[key] += r[key]
    n_prof = prof["steps"]
    stream_ms = prof["stream_ms"] / n_prof
    prep_ms = prof["prep_ms"] / n_prof
    merge_ms = prof["merge_ms"] / n_prof
    serial_step_ms = prof["step_ms"] / n_prof

    # chunk eviction: the same timing mode step by step on layer 0's cache,
    # split into evicting steps (the stage is full) and staging steps
    by_type = None
    if args.chunk > 1:
        he0 = handles[0]
        acc = {"evict": [0.0, 0.0, 0.0, 0], "stage": [0.0, 0.0, 0.0, 0]}
        for t in range(8 * args.chunk):
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

    # end to end through the host-buffer entry point: H2D of q, k, v and D2H of
    # out inside every step (pinned host memory), one layer
    he0 = handles[0]
    qh = torch.empty((R,) + tuple(inputs[0][0].shape[1:]), dtype=inputs[0][0].dtype).pin_memory()
    kh = torch.empty((R,) + tuple(inputs[0][1].shape[1:]), dtype=inputs[0][1].dtype).pin_memory()
    vh = torch.empty_like(kh).pin_memory()
    qh.copy_(inputs[0][0].cpu())
    kh.copy_(inputs[0][1].cpu())
    vh.copy_(inputs[0][2].cpu())
    oh = torch.empty(tuple(inputs[0][3].shape), dtype=torch.float32).pin_memory()
    for t in range(3):
        he_step_host(he0.h, qh[t], kh[t], vh[t], oh, stream)
    if dist_on:
        torch.distributed.barrier()
    # the C entry point itself, with the host addresses taken once (as a C
    # caller holds them); the copies and the synchronisation stay inside it
    step_host_raw = hepkg.lib().he_step_host
    qhp = [qh[t].data_ptr() for t in range(R)]
    khp = [kh[t].data_ptr() for t in range(R)]
    vhp = [vh[t].data_ptr() for t in range(R)]
    ohp, sh = oh.data_ptr(), stream.cuda_stream
    n_e2e = args.e2e_steps
    t0 = time.perf_counter()
    for i in range(n_e2e):
        t = i % R
        rc = step_host_raw(he0.h, qhp[t], khp[t], vhp[t], ohp, sh)
        if rc:
            raise HashEvictError("he_step_host", rc)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, dev)
    h2d = qh[0].numel() * qh.element_size() + 2 * kh[0].numel() * kh.element_size()
    d2h = oh.numel() * oh.element_size()

    for he in handles:
        he.close()

    steps_total = K * world
    value = steps_total / (elapsed_ms / 1e3)
    peak, peak_kind = measured_peaks()
    eb = 2 if w.dtype == "bf16" else 4
    occ = w.budget + (args.chunk - 1) / 2  # resident rows (chunk eviction: a cycle's mean)
    U = w.batch * w.kv_heads
    # K and V rows of every resident slot (int8 value rows and their scales with
    # an int8 value cache)
    stream_bytes = int(U * occ * (w.head_dim * eb + (w.head_dim + 4 if args.v_int8
                                                       else w.head_dim * eb)))
    achieved = stream_bytes / (stream_ms / 1e3) / 1e9
    step_gbs = step_bytes / (elapsed_ms / K / 1e3) / 1e9
    launches_per_step = 3 if w.dtype == "bf16" else 1
    res = {
        "metric": "HashEvict decode steps/s (hash+evict+attend); achieved HBM GB/s vs B300 peak",
        "value": value,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": elapsed_ms / K,
        "eager": {"value": n_eager * world / (eager_ms / 1e3), "unit": "steps/s",
                  "ms_per_step": eager_ms / n_eager, "host_ms_per_step": host_s * 1e3 / n_eager,
                  "note": "one he_step call per step from Python (ctypes), no graph"},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "tokens_per_s": value * w.batch,
        "model_steps_per_s": (value / L if w.layers > 1 and L == w.layers else None),
        "config": config_of(w, args, {
            "layers_rotated": L, "ring_tokens_per_layer": R,
            "timed_region": f"{replays} replays of a CUDA graph of {GS} he_step calls "
                            f"({Rg} tokens per layer, round robin over the {L} layers)",
            "l2": f"inputs larger than L2: steps rotate over {L} layer caches of "
                  f"{step_bytes / 2**20:.0f} MiB each",
            "parallelism": f"{world} independent replica(s), layers sharded by rank, no collective",
            "launch": info}),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "peak_source": (f"{peak_kind}: MEASURED_PEAKS.json hbm_gbs (of measured)"
                                     if peak_kind == "measured" else "fallback 6.4 TB/s"),
                     "traffic": profiled_traffic(),
                     "kernel": "he::stream_kernel (cache-streaming attention partials)",
                     "algorithmic_bytes_per_launch": stream_bytes,
                     "kernel_ms": stream_ms,
                     "timing": f"CUDA events on the launching stream around each launch, "
                               f"mean over {n_prof} launches in a pass after the timed region",
                     "other_kernels_ms": {"prep (codes + eviction)": prep_ms,
                                          "merge (LSE merge + overwrite)": merge_ms,
                                          "serialised step": serial_step_ms},
                     "by_step_type": by_type,
                     "step": {"algorithmic_bytes": step_bytes, "achieved": step_gbs,
                              "frac": step_gbs / peak,
                              "note": "he_step_bytes / ms_per_step of the timed region "
                                      "(pipelined: prep overlaps the stream kernel)"}},
        "e2e": {"value": n_e2e / e2e_s * world, "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "api": "he_step_host, the C entry point (host buffers; H2D of q, k, v, the "
                       "step, D2H of out and a stream synchronisation inside every call)"},
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
    }
    return res, w


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        w = workload_from(args)
        val, cores, sample, el = run_cpu_baseline(w, args.ref_seconds, steps=args.steps,
                                                  threshold=args.threshold, decay=args.decay,
                                                  v_int8=args.v_int8, chunk=args.chunk)
        res = {
            "metric": "HashEvict decode steps/s (hash+evict+attend); achieved HBM GB/s vs B300 peak",
            "impl": "reference", "value": val, "unit": "steps/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / val,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, args),
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
    res, w = run_ours(args, rank, world, dist_on)
    if rank == 0:
        if not args.no_cpu_baseline:
            val, cores, sample, el = run_cpu_baseline(w, args.cpu_seconds,
                                                      threshold=args.threshold, decay=args.decay,
                                                      v_int8=args.v_int8, chunk=args.chunk)
            res["cpu_baseline"] = {"value": val, "unit": "steps/s", "cores": cores,
                                   "kind": "oracle", "sample": sample}
        print(json.dumps(res))
    if dist_on:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
