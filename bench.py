#!/usr/bin/env python3
"""Benchmark of the HashEvict decode step (hash + evict + attend) on B300.

One step = one call of the fused step (one kernel launch) for one attention
layer over the whole batch: code the query heads and the new key, score every
cached slot by group-summed Hamming distance, evict the most dissimilar slot,
write the new token into it, and attend over the retained cache.

Default workload: the Llama-3-8B-shaped layer (batch 8, 32 query / 8 KV heads,
head_dim 128, bf16, 32-bit codes, budget 4096 of an 8192-token prompt).  The
cache of a layer (129 MiB) is about the size of L2 (126 MB), so the timed steps
rotate over several independent layers (4 by default, 516 MiB): every step
reads a cache that the previous steps evicted from L2.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle (the
reported baseline) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "step_kernel_llama8b_b8.md")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--bits", type=int, default=None, help="override the code length")
    ap.add_argument("--layers", type=int, default=4, help="independent layer caches rotated")
    ap.add_argument("--ring", type=int, default=512, help="distinct step inputs per layer")
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU work of the oracle baseline sample")
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
    csrc = os.path.join(ROOT, "lsh_pre_attention_decode_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the step kernel from the committed ncu summary, if
    it was taken on the current kernel source; else None."""
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
    return w


def config_of(w: synth.Workload, args, extra=None):
    c = {"workload": f"{w.name}: {w.description}", "batch": w.batch, "heads": w.heads,
         "kv_heads": w.kv_heads, "head_dim": w.head_dim, "bits": w.bits, "budget": w.budget,
         "prompt": w.prompt, "dtype": w.dtype,
         "cache_fill": "first `budget` prompt tokens; timed steps are streamed tokens "
                       "(eviction on every step)"}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline; test infrastructure, never on the product path)
# ---------------------------------------------------------------------------

def run_cpu_baseline(w: synth.Workload, target_s: float):
    """Times the CPU oracle, as it stands, on a bounded sample of the workload:
    every (batch, KV head) unit of one layer, the first S streamed tokens, all
    cores (one thread per unit, the oracle releases the GIL).  Returns
    (steps_per_s, cores, sample description, seconds)."""
    import concurrent.futures as cf
    import oracle
    o = oracle.load()
    cores = os.cpu_count() or 1
    units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    W = o.projection(w.projection_seed(0), w.head_dim, w.bits, w.dtype)

    def prep(u):
        b, j = u
        st = o.unit_fill(W, w.budget, synth.host_unit_kv(w, "key", b, j, 0, w.budget),
                         synth.host_unit_kv(w, "value", b, j, 0, w.budget))
        return st

    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        states = list(ex.map(prep, units))

    def run(u, st, t0, n):
        b, j = u
        q = synth.host_unit_queries(w, b, j, w.budget + t0, n)
        k = synth.host_unit_kv(w, "key", b, j, w.budget + t0, n)
        v = synth.host_unit_kv(w, "value", b, j, w.budget + t0, n)
        t = time.perf_counter()
        o.unit_stream(st, q, k, v)
        return time.perf_counter() - t

    # calibrate with one step, then size the sample to about target_s of wall time
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        t = time.perf_counter()
        list(ex.map(lambda a: run(*a, 0, 1), zip(units, states)))
        one = time.perf_counter() - t
    n = max(1, min(w.streamed - 1, int(target_s / max(one, 1e-6))))
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        t = time.perf_counter()
        list(ex.map(lambda a: run(*a, 1, n), zip(units, states)))
        el = time.perf_counter() - t
    sample = (f"{w.name}, layer 0, all {len(units)} (batch, KV head) units, streamed tokens "
              f"1..{n} after a full cache ({n} steps), hash+evict+attend (fp64 attention), "
              f"{cores} threads over units; input generation excluded")
    return n / el, cores, sample, el


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, rank: int, world: int, dist_on: bool):
    import torch
    import lsh_pre_attention_decode_b300 as hepkg
    from lsh_pre_attention_decode_b300 import HashEvict, he_step, he_step_host

    w = workload_from(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    L = args.layers
    R = args.ring
    # independent shards: rank r takes layers r*L .. r*L+L-1 (weak scaling, no collective)
    layers = [rank * L + i for i in range(L)]
    handles, inputs = [], []
    for layer in layers:
        he = HashEvict(w.batch, w.heads, w.kv_heads, w.head_dim, w.bits, w.budget, w.dtype,
                       seed=w.projection_seed(layer))
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

    cursor = [0]

    def step():
        i = cursor[0]
        li = i % L
        t = (i // L) % R
        q, k, v, out = inputs[li]
        he_step(handles[li].h, q[t], k[t], v[t], out, stream)
        cursor[0] += 1

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    K = args.steps
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    elapsed_ms = e0.elapsed_time(e1)
    if dist_on:
        t = torch.tensor([elapsed_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())

    # per-launch durations of the step kernel (events bracket each launch)
    nk = min(K, 2000)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(nk)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(nk)]
    for i in range(nk):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    kern_ms = float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)]))

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
    n_e2e = args.e2e_steps
    t0 = time.perf_counter()
    for i in range(n_e2e):
        t = i % R
        he_step_host(he0.h, qh[t], kh[t], vh[t], oh, stream)
    e2e_s = time.perf_counter() - t0
    if dist_on:
        tt = torch.tensor([e2e_s], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(tt.item())
    h2d = qh[0].numel() * qh.element_size() + 2 * kh[0].numel() * kh.element_size()
    d2h = oh.numel() * oh.element_size()

    for he in handles:
        he.close()

    steps_total = K * world
    value = steps_total / (elapsed_ms / 1e3)
    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (kern_ms / 1e3) / 1e9
    res = {
        "metric": "HashEvict decode steps/s (hash+evict+attend); achieved HBM GB/s vs B300 peak",
        "value": value,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": elapsed_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "tokens_per_s": value * w.batch,
        "config": config_of(w, args, {
            "layers_rotated": L, "ring_tokens_per_layer": R,
            "l2": f"inputs larger than L2: steps rotate over {L} layer caches of "
                  f"{step_bytes / 2**20:.0f} MiB each",
            "parallelism": f"{world} independent replica(s), layers sharded by rank, no collective",
            "launch": info}),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json "
                     "hbm_gbs)" if peak_kind == "measured" else "fallback 6.4 TB/s",
                     "traffic": profiled_traffic(), "algorithmic_bytes_per_launch": step_bytes,
                     "kernel_ms": kern_ms, "kernel": "he::step_kernel (one launch per step)"},
        "e2e": {"value": n_e2e / e2e_s * world, "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "api": "he_step_host (host buffers; copies and synchronisation inside)"},
        "gpu_launches": K,
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
        val, cores, sample, el = run_cpu_baseline(w, args.cpu_seconds)
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
            val, cores, sample, el = run_cpu_baseline(w, args.cpu_seconds)
            res["cpu_baseline"] = {"value": val, "unit": "steps/s", "cores": cores,
                                   "kind": "oracle", "sample": sample}
        print(json.dumps(res))
    if dist_on:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
