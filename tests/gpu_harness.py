"""Shared helpers of the GPU parity tests: run a workload's token stream through
the CUDA library (via the C ABI binding) and through the CPU oracle, and
compare.  The oracle's inputs always come from the host build of the generator;
the GPU side takes either the same host tensors or the device build of the
generator (checked bit-exact against the host build in test_gpu_generator).
"""
from __future__ import annotations

import concurrent.futures as cf
from dataclasses import dataclass

import numpy as np

import oracle
import synth

# Attention-output tolerance against the fp64 oracle on the identical retained cache.
MAX_ABS_TOL = 1e-2
MEAN_ABS_TOL = 1e-3


def torch_from_host(a: np.ndarray, device="cuda"):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(a.copy()).to(device)


def host_from_torch(t) -> np.ndarray:
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@dataclass
class GpuRun:
    evicted: np.ndarray        # [steps][batch][kv_heads]
    outs: dict                 # step index -> out [batch][heads][D] float32
    state: tuple | None        # (K, V, codes, occupancy) after the run
    prof: dict | None = None   # summed kernel times of the library's timing mode


def make_handle(w: synth.Workload, layer: int = 0, threshold: float = 0.0, decay: float = 0.0,
                v_int8: bool = False, chunk: int = 1):
    from lsh_pre_attention_decode_b300 import HashEvict
    return HashEvict(w.batch, w.heads, w.kv_heads, w.head_dim, w.bits, w.budget, w.dtype,
                     seed=w.projection_seed(layer), threshold=threshold, decay=decay,
                     v_int8=v_int8, chunk=chunk)


def run_gpu(w: synth.Workload, fill_n: int, steps: int, out_steps=(), layer: int = 0,
            device_gen: bool = False, read_state: bool = False, batch_tokens: int = 256,
            profile: bool = False, threshold: float = 0.0, decay: float = 0.0,
            v_int8: bool = False, chunk: int = 1) -> GpuRun:
    """Fill with prompt tokens [0, fill_n), then stream tokens fill_n .. fill_n+steps-1
    (generated batch_tokens at a time).  With decay > 0 the returned state also
    holds the per-slot scores; with an int8 value cache, V is int8 and the value
    scales follow; chunk > 1: chunk eviction (state rows budget + chunk - 1)."""
    import torch
    out_steps = set(out_steps)
    he = make_handle(w, layer, threshold, decay, v_int8, chunk)
    try:
        if fill_n > 0:
            if device_gen:
                K = synth.gpu_kv(w, "key", 0, fill_n, layer)
                V = synth.gpu_kv(w, "value", 0, fill_n, layer)
            else:
                K = torch_from_host(synth.host_kv(w, "key", 0, fill_n, layer))
                V = torch_from_host(synth.host_kv(w, "value", 0, fill_n, layer))
            he.fill(K, V)
            del K, V
        else:
            he.fill(None, None)
        if profile:
            he.profile_start(steps)
        evicted = np.empty((steps, w.batch, w.kv_heads), np.int32)
        outs = {}
        out = torch.empty((w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
        for c0 in range(0, steps, batch_tokens):
            n = min(batch_tokens, steps - c0)
            t0 = fill_n + c0
            if device_gen:
                q = synth.gpu_queries(w, t0, n, layer)
                k = synth.gpu_kv(w, "key", t0, n, layer, token_major=True)
                v = synth.gpu_kv(w, "value", t0, n, layer, token_major=True)
            else:
                q = torch_from_host(synth.host_queries(w, t0, n, layer))
                k = torch_from_host(synth.host_kv(w, "key", t0, n, layer, token_major=True))
                v = torch_from_host(synth.host_kv(w, "value", t0, n, layer, token_major=True))
            for i in range(n):
                he.step(q[i], k[i], v[i], out)
                evicted[c0 + i] = he.last_evicted()
                if c0 + i in out_steps:
                    outs[c0 + i] = out.cpu().numpy().copy()
        prof = he.profile_stop() if profile else None
        state = he.state() if read_state else None
        if read_state:
            state = state + (he.scores() if decay > 0.0 else None,
                             he.vscales() if v_int8 else None)
        return GpuRun(evicted, outs, state, prof)
    finally:
        he.close()


@dataclass
class OracleRun:
    evicted: np.ndarray      # [steps]
    outs: np.ndarray         # [len(out_steps)][G][D] float64
    codes: np.ndarray
    K: np.ndarray
    V: np.ndarray
    occupancy: int
    score: np.ndarray | None = None  # per-slot scores (score memory only)
    Vq: np.ndarray | None = None     # int8 value cache: rows ...
    Vs: np.ndarray | None = None     # ... and scales


def run_oracle_unit(w: synth.Workload, b: int, j: int, fill_n: int, steps: int, out_steps=(),
                    layer: int = 0, threshold: float = 0.0, decay: float = 0.0,
                    v_int8: bool = False, chunk: int = 1) -> OracleRun:
    o = oracle.load()
    W = o.projection(w.projection_seed(layer), w.head_dim, w.bits, w.dtype)
    Kin = synth.host_unit_kv(w, "key", b, j, 0, fill_n, layer)
    Vin = synth.host_unit_kv(w, "value", b, j, 0, fill_n, layer)
    if chunk > 1:
        st = o.unit_fill_chunk(W, w.budget, chunk, Kin, Vin, tau=threshold)
    else:
        st = o.unit_fill(W, w.budget, Kin, Vin, tau=threshold, memory=decay > 0.0, vq=v_int8)
    q = synth.host_unit_queries(w, b, j, fill_n, steps, layer)
    k = synth.host_unit_kv(w, "key", b, j, fill_n, steps, layer)
    v = synth.host_unit_kv(w, "value", b, j, fill_n, steps, layer)
    want = np.zeros(steps, np.uint8)
    for s in out_steps:
        want[s] = 1
    r = o.unit_stream(st, q, k, v, want_out=want, decay=decay)
    return OracleRun(r["evicted"], r["out"], st.codes, st.K, st.V, st.occupancy, st.score,
                     st.Vq, st.Vs)


def run_oracle_units(w, units, fill_n, steps, out_steps=(), layer=0, threads=8,
                     threshold: float = 0.0, decay: float = 0.0, v_int8: bool = False,
                     chunk: int = 1):
    """Oracle over several (b, j) units in parallel threads (ctypes releases the GIL)."""
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = {u: ex.submit(run_oracle_unit, w, u[0], u[1], fill_n, steps, out_steps, layer,
                             threshold, decay, v_int8, chunk)
                for u in units}
        return {u: f.result() for u, f in futs.items()}


def compare(w: synth.Workload, g: GpuRun, orc: dict, out_steps=(), check_state: bool = False):
    """Bit-exact evictions, outputs within tolerance, optional cache state."""
    out_steps = sorted(out_steps)
    worst_max, worst_mean = 0.0, 0.0
    for (b, j), r in orc.items():
        ge = g.evicted[:, b, j]
        if not np.array_equal(ge, r.evicted):
            bad = np.nonzero(ge != r.evicted)[0]
            raise AssertionError(f"unit ({b},{j}): evictions differ first at step {bad[0]}: "
                                 f"gpu {ge[bad[0]]} oracle {r.evicted[bad[0]]} "
                                 f"({len(bad)} of {len(ge)} steps differ)")
        for i, s in enumerate(out_steps):
            got = g.outs[s][b, j * w.group:(j + 1) * w.group].astype(np.float64)
            err = np.abs(got - r.outs[i])
            worst_max = max(worst_max, float(err.max()))
            worst_mean = max(worst_mean, float(err.mean()))
        if check_state:
            K, V, codes, occ = g.state[:4]
            assert occ == r.occupancy
            assert np.array_equal(codes[b, j].astype(np.uint64), r.codes), f"codes ({b},{j})"
            assert np.array_equal(K[b, j], r.K), f"K ({b},{j})"
            if r.Vq is not None:  # int8 value cache: rows and scales, exactly
                assert np.array_equal(V[b, j], r.Vq), f"int8 V ({b},{j})"
                assert np.array_equal(g.state[5][b, j], r.Vs), f"value scales ({b},{j})"
            else:
                assert np.array_equal(V[b, j], r.V), f"V ({b},{j})"
    assert worst_max <= MAX_ABS_TOL, f"max-abs error {worst_max}"
    assert worst_mean <= MEAN_ABS_TOL, f"mean-abs error {worst_mean}"
    return worst_max, worst_mean
