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


def make_handle(w: synth.Workload, layer: int = 0, threshold=0.0, decay: float = 0.0,
                v_format: str = "elem", chunk: int = 1, engine: str = "pipeline"):
    """threshold: a float, or "median" for the per-bit median thresholds."""
    from lsh_pre_attention_decode_b300 import HashEvict
    median = threshold == "median"
    return HashEvict(w.batch, w.heads, w.kv_heads, w.head_dim, w.bits, w.budget, w.dtype,
                     seed=w.projection_seed(layer), threshold=0.0 if median else threshold,
                     decay=decay, v_format=v_format, chunk=chunk, engine=engine,
                     tau_mode="median" if median else "fixed")


def run_gpu(w: synth.Workload, fill_n: int, steps: int, out_steps=(), layer: int = 0,
            device_gen: bool = False, read_state: bool = False, batch_tokens: int = 256,
            profile: bool = False, threshold=0.0, decay: float = 0.0,
            v_format: str = "elem", chunk: int = 1, engine: str = "pipeline") -> GpuRun:
    """Fill with prompt tokens [0, fill_n), then stream tokens fill_n .. fill_n+steps-1
    (generated batch_tokens at a time).  With decay > 0 the returned state also
    holds the per-slot scores; with a quantised value cache (v_format "int8" or
    "fp8"), V holds the byte rows and the value scales follow; with threshold
    "median" the per-bit thresholds follow; chunk > 1: chunk eviction (state
    rows budget + chunk - 1)."""
    import torch
    out_steps = set(out_steps)
    he = make_handle(w, layer, threshold, decay, v_format, chunk, engine)
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
                             he.vscales() if v_format != "elem" else None,
                             he.thresholds() if threshold == "median" else None)
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
    Vq: np.ndarray | None = None     # quantised value cache: byte rows ...
    Vs: np.ndarray | None = None     # ... and scales
    tauv: np.ndarray | None = None   # per-bit median thresholds


def run_oracle_unit(w: synth.Workload, b: int, j: int, fill_n: int, steps: int, out_steps=(),
                    layer: int = 0, threshold=0.0, decay: float = 0.0,
                    v_format: str = "elem", chunk: int = 1) -> OracleRun:
    o = oracle.load()
    median = threshold == "median"
    tau = 0.0 if median else threshold
    W = o.projection(w.projection_seed(layer), w.head_dim, w.bits, w.dtype)
    Kin = synth.host_unit_kv(w, "key", b, j, 0, fill_n, layer)
    Vin = synth.host_unit_kv(w, "value", b, j, 0, fill_n, layer)
    if chunk > 1:
        st = o.unit_fill_chunk(W, w.budget, chunk, Kin, Vin, tau=tau, median=median)
    else:
        st = o.unit_fill(W, w.budget, Kin, Vin, tau=tau, memory=decay > 0.0,
                         vq=False if v_format == "elem" else v_format, median=median)
    q = synth.host_unit_queries(w, b, j, fill_n, steps, layer)
    k = synth.host_unit_kv(w, "key", b, j, fill_n, steps, layer)
    v = synth.host_unit_kv(w, "value", b, j, fill_n, steps, layer)
    want = np.zeros(steps, np.uint8)
    for s in out_steps:
        want[s] = 1
    r = o.unit_stream(st, q, k, v, want_out=want, decay=decay)
    return OracleRun(r["evicted"], r["out"], st.codes, st.K, st.V, st.occupancy, st.score,
                     st.Vq, st.Vs, st.tauv)


def run_oracle_units(w, units, fill_n, steps, out_steps=(), layer=0, threads=8,
                     threshold=0.0, decay: float = 0.0, v_format: str = "elem",
                     chunk: int = 1):
    """Oracle over several (b, j) units in parallel threads (ctypes releases the GIL)."""
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = {u: ex.submit(run_oracle_unit, w, u[0], u[1], fill_n, steps, out_steps, layer,
                             threshold, decay, v_format, chunk)
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
            if r.Vq is not None:  # quantised value cache: byte rows and scales, exactly
                assert np.array_equal(V[b, j], r.Vq), f"V bytes ({b},{j})"
                assert np.array_equal(g.state[5][b, j], r.Vs), f"value scales ({b},{j})"
            else:
                assert np.array_equal(V[b, j], r.V), f"V ({b},{j})"
            if r.tauv is not None:  # per-bit median thresholds, exactly
                assert np.array_equal(g.state[6][b, j], r.tauv), f"thresholds ({b},{j})"
    assert worst_max <= MAX_ABS_TOL, f"max-abs error {worst_max}"
    assert worst_mean <= MEAN_ABS_TOL, f"mean-abs error {worst_mean}"
    return worst_max, worst_mean


# ---------------------------------------------------------------------------
# steps issued back to back (no host synchronisation between them), as a
# serving loop and the benchmark issue them
# ---------------------------------------------------------------------------

@dataclass
class B2BRun:
    evicted: dict   # layer -> [total steps][batch][kv_heads] from the device eviction log
    outs: dict      # (layer, step) -> out [batch][heads][D] float32
    states: dict    # layer -> (K, V, codes, occupancy, vscales, scores, thresholds or None)
    tokens: list    # per layer step -> token index (the stream each layer saw)


def run_gpu_b2b(w: synth.Workload, fill_n: int, tokens: int, out_steps=(), layers: int = 1,
                graph: bool = False, replays: int = 2, warm: int = 0, threshold=0.0,
                decay: float = 0.0, v_format: str = "elem", chunk: int = 1,
                hold_ms: float = 20.0, engine: str = "pipeline") -> B2BRun:
    """Fill `layers` independent caches with prompt tokens [0, fill_n), then
    issue steps round robin over the layers (layer 0 token t, layer 1 token t,
    ...) with no host synchronisation, each step writing the slots it wrote to
    a device eviction log.

    Eager (graph=False): `tokens` tokens per layer, fill_n .. fill_n + tokens - 1.
    Graph: `warm` eager tokens per layer first, then a CUDA graph of the next
    `tokens` tokens per layer is captured and replayed `replays` times back to
    back, so each layer sees warm tokens, then its `tokens` captured tokens
    `replays` times over (the inputs of a replay are the captured ones).

    Before the first step a sleep kernel holds the stream for `hold_ms`, so that
    every launch is queued before any runs.  out_steps are indices into a
    layer's step sequence whose output is kept (each in its own buffer; in
    graph mode only those of the last replay survive, so pass those).  The
    host reads anything back only once, after the last step."""
    import ctypes
    import torch
    from lsh_pre_attention_decode_b300 import he_set_evict_log, lib
    L = layers
    U = w.batch * w.kv_heads
    n_steps = warm + tokens * replays if graph else tokens
    tok_of = ([fill_n + t for t in range(warm)] +
              [fill_n + warm + t for _ in range(replays) for t in range(tokens)]) if graph else \
        [fill_n + t for t in range(tokens)]
    out_set = set(out_steps)
    handles, logs, ins, outs, scratch = [], [], [], [], []
    he_step_raw = lib().he_step
    try:
        for layer in range(L):
            he = make_handle(w, layer, threshold, decay, v_format, chunk, engine)
            handles.append(he)
            if fill_n > 0:
                he.fill(synth.gpu_kv(w, "key", 0, fill_n, layer),
                        synth.gpu_kv(w, "value", 0, fill_n, layer))
            else:
                he.fill(None, None)
            n_in = warm + tokens if graph else tokens
            q = synth.gpu_queries(w, fill_n, n_in, layer)
            k = synth.gpu_kv(w, "key", fill_n, n_in, layer, token_major=True)
            v = synth.gpu_kv(w, "value", fill_n, n_in, layer, token_major=True)
            ins.append((q, k, v))
            log = torch.full((n_steps, U), -7, dtype=torch.int32, device="cuda")
            cnt = torch.zeros(U, dtype=torch.int32, device="cuda")
            he_set_evict_log(he.h, log, cnt, n_steps)
            logs.append((log, cnt))
            outs.append({s: torch.full((w.batch, w.heads, w.head_dim), float("nan"),
                                       dtype=torch.float32, device="cuda") for s in out_set})
            scratch.append(torch.empty((w.batch, w.heads, w.head_dim), dtype=torch.float32,
                                       device="cuda"))
        torch.cuda.synchronize()

        def issue(step_idx, inp_idx, stream_ptr):
            for layer in range(L):
                q, k, v = ins[layer]
                o = outs[layer].get(step_idx, scratch[layer])
                rc = he_step_raw(handles[layer].h, ctypes.c_void_p(q[inp_idx].data_ptr()),
                                 ctypes.c_void_p(k[inp_idx].data_ptr()),
                                 ctypes.c_void_p(v[inp_idx].data_ptr()),
                                 ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(stream_ptr))
                assert rc == 0, rc

        cur = torch.cuda.current_stream()
        cycles = int(hold_ms * 1e-3 * 2.0e9)
        if not graph:
            torch.cuda._sleep(cycles)
            for t in range(tokens):
                issue(t, t, cur.cuda_stream)
        else:
            torch.cuda._sleep(cycles)
            for t in range(warm):
                issue(t, t, cur.cuda_stream)
            g = torch.cuda.CUDAGraph()
            # capture: the output buffers of the steps of the last replay
            last0 = warm + (replays - 1) * tokens
            with torch.cuda.graph(g):
                cs = torch.cuda.current_stream().cuda_stream
                for t in range(tokens):
                    issue(last0 + t, warm + t, cs)
            torch.cuda._sleep(cycles)
            for _ in range(replays):
                g.replay()
        torch.cuda.synchronize()
        evicted, res_outs, states = {}, {}, {}
        for layer in range(L):
            log, cnt = logs[layer]
            c = cnt.cpu().numpy()
            assert (c == n_steps).all(), f"layer {layer}: {c.min()}..{c.max()} logged, {n_steps} steps"
            evicted[layer] = log.cpu().numpy().reshape(n_steps, w.batch, w.kv_heads)
            for s, o in outs[layer].items():
                res_outs[(layer, s)] = o.cpu().numpy()
            he = handles[layer]
            st = he.state()
            states[layer] = st + (he.vscales() if v_format != "elem" else None,
                                  he.scores() if decay > 0.0 else None,
                                  he.thresholds() if threshold == "median" else None)
        return B2BRun(evicted, res_outs, states, tok_of)
    finally:
        for he in handles:
            he.close()


def oracle_b2b(w: synth.Workload, units, fill_n: int, tok_of, out_steps=(), layer: int = 0,
               threshold=0.0, decay: float = 0.0, v_format: str = "elem",
               chunk: int = 1, threads: int = 8) -> dict:
    """The oracle over the token sequence tok_of (token indices, repeats
    allowed) for the given (b, j) units of one layer."""
    o = oracle.load()
    W = o.projection(w.projection_seed(layer), w.head_dim, w.bits, w.dtype)
    median = threshold == "median"
    tau = 0.0 if median else threshold
    lo, hi = min(tok_of), max(tok_of) + 1
    sel = np.asarray(tok_of) - lo
    want = np.zeros(len(tok_of), np.uint8)
    for s in out_steps:
        want[s] = 1

    def one(u):
        b, j = u
        Kin = synth.host_unit_kv(w, "key", b, j, 0, fill_n, layer)
        Vin = synth.host_unit_kv(w, "value", b, j, 0, fill_n, layer)
        if chunk > 1:
            st = o.unit_fill_chunk(W, w.budget, chunk, Kin, Vin, tau=tau, median=median)
        else:
            st = o.unit_fill(W, w.budget, Kin, Vin, tau=tau, memory=decay > 0.0,
                             vq=False if v_format == "elem" else v_format, median=median)
        q = synth.host_unit_queries(w, b, j, lo, hi - lo, layer)[sel]
        k = synth.host_unit_kv(w, "key", b, j, lo, hi - lo, layer)[sel]
        v = synth.host_unit_kv(w, "value", b, j, lo, hi - lo, layer)[sel]
        r = o.unit_stream(st, q, k, v, want_out=want, decay=decay)
        return OracleRun(r["evicted"], r["out"], st.codes, st.K, st.V, st.occupancy, st.score,
                         st.Vq, st.Vs, st.tauv)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = {u: ex.submit(one, u) for u in units}
        return {u: f.result() for u, f in futs.items()}


def compare_b2b(w: synth.Workload, g: B2BRun, layer: int, orc: dict, out_steps=()):
    """Every logged eviction bit-exact, the final cache state of each unit
    byte-exact, kept outputs within the tolerance."""
    out_steps = sorted(out_steps)
    K, V, codes, occ, vs, sc, tv = g.states[layer]
    worst_max = worst_mean = 0.0
    for (b, j), r in orc.items():
        ge = g.evicted[layer][:, b, j]
        if not np.array_equal(ge, r.evicted):
            bad = np.nonzero(ge != r.evicted)[0]
            raise AssertionError(f"layer {layer} unit ({b},{j}): evictions differ first at step "
                                 f"{bad[0]}: gpu {ge[bad[0]]} oracle {r.evicted[bad[0]]} "
                                 f"({len(bad)} of {len(ge)} steps differ)")
        assert occ == r.occupancy
        assert np.array_equal(codes[b, j].astype(np.uint64), r.codes), f"codes ({b},{j})"
        assert np.array_equal(K[b, j], r.K), f"K ({b},{j})"
        if r.Vq is not None:
            assert np.array_equal(V[b, j], r.Vq), f"V bytes ({b},{j})"
            assert np.array_equal(vs[b, j], r.Vs), f"value scales ({b},{j})"
        else:
            assert np.array_equal(V[b, j], r.V), f"V ({b},{j})"
        if r.score is not None:
            assert np.array_equal(sc[b, j], r.score), f"scores ({b},{j})"
        if r.tauv is not None:
            assert np.array_equal(tv[b, j], r.tauv), f"thresholds ({b},{j})"
        for i, s in enumerate(out_steps):
            got = g.outs[(layer, s)][b, j * w.group:(j + 1) * w.group].astype(np.float64)
            err = np.abs(got - r.outs[i])
            worst_max = max(worst_max, float(err.max()))
            worst_mean = max(worst_mean, float(err.mean()))
    assert worst_max <= MAX_ABS_TOL, f"max-abs error {worst_max}"
    assert worst_mean <= MEAN_ABS_TOL, f"mean-abs error {worst_mean}"
    return worst_max, worst_mean
