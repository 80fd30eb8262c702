"""Run by test_gpu_debug_build in a process of its own: the parity cases below
against the bounds-checked build of the library (every computed global access
of the step kernels checked; a failed check is reported as HE_EDEVICE)."""
import sys

import lsh_pre_attention_decode_b300._binding as binding
from lsh_pre_attention_decode_b300 import _build

binding.LIB = _build.DEBUG_LIB  # before the library is first loaded

import synth  # noqa: E402
from gpu_harness import compare, run_gpu, run_oracle_units  # noqa: E402


def case(w, fill_n, steps, units, engine="pipeline", **kw):
    out_steps = sorted({0, steps // 2, steps - 1})
    g = run_gpu(w, fill_n, steps, out_steps, read_state=True, engine=engine, **kw)
    orc = run_oracle_units(w, units, fill_n, steps, out_steps, **kw)
    compare(w, g, orc, out_steps, check_state=True)


def noalloc_case():
    """The allocation-free attention entry point (same stream kernel) on the
    cache the step leaves, against the step's own output.  A failed bounds
    check inside its kernels sets the scratch array's error word, which turns
    the whole output into NaN: the finiteness check below catches it."""
    import torch
    from gpu_harness import MAX_ABS_TOL, MEAN_ABS_TOL, make_handle, torch_from_host
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=2, budget=300, prompt=600)
    he = make_handle(w)
    try:
        he.fill(torch_from_host(synth.host_kv(w, "key", 0, w.budget)),
                torch_from_host(synth.host_kv(w, "value", 0, w.budget)))
        q = torch_from_host(synth.host_queries(w, w.budget, 1))[0]
        k = torch_from_host(synth.host_kv(w, "key", w.budget, 1, token_major=True))[0]
        v = torch_from_host(synth.host_kv(w, "value", w.budget, 1, token_major=True))[0]
        ref = he.step(q, k, v)
        K, V, _, occ = he.state()
        out = torch.full_like(ref, float("nan"))
        binding.he_attend_noalloc(w.batch, w.heads, w.kv_heads, w.head_dim, w.budget, occ,
                                  torch_from_host(K), torch_from_host(V), q, out)
        torch.cuda.synchronize()
        err = (out - ref).abs()
        assert torch.isfinite(out).all()
        assert err.max().item() <= MAX_ABS_TOL and err.mean().item() <= MEAN_ABS_TOL
        he.last_evicted()  # HE_EDEVICE here if a check of the step's own kernels failed
    finally:
        he.close()


def main():
    base = synth.WORKLOADS["llama8b_b8"]
    cases = [
        ("ragged budget, appends", base.with_(batch=2, budget=333, prompt=700), 300, 40, {}),
        ("units of many tiles", base.with_(batch=2, budget=3000, prompt=3100), 3000, 6, {}),
        ("chunk eviction", base.with_(batch=2, budget=480, prompt=960), 480, 40, {"chunk": 8}),
        ("int8 values", base.with_(batch=2, budget=300, prompt=600), 300, 20, {"v_format": "int8"}),
        ("fp8 values", base.with_(batch=2, budget=300, prompt=600), 300, 20, {"v_format": "fp8"}),
        ("score memory", base.with_(batch=2, budget=333, prompt=700), 320, 30, {"decay": 0.5}),
        ("median thresholds", base.with_(batch=2, budget=333, prompt=700), 320, 30,
         {"threshold": "median"}),
        ("G = 8, D = 64", base.with_(batch=2, heads=64, head_dim=64, bits=16, budget=200,
                                     prompt=400), 200, 20, {}),
        ("single-kernel engine", base.with_(batch=2, budget=3000, prompt=3100), 2990, 20,
         {"engine": "fused"}),
    ]
    for name, w, fill_n, steps, kw in cases:
        units = [(b, j) for b in range(w.batch) for j in (0, w.kv_heads - 1)]
        case(w, fill_n, steps, units, **kw)
        print("ok", name, flush=True)
    noalloc_case()
    print("ok allocation-free attention", flush=True)
    assert binding.lib()._name == _build.DEBUG_LIB


if __name__ == "__main__":
    main()
    sys.exit(0)
