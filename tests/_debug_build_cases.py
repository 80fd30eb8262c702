"""Run by test_gpu_debug_build in a process of its own: the parity cases below
against the bounds-checked build of the library (every computed global access
of the step kernels checked; a failed check is reported as HE_EDEVICE)."""
import sys

import lsh_pre_attention_decode_b300._binding as binding
from lsh_pre_attention_decode_b300 import _build

binding.LIB = _build.DEBUG_LIB  # before the library is first loaded

import synth  # noqa: E402
from gpu_harness import compare, run_gpu, run_oracle_units  # noqa: E402


def case(w, fill_n, steps, units, **kw):
    out_steps = sorted({0, steps // 2, steps - 1})
    g = run_gpu(w, fill_n, steps, out_steps, read_state=True, **kw)
    orc = run_oracle_units(w, units, fill_n, steps, out_steps, **kw)
    compare(w, g, orc, out_steps, check_state=True)


def main():
    base = synth.WORKLOADS["llama8b_b8"]
    cases = [
        ("ragged budget, appends", base.with_(batch=2, budget=333, prompt=700), 300, 40, {}),
        ("units of many tiles", base.with_(batch=2, budget=3000, prompt=3100), 3000, 6, {}),
        ("chunk eviction", base.with_(batch=2, budget=480, prompt=960), 480, 40, {"chunk": 8}),
        ("int8 values", base.with_(batch=2, budget=300, prompt=600), 300, 20, {"v_int8": True}),
        ("score memory", base.with_(batch=2, budget=333, prompt=700), 320, 30, {"decay": 0.5}),
        ("G = 8, D = 64", base.with_(batch=2, heads=64, head_dim=64, bits=16, budget=200,
                                     prompt=400), 200, 20, {}),
    ]
    for name, w, fill_n, steps, kw in cases:
        units = [(b, j) for b in range(w.batch) for j in (0, w.kv_heads - 1)]
        case(w, fill_n, steps, units, **kw)
        print("ok", name, flush=True)
    assert binding.lib()._name == _build.DEBUG_LIB


if __name__ == "__main__":
    main()
    sys.exit(0)
