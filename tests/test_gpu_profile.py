"""The library's kernel timing mode (events between a step's kernels) must not
change what a step computes, and must report a positive time per kernel."""
import numpy as np
import pytest

import synth
from tests.gpu_harness import run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["llama8b_b8", "tiny_fp32"])
def test_timing_mode_is_transparent(name):
    w = synth.WORKLOADS[name].with_(batch=2, budget=300)
    steps = 12
    a = run_gpu(w, w.budget, steps, out_steps=range(steps), read_state=True)
    b = run_gpu(w, w.budget, steps, out_steps=range(steps), read_state=True, profile=True)
    assert np.array_equal(a.evicted, b.evicted)
    for s in range(steps):
        assert np.array_equal(a.outs[s], b.outs[s])
    for x, y in zip(a.state, b.state):
        assert np.array_equal(np.asarray(x), np.asarray(y))
    p = b.prof
    assert p["steps"] == steps
    assert p["stream_ms"] > 0 and p["step_ms"] > 0
    if w.dtype == "bf16":
        assert p["prep_ms"] > 0 and p["merge_ms"] > 0
    parts = p["stream_ms"] + p["prep_ms"] + p["merge_ms"]
    assert abs(parts - p["step_ms"]) <= 0.05 * p["step_ms"] + 0.01
