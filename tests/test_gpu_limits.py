"""The largest shapes the library accepts, at sizes that still fit one GPU
comfortably: the most (batch, KV head) units (2^16, more units than any grid
dimension of one unit per CTA would want, and several units per merge CTA),
and a unit of 2^22 slots (tile coordinates far into the cache).  Evictions,
the cache and outputs against the oracle on sampled units."""
import numpy as np
import pytest

import synth
from gpu_harness import compare, run_gpu, run_oracle_units

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_pre_attention_decode_b300 as he
    he.lib()


@pytest.mark.parametrize("engine", ["pipeline", "fused"])
def test_most_units(engine):
    """batch 8192 x 8 KV heads = 65536 units (the limit), G = 1, D = 64,
    8-bit codes, budget 3: appends, then an eviction on every step."""
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=8192, heads=8, kv_heads=8, head_dim=64,
                                            bits=8, budget=3, prompt=16)
    steps = 6
    out_steps = [0, 5]
    g = run_gpu(w, 2, steps, out_steps, read_state=True, device_gen=True, engine=engine)
    units = [(0, 0), (1, 5), (4095, 3), (4096, 0), (8191, 7)]
    orc = run_oracle_units(w, units, 2, steps, out_steps)
    compare(w, g, orc, out_steps, check_state=True)
    assert (g.evicted[steps - 1] >= 0).all()


def test_long_unit():
    """One unit of 2^22 slots (G = 4, D = 64, 16-bit codes): 65536 tiles."""
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=1, heads=4, kv_heads=1, head_dim=64, bits=16,
                                            budget=1 << 22, prompt=(1 << 22) + 16)
    steps = 3
    out_steps = [0, 2]
    g = run_gpu(w, w.budget, steps, out_steps, device_gen=True)
    orc = run_oracle_units(w, [(0, 0)], w.budget, steps, out_steps)
    compare(w, g, orc, out_steps)


def test_median_thresholds_in_several_scratch_groups():
    """Per-bit medians of 17 units of 2^18 filled keys at 64-bit codes: the
    fill's projection scratch (64 x 2^18 floats per unit, 1 GiB at most at a
    time) takes two groups of units.  The thresholds of a unit of each group
    and its codes against the oracle."""
    import oracle
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=17, heads=4, kv_heads=1, bits=64,
                                            budget=1 << 18, prompt=(1 << 18) + 8)
    g = run_gpu(w, w.budget, 0, (), read_state=True, device_gen=True, threshold="median")
    o = oracle.load()
    W = o.projection(w.projection_seed(), w.head_dim, w.bits, w.dtype)
    for b in (0, 16):
        K = synth.host_unit_kv(w, "key", b, 0, 0, w.budget)
        tv = o.median_thresholds(K, W)
        assert np.array_equal(g.state[6][b, 0], tv), b
        assert np.array_equal(g.state[2][b, 0, :4096].astype(np.uint64), o.code(K[:4096], W, tv))
