"""GPU parity of the two eviction options: the binarisation threshold tau (bit j
= projection_j > tau; the method section names the threshold as a design
choice) and per-slot score memory gamma (A = fmaf(gamma, A, d) at every
evicting step, the largest A evicted, a written slot restarting at 0).

Codes, evictions and scores are compared bit for bit with the CPU oracle (both
sides take every decision in fp32 with the same fused multiply-adds); outputs
within the attention tolerance."""
import numpy as np
import pytest

import oracle
import synth
from gpu_harness import (compare, host_from_torch, make_handle, run_gpu, run_oracle_units,
                         torch_from_host)

pytestmark = pytest.mark.gpu


def small(name, **kw):
    return synth.WORKLOADS[name].with_(**kw)


@pytest.mark.parametrize("dtype,D,bits", [("bf16", 128, 32), ("bf16", 64, 8), ("fp32", 128, 64),
                                          ("fp32", 64, 16)])
@pytest.mark.parametrize("tau", [0.75, -1.5, 3.0])
def test_codes_with_threshold(dtype, D, bits, tau):
    import torch
    w = small("llama8b_b8", head_dim=D, bits=bits, dtype=dtype, batch=1, budget=64)
    o = oracle.load()
    W = o.projection(w.projection_seed(), D, bits, dtype)
    x = synth.host_kv(w, "key", 0, 300)[0].reshape(-1, D)
    he = make_handle(w, threshold=tau)
    try:
        codes = torch.empty(x.shape[0], dtype={8: torch.uint8, 16: torch.int16, 32: torch.int32,
                                               64: torch.int64}[bits], device="cuda")
        from lsh_pre_attention_decode_b300 import he_codes
        he_codes(he.h, torch_from_host(x), x.shape[0], codes)
        got = host_from_torch(codes).view({8: np.uint8, 16: np.uint16, 32: np.uint32,
                                           64: np.uint64}[bits]).astype(np.uint64)
    finally:
        he.close()
    want = o.code(x, W, tau)
    assert np.array_equal(got, want)
    # the threshold changes codes (the case is not vacuous)
    assert not np.array_equal(want, o.code(x, W, 0.0))


def _stream(w, fill_n, steps, out_every, units=None, threshold=0.0, decay=0.0):
    out_steps = sorted(set(range(0, steps, out_every)) | {steps - 1})
    g = run_gpu(w, fill_n, steps, out_steps, read_state=True, threshold=threshold, decay=decay)
    if units is None:
        units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    orc = run_oracle_units(w, units, fill_n, steps, out_steps, threshold=threshold, decay=decay)
    compare(w, g, orc, out_steps, check_state=True)
    if decay > 0.0:
        scores = g.state[4]
        for (b, j), r in orc.items():
            assert np.array_equal(scores[b, j], r.score), f"scores of unit ({b},{j})"
    return g, orc


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_stream_with_threshold(dtype):
    w = small("llama8b_b8", batch=2, budget=300, prompt=600, decode=8, dtype=dtype)
    _stream(w, w.budget, 70, 13, threshold=0.6)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("decay", [0.5, 1.0])
def test_stream_with_score_memory(dtype, decay):
    """Full cache, appends first (fill below the budget), ragged budget."""
    w = small("llama8b_b8", batch=2, budget=333, prompt=700, decode=8, dtype=dtype)
    g, orc = _stream(w, 320, 90, 17, decay=decay)
    # the memory changes the evictions (the case is not vacuous)
    ref = run_oracle_units(w, [(0, 0)], 320, 90)
    assert not np.array_equal(ref[(0, 0)].evicted, orc[(0, 0)].evicted)


def test_score_memory_chunked_scan_and_threshold():
    """A budget above one scan chunk of the codes/eviction kernel (several CTAs
    update one unit's scores), with a threshold and memory together."""
    w = small("llama8b_b8", batch=1, budget=9000, prompt=18000, decode=4)
    _stream(w, w.budget, 24, 7, units=[(0, 0), (0, 3), (0, 7)], threshold=-0.4, decay=0.75)


def test_memory_zero_equals_the_method():
    """decay 0 allocates no scores and takes the method's path: identical to a
    default handle."""
    w = small("llama8b_b8", batch=2, budget=200, prompt=400, decode=4)
    a = run_gpu(w, w.budget, 40, [0, 39], read_state=True, decay=0.0)
    b = run_gpu(w, w.budget, 40, [0, 39], read_state=True)
    assert np.array_equal(a.evicted, b.evicted)
    for s in (0, 39):
        assert np.array_equal(a.outs[s], b.outs[s])


@pytest.mark.slow
def test_score_memory_full_llama8b_b8_sampled():
    """Score memory (gamma 0.5, the benchmark's option) on the Llama-3-8B-shaped
    layer at full size (batch 8, budget 4096, the benchmark's launch
    configuration): 48 steps' evictions and outputs, the final cache and every
    slot's score of sampled units."""
    w = synth.WORKLOADS["llama8b_b8"]
    steps = 48
    out_steps = [0, 23, 47]
    g = run_gpu(w, w.budget, steps, out_steps, read_state=True, device_gen=True, decay=0.5)
    units = [(0, 0), (3, 5), (7, 7)]
    orc = run_oracle_units(w, units, w.budget, steps, out_steps, decay=0.5)
    compare(w, g, orc, out_steps, check_state=True)
    scores = g.state[4]
    for (b, j), r in orc.items():
        assert np.array_equal(scores[b, j], r.score), f"scores of unit ({b},{j})"
    # the memory changes the evictions (the case is not vacuous)
    ref = run_oracle_units(w, [(0, 0)], w.budget, steps)
    assert not np.array_equal(ref[(0, 0)].evicted, orc[(0, 0)].evicted)
