"""GPU parity of the per-bit median thresholds (tau_mode HE_TAU_MEDIAN): the
binarisation threshold of bit j, per (batch, KV head), is the lower median of
the projections of that unit's filled keys onto column j of W (the method
section names the binarisation threshold as a design choice; this is the
per-bit reading that splits the cached keys in half), fixed until the next
fill.

The thresholds, codes and evictions are compared with the CPU oracle bit for
bit (both sides form the projections with the same fp32 fused multiply-add
chains and take the same order statistic), outputs within the attention
tolerance."""
import numpy as np
import pytest

import oracle
import synth
from gpu_harness import compare, make_handle, run_gpu, run_oracle_units, torch_from_host

pytestmark = pytest.mark.gpu


def small(name, **kw):
    return synth.WORKLOADS[name].with_(**kw)


@pytest.mark.parametrize("dtype,D,bits,budget,fill", [
    ("bf16", 128, 32, 512, 500), ("bf16", 128, 64, 300, 300), ("bf16", 64, 8, 200, 199),
    ("bf16", 128, 16, 1000, 999), ("bf16", 128, 32, 64, 1), ("bf16", 128, 32, 64, 2),
    ("fp32", 128, 32, 256, 255), ("fp32", 64, 64, 100, 100)])
def test_fill_thresholds_and_codes(dtype, D, bits, budget, fill):
    """The thresholds and the filled keys' codes, every unit; each bit set in
    floor(n / 2) of the keys where the projections are distinct."""
    w = small("llama8b_b8", batch=2, head_dim=D, bits=bits, dtype=dtype, budget=budget,
              prompt=2 * budget)
    g = run_gpu(w, fill, 0, (), read_state=True, threshold="median")
    o = oracle.load()
    W = o.projection(w.projection_seed(), D, bits, dtype)
    codes, tv = g.state[2], g.state[6]
    nonzero = 0
    for b in range(w.batch):
        for j in range(w.kv_heads):
            K = synth.host_unit_kv(w, "key", b, j, 0, fill)
            want = o.median_thresholds(K, W)
            assert np.array_equal(tv[b, j], want), (b, j)
            c = o.code(K, W, want)
            assert np.array_equal(codes[b, j, :fill].astype(np.uint64), c), (b, j)
            nonzero += int(np.count_nonzero(want))
            for bit in range(bits):
                ones = int(sum((int(x) >> bit) & 1 for x in c))
                assert ones <= fill // 2
    if fill > 1:
        assert nonzero > 0  # (the thresholds are not the sign test's zeros)


def _stream(w, fill_n, steps, out_every, **opt):
    out_steps = sorted(set(range(0, steps, out_every)) | {steps - 1})
    g = run_gpu(w, fill_n, steps, out_steps, read_state=True, threshold="median", **opt)
    units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    orc = run_oracle_units(w, units, fill_n, steps, out_steps, threshold="median",
                           **{k: v for k, v in opt.items() if k != "engine"})
    compare(w, g, orc, out_steps, check_state=True)
    return g, orc


@pytest.mark.parametrize("case,shape,fill,steps,opt", [
    ("llama shape, ragged", dict(batch=2, budget=512, prompt=1024), 500, 80, {}),
    ("score memory", dict(batch=1, budget=333, prompt=700), 320, 70, {"decay": 0.5}),
    ("fp8 values", dict(batch=2, budget=300, prompt=600), 300, 60, {"v_format": "fp8"}),
    ("int8 values", dict(batch=1, budget=300, prompt=600), 300, 40, {"v_format": "int8"}),
    ("chunks of 8", dict(batch=2, budget=480, prompt=960), 480, 60, {"chunk": 8}),
    ("G = 8, D = 64", dict(batch=2, heads=64, head_dim=64, bits=16, budget=200, prompt=400),
     200, 40, {}),
    ("fp32", dict(batch=2, budget=256, prompt=512, dtype="fp32"), 256, 40, {}),
    ("single-kernel engine", dict(batch=2, budget=512, prompt=1024), 512, 60,
     {"engine": "fused"}),
    ("empty fill: zeros, appends", dict(batch=1, budget=64, prompt=200), 0, 100, {}),
], ids=lambda x: x if isinstance(x, str) else "")
def test_stream_with_median_thresholds(case, shape, fill, steps, opt):
    w = small("llama8b_b8", **shape)
    _stream(w, fill, steps, 13, **opt)


def test_median_changes_evictions():
    """The per-bit medians change the evictions against the sign test on the
    synthetic keys (outlier channels shift the projections): not vacuous."""
    w = small("llama8b_b8", batch=1, budget=256, prompt=512)
    a = run_oracle_units(w, [(0, 0)], 256, 60, threshold="median")
    b = run_oracle_units(w, [(0, 0)], 256, 60)
    assert not np.array_equal(a[(0, 0)].evicted, b[(0, 0)].evicted)


def test_codes_entry_point_rejects_median_handles():
    """he_codes codes rows of no unit: a median handle's thresholds are per
    unit, so the call is refused; the scalar handle's is not."""
    import torch
    from lsh_pre_attention_decode_b300 import HashEvictError, he_codes
    w = small("llama8b_b8", batch=1, budget=64)
    x = torch.zeros((4, w.head_dim), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(4, dtype=torch.int32, device="cuda")
    with make_handle(w, threshold="median") as he:
        with pytest.raises(HashEvictError):
            he_codes(he.h, x, 4, c)
    with make_handle(w) as he:
        he_codes(he.h, x, 4, c)


def test_refill_recomputes_thresholds():
    """A second fill sets the thresholds from its own keys."""
    w = small("llama8b_b8", batch=1, budget=128, prompt=512)
    o = oracle.load()
    W = o.projection(w.projection_seed(), w.head_dim, w.bits, w.dtype)
    with make_handle(w, threshold="median") as he:
        for t0 in (0, 200):
            K = synth.host_kv(w, "key", t0, 128)
            he.fill(torch_from_host(K), torch_from_host(synth.host_kv(w, "value", t0, 128)))
            for j in range(w.kv_heads):
                assert np.array_equal(he.thresholds()[0, j], o.median_thresholds(K[0, j], W))


@pytest.mark.slow
def test_full_llama8b_b8_sampled():
    """Per-bit median thresholds on the Llama-3-8B-shaped layer at full size
    (batch 8, budget 4096, the benchmark's launch configuration): the
    thresholds, 48 steps' evictions and outputs, and the final cache of
    sampled units."""
    w = synth.WORKLOADS["llama8b_b8"]
    steps = 48
    out_steps = [0, 23, 47]
    g = run_gpu(w, w.budget, steps, out_steps, read_state=True, device_gen=True,
                threshold="median")
    units = [(0, 0), (3, 5), (7, 7)]
    orc = run_oracle_units(w, units, w.budget, steps, out_steps, threshold="median")
    compare(w, g, orc, out_steps, check_state=True)
