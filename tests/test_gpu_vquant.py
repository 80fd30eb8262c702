"""GPU parity of the quantised value cache, both byte formats:
* int8 (v_format HE_VFMT_INT8): q = v / s rounded half to even with
  s = max |v| / 127, attended as q * s;
* fp8 (v_format HE_VFMT_FP8): c = the E4M3 value nearest to v / s (ties to
  the even mantissa) with s = max |v| / 448, attended as c * s.
Keys, codes and evictions are those of the method.

The stored rows and scales are compared with the CPU oracle bit for bit (the
quantisation is one fp32 division and one rounding on both sides), evictions
bit for bit, outputs within the attention tolerance against fp64 attention
over the identical stored values."""
import numpy as np
import pytest

import oracle
import synth
from gpu_harness import (MAX_ABS_TOL, MEAN_ABS_TOL, compare, make_handle, run_gpu,
                         run_oracle_units, torch_from_host)

pytestmark = pytest.mark.gpu


def small(name, **kw):
    return synth.WORKLOADS[name].with_(**kw)


FORMATS = ["int8", "fp8"]


def _stream(w, fill_n, steps, out_every, fmt, units=None, **opt):
    out_steps = sorted(set(range(0, steps, out_every)) | {steps - 1})
    g = run_gpu(w, fill_n, steps, out_steps, read_state=True, v_format=fmt, **opt)
    if units is None:
        units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    orc = run_oracle_units(w, units, fill_n, steps, out_steps, v_format=fmt, **opt)
    return compare(w, g, orc, out_steps, check_state=True)


@pytest.mark.parametrize("fmt", FORMATS)
def test_fill_quantises_exactly(fmt):
    w = small("llama8b_b8", batch=2, budget=200, prompt=400, decode=4)
    g = run_gpu(w, 150, 0, (), read_state=True, v_format=fmt)
    o = oracle.load()
    V = synth.host_kv(w, "value", 0, 150)
    for b in range(w.batch):
        for j in range(w.kv_heads):
            q, sc = o.quantize_rows(V[b, j], fmt)
            assert np.array_equal(g.state[1][b, j, :150], q)
            assert np.array_equal(g.state[5][b, j, :150], sc)


def _edge_rows(rng, n, D):
    """bf16 value rows whose fp8 codes hit the format's edges: row maximum 448
    (so s = 1 and v / s = v exactly), E4M3 midpoints (ties to the even
    mantissa), subnormals and the midpoint below the smallest one, negative
    values that round to -0, exact zeros of both signs, and random magnitudes
    from 2^-14 to 2^8 of either sign."""
    from test_gpu_evicted_dominant import bf16_bits
    edges = [448.0, -448.0, 1.0625, -1.1875, 2.0 ** -10, -(2.0 ** -10), 1.5 * 2.0 ** -9,
             2.0 ** -11, -(2.0 ** -12), 0.0, -0.0, 0.875 * 2.0 ** -6, 2.0 ** -6, 232.0, 240.0,
             -424.0, 3.0 * 2.0 ** -10, 5.0 * 2.0 ** -10]
    rows = np.sign(rng.standard_normal((n, D))) * np.exp2(rng.uniform(-14, 8, (n, D)))
    for i in range(n):
        k = rng.integers(0, len(edges))
        idx = rng.permutation(D)[:len(edges)]
        rows[i, idx] = np.roll(edges, k)
        rows[i, rng.integers(0, D)] = 448.0 if i % 2 else -448.0
    out = bf16_bits(rows)
    # (the exact zeros keep their sign through the bf16 bit patterns)
    return out


def test_fp8_edge_rows_bit_exact():
    """fp8 codes on the format's edges, from the fill kernel and from the step
    (the new token's row written by the merge), against the oracle's E4M3
    rounding: every byte and every scale."""
    import torch
    w = small("llama8b_b8", batch=1, heads=4, kv_heads=1, budget=128, prompt=256)
    D = w.head_dim
    rng = np.random.default_rng(8)
    K = synth.host_kv(w, "key", 0, w.budget)
    V = _edge_rows(rng, w.budget, D)[None, None]
    o = oracle.load()
    he = make_handle(w, v_format="fp8")
    try:
        he.fill(torch_from_host(K), torch_from_host(V))
        st = he.state()
        q, sc = o.quantize_rows(V[0, 0], "fp8")
        assert np.array_equal(st[1][0, 0], q)
        assert np.array_equal(he.vscales()[0, 0], sc)
        vnew = _edge_rows(rng, 6, D)
        qs = synth.host_queries(w, w.budget, 6)
        ks = synth.host_kv(w, "key", w.budget, 6, token_major=True)
        for t in range(6):
            he.step(torch_from_host(qs[t]), torch_from_host(ks[t]),
                    torch_from_host(vnew[t][None, None]))
            slot = int(he.last_evicted()[0, 0])
            st = he.state()
            q1, s1 = o.quantize_rows(vnew[t][None], "fp8")
            assert np.array_equal(st[1][0, 0, slot], q1[0]), t
            assert he.vscales()[0, 0, slot] == s1[0], t
    finally:
        he.close()


@pytest.mark.parametrize("fmt", FORMATS)
def test_llama_shape_stream(fmt):
    """32/8 heads, D 128, budget 512 (several tiles, ragged fills), every unit."""
    w = small("llama8b_b8", batch=2, budget=512, prompt=1024, decode=32)
    _stream(w, 500, 80, 17, fmt)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("G,D", [(1, 128), (2, 64), (8, 128), (8, 64)])
def test_group_sizes_and_dims(G, D, fmt):
    w = small("llama8b_b8", batch=2, heads=4 * G, kv_heads=4, head_dim=D, budget=200,
              prompt=400, decode=8, bits=32)
    _stream(w, w.budget, 60, 11, fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_with_threshold_and_score_memory(fmt):
    w = small("llama8b_b8", batch=1, budget=333, prompt=700, decode=8)
    _stream(w, 320, 70, 13, fmt, threshold=0.4, decay=0.5)


@pytest.mark.parametrize("fmt", FORMATS)
def test_many_ctas_per_unit(fmt):
    w = small("long_128k", batch=1, heads=4, kv_heads=1, budget=20000, prompt=40000, decode=4)
    _stream(w, w.budget, 12, 5, fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_dominant_evicted_slot_is_recomputed(fmt):
    """The evicted slot carries most of its partial's mass: the exact recompute
    reads the byte rows; the output still equals the oracle's."""
    import torch
    from test_gpu_evicted_dominant import bf16_bits, to_f64
    bits = 16
    w = small("llama8b_b8", batch=1, heads=4, kv_heads=1, budget=256, bits=bits, prompt=512)
    D, B, G = w.head_dim, w.budget, w.group
    o = oracle.load()
    rng = np.random.default_rng(5)
    W = o.projection(w.projection_seed(), D, bits, "bf16")
    Wf = to_f64(W)
    q0 = to_f64(bf16_bits(rng.standard_normal(D)))
    s = np.sign(Wf.T @ q0)
    P = np.eye(D) - np.outer(q0, q0) / (q0 @ q0)
    A = (P @ Wf).T
    alpha = 30.0 * np.sqrt(D) / (q0 @ q0) / np.log2(np.e)
    r = A.T @ np.linalg.solve(A @ A.T, -alpha * (Wf.T @ q0) - s * 40.0)
    K = bf16_bits(rng.standard_normal((B, D)) * 0.5)
    V = bf16_bits(rng.standard_normal((B, D)))
    slot = 77
    K[slot] = bf16_bits(alpha * q0 + r)
    q = np.broadcast_to(bf16_bits(q0), (G, D)).copy()
    knew, vnew = bf16_bits(rng.standard_normal(D)), bf16_bits(rng.standard_normal(D))
    st = o.unit_fill(W, B, K, V, vq=fmt)
    r_or = o.unit_stream(st, q[None], knew[None], vnew[None])
    assert r_or["evicted"].tolist() == [slot]
    he = make_handle(w, v_format=fmt)
    try:
        he.fill(torch_from_host(K[None, None]), torch_from_host(V[None, None]))
        out = he.step(torch_from_host(q[None]), torch_from_host(knew[None, None]),
                      torch_from_host(vnew[None, None]))
        assert he.last_evicted().tolist() == [[slot]]
        got = out.cpu().numpy()[0].astype(np.float64)
        assert he.recompute_count == 1
    finally:
        he.close()
    err = np.abs(got - r_or["out"][0])
    assert err.max() <= MAX_ABS_TOL and err.mean() <= MEAN_ABS_TOL, (err.max(), err.mean())


@pytest.mark.parametrize("fmt", FORMATS)
def test_more_units_than_sms(fmt):
    """Batch 40 x 8 KV heads = 320 units: the merge CTAs take several units
    each; every unit's rows, scales and evictions are checked."""
    w = small("serving_b64", batch=40, budget=96, prompt=300, decode=8)
    _stream(w, 90, 40, 13, fmt)


@pytest.mark.slow
@pytest.mark.parametrize("fmt", FORMATS)
def test_full_llama8b_b8_sampled(fmt):
    """The Llama-3-8B-shaped layer at full size (batch 8, 32/8 heads, budget
    4096) in the launch configuration the benchmark times (296 stream CTAs,
    three ring stages, the two-group split): 48 streamed steps; sampled units'
    evictions, outputs and final byte rows and scales against the oracle."""
    w = synth.WORKLOADS["llama8b_b8"]
    steps = 48
    out_steps = [0, 23, 47]
    g = run_gpu(w, w.budget, steps, out_steps, read_state=True, device_gen=True, v_format=fmt)
    units = [(0, 0), (3, 5), (7, 7)]
    orc = run_oracle_units(w, units, w.budget, steps, out_steps, v_format=fmt)
    compare(w, g, orc, out_steps, check_state=True)


@pytest.mark.slow
def test_full_32layer_fp8_sampled_layers():
    """The 32-layer workload's layer shape (batch 16, budget 9728) with fp8
    values: 40 steps of layers 0 and 31 on sampled units."""
    w = synth.WORKLOADS["llama8b_32layer"]
    steps = 40
    out_steps = [0, 39]
    for layer in (0, 31):
        g = run_gpu(w, w.budget, steps, out_steps, layer=layer, device_gen=True,
                    v_format="fp8")
        orc = run_oracle_units(w, [(0, 0), (15, 7)], w.budget, steps, out_steps, layer=layer,
                               v_format="fp8")
        compare(w, g, orc, out_steps)
