"""GPU parity of the int8 value cache (v_format HE_VFMT_INT8): value rows stored
as q = v / s rounded half to even with s = max |v| / 127, attended as q * s;
keys, codes and evictions are those of the method.

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


def _stream(w, fill_n, steps, out_every, units=None, **opt):
    out_steps = sorted(set(range(0, steps, out_every)) | {steps - 1})
    g = run_gpu(w, fill_n, steps, out_steps, read_state=True, v_int8=True, **opt)
    if units is None:
        units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    orc = run_oracle_units(w, units, fill_n, steps, out_steps, v_int8=True, **opt)
    return compare(w, g, orc, out_steps, check_state=True)


def test_fill_quantises_exactly():
    w = small("llama8b_b8", batch=2, budget=200, prompt=400, decode=4)
    g = run_gpu(w, 150, 0, (), read_state=True, v_int8=True)
    o = oracle.load()
    V = synth.host_kv(w, "value", 0, 150)
    for b in range(w.batch):
        for j in range(w.kv_heads):
            q, sc = o.quantize_rows(V[b, j])
            assert np.array_equal(g.state[1][b, j, :150], q)
            assert np.array_equal(g.state[5][b, j, :150], sc)


def test_llama_shape_stream():
    """32/8 heads, D 128, budget 512 (several tiles, ragged fills), every unit."""
    w = small("llama8b_b8", batch=2, budget=512, prompt=1024, decode=32)
    _stream(w, 500, 80, 17)


@pytest.mark.parametrize("G,D", [(1, 128), (2, 64), (8, 128), (8, 64)])
def test_group_sizes_and_dims(G, D):
    w = small("llama8b_b8", batch=2, heads=4 * G, kv_heads=4, head_dim=D, budget=200,
              prompt=400, decode=8, bits=32)
    _stream(w, w.budget, 60, 11)


def test_with_threshold_and_score_memory():
    w = small("llama8b_b8", batch=1, budget=333, prompt=700, decode=8)
    _stream(w, 320, 70, 13, threshold=0.4, decay=0.5)


def test_many_ctas_per_unit():
    w = small("long_128k", batch=1, heads=4, kv_heads=1, budget=20000, prompt=40000, decode=4)
    _stream(w, w.budget, 12, 5)


def test_dominant_evicted_slot_is_recomputed():
    """The evicted slot carries most of its partial's mass: the exact recompute
    reads int8 rows; the output still equals the oracle's."""
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
    st = o.unit_fill(W, B, K, V, vq=True)
    r_or = o.unit_stream(st, q[None], knew[None], vnew[None])
    assert r_or["evicted"].tolist() == [slot]
    he = make_handle(w, v_int8=True)
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


def test_more_units_than_sms():
    """Batch 40 x 8 KV heads = 320 units: the merge CTAs take several units
    each; every unit's rows, scales and evictions are checked."""
    w = small("serving_b64", batch=40, budget=96, prompt=300, decode=8)
    _stream(w, 90, 40, 13)
