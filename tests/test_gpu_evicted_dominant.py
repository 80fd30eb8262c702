"""The evicted slot carries most of the softmax mass of its attention partial.

The bf16 step takes the evicted slot out of the attention partial that holds it;
when the slot carries more than half of that partial's mass it recomputes the
partial exactly instead of subtracting (both engines: the three-kernel pipeline
and the single fused kernel).  Here a key is built to be both the most
Hamming-dissimilar to the query (all code bits flipped: evicted) and the key
with by far the largest logit, so the exact path must run, and the result must
still equal the oracle's (which never attends to the evicted slot).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_harness import MAX_ABS_TOL, MEAN_ABS_TOL, make_handle, torch_from_host

pytestmark = pytest.mark.gpu


def bf16_bits(a):
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def to_f64(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# (bits, budget, slot): one unit of 4 tiles, and one of 375 tiles spread over
# every stream CTA, with the slot (tile 340) inside one CTA's range (32-bit
# codes there: no random key of 24000 ties the constructed distance).
@pytest.mark.parametrize("engine", ["pipeline", "fused"])
@pytest.mark.parametrize("bits,budget,slot", [(8, 256, 77), (16, 256, 77), (32, 24000, 21773)])
def test_dominant_evicted_slot_is_recomputed(bits, budget, slot, engine):
    import torch
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=1, heads=4, kv_heads=1, budget=budget,
                                            bits=bits, prompt=2 * budget)
    D, B, G = w.head_dim, w.budget, w.group
    o = oracle.load()
    rng = np.random.default_rng(bits)
    W = o.projection(w.projection_seed(), D, bits, "bf16")
    Wf = to_f64(W)
    q0 = to_f64(bf16_bits(rng.standard_normal(D)))
    # k* = alpha q0 + r, r orthogonal to q0, with every projection sign flipped
    s = np.sign(Wf.T @ q0)
    P = np.eye(D) - np.outer(q0, q0) / (q0 @ q0)
    A = (P @ Wf).T                       # [bits][D]
    alpha = 30.0 * np.sqrt(D) / (q0 @ q0) / np.log2(np.e)
    b = -alpha * (Wf.T @ q0) - s * 40.0
    r = A.T @ np.linalg.solve(A @ A.T, b)
    kstar = bf16_bits(alpha * q0 + r)
    cq = o.code(bf16_bits(q0)[None, :], W)[0]
    ck = o.code(kstar[None, :], W)[0]
    assert bin(int(cq) ^ int(ck)).count("1") == bits, "construction did not flip every bit"
    K = bf16_bits(rng.standard_normal((B, D)) * 0.5)
    V = bf16_bits(rng.standard_normal((B, D)))
    K[slot] = kstar
    q = np.broadcast_to(bf16_bits(q0), (G, D)).copy()
    knew = bf16_bits(rng.standard_normal(D))
    vnew = bf16_bits(rng.standard_normal(D))

    st = o.unit_fill(W, B, K, V)
    # the evicted key must dominate the 128 slots around it in the cache before
    # the step (a stream CTA's range holds at least one 64-slot tile)
    lo = slot // 128 * 128
    logits = (to_f64(K[lo:lo + 128]) @ q0) / np.sqrt(D)
    assert np.argmax(logits) == slot - lo and logits.max() - np.sort(logits)[-2] > 10
    r_or = o.unit_stream(st, q[None], knew[None], vnew[None])
    assert r_or["evicted"].tolist() == [slot]

    he = make_handle(w, engine=engine)
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


def test_dominant_slot_with_several_units_per_merge_cta():
    """More units than SMs (160 units of one KV head, 4 tiles each): the merge
    CTAs take several units each; one unit's evicted slot dominates its
    partial, so that CTA recomputes it while its other units merge normally."""
    import torch
    from gpu_harness import compare, run_oracle_units  # noqa: F401
    bits, budget, slot, ud = 16, 256, 77, 77
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=160, heads=4, kv_heads=1, budget=budget,
                                            bits=bits, prompt=2 * budget)
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
    b = -alpha * (Wf.T @ q0) - s * 40.0
    r = A.T @ np.linalg.solve(A @ A.T, b)
    kstar = bf16_bits(alpha * q0 + r)
    K = bf16_bits(rng.standard_normal((w.batch, 1, B, D)) * 0.5)
    V = bf16_bits(rng.standard_normal((w.batch, 1, B, D)))
    K[ud, 0, slot] = kstar
    q = bf16_bits(rng.standard_normal((w.batch, G, D)))
    q[ud] = np.broadcast_to(bf16_bits(q0), (G, D))
    knew = bf16_bits(rng.standard_normal((w.batch, 1, D)))
    vnew = bf16_bits(rng.standard_normal((w.batch, 1, D)))

    he = make_handle(w)
    try:
        he.fill(torch_from_host(K), torch_from_host(V))
        out = he.step(torch_from_host(q), torch_from_host(knew), torch_from_host(vnew))
        ev = he.last_evicted()
        got = out.cpu().numpy().astype(np.float64)
        assert he.recompute_count == 1
        state = he.state()
    finally:
        he.close()
    assert ev[ud, 0] == slot
    worst = 0.0
    for u in [0, 1, 75, 76, 77, 78, 79, 80, 159]:  # the dominant unit and its merge CTA's others
        st = o.unit_fill(W, B, K[u, 0], V[u, 0])
        r_or = o.unit_stream(st, q[u][None], knew[u, 0][None], vnew[u, 0][None])
        assert ev[u, 0] == r_or["evicted"][0], u
        err = np.abs(got[u] - r_or["out"][0])
        assert err.max() <= MAX_ABS_TOL and err.mean() <= MEAN_ABS_TOL, (u, err.max(), err.mean())
        assert np.array_equal(state[0][u, 0], st.K) and np.array_equal(state[1][u, 0], st.V), u
        worst = max(worst, float(err.max()))
