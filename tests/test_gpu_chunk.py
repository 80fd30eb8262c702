"""GPU parity of chunk eviction: the budget cut into aligned chunks of c slots,
a chunk scored by the sum of its slots' group-summed Hamming distances (the
HashEvict paper's scores, technical framework steps 3-4, taken in the contiguous
chunks of the ChunkKV page's method), new tokens staged in the c - 1 rows after
the budget, and the token that would overflow the stage evicting the
highest-scoring chunk (ties: lowest) with the staged tokens, then itself,
taking the chunk's slots.

Evictions, codes and the whole cache (staged rows included) are compared bit
for bit with the CPU oracle; outputs within the attention tolerance."""
import numpy as np
import pytest

import oracle
import synth
from gpu_harness import (MAX_ABS_TOL, MEAN_ABS_TOL, compare, make_handle, run_gpu,
                         run_oracle_units, torch_from_host)

pytestmark = pytest.mark.gpu


def small(**kw):
    return synth.WORKLOADS["llama8b_b8"].with_(**kw)


def _stream(w, fill_n, steps, out_every, chunk, threshold=0.0, units=None):
    out_steps = sorted(set(range(0, steps, out_every)) | {steps - 1})
    g = run_gpu(w, fill_n, steps, out_steps, read_state=True, chunk=chunk, threshold=threshold)
    if units is None:
        units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    orc = run_oracle_units(w, units, fill_n, steps, out_steps, chunk=chunk, threshold=threshold)
    compare(w, g, orc, out_steps, check_state=True)
    # the stream reached chunk evictions (the case is not vacuous)
    assert (g.evicted >= 0).any()
    return g, orc


@pytest.mark.parametrize("chunk", [2, 3, 8, 10, 16])
@pytest.mark.parametrize("D,bits,heads", [(128, 32, 32), (64, 8, 8), (128, 64, 64)])
def test_chunk_stream(chunk, D, bits, heads):
    """Appends below the budget, staging, several eviction cycles; ragged
    budgets (not a multiple of the 64-slot tile), G = 4, 1 and 8."""
    budget = 25 * chunk
    w = small(batch=2, heads=heads, head_dim=D, bits=bits, budget=budget, prompt=2 * budget,
              decode=8)
    _stream(w, budget - 5, 4 * chunk + 12, 3, chunk)


def test_chunk_from_empty_cache():
    """An empty cache fills by appends, then stages, then evicts chunks."""
    w = small(batch=1, budget=24, prompt=64, decode=8)
    _stream(w, 0, 60, 1, 4)


@pytest.mark.parametrize("chunk,budget", [(3, 3000), (6, 3000), (16, 3008)])
def test_chunk_many_contributors(chunk, budget):
    """Units of 47 tiles spread over every stream CTA: chunks that cross a tile
    (and a CTA's range) leave two partials."""
    w = small(batch=2, budget=budget, prompt=budget + 64, decode=8)
    units = [(0, 0), (0, 5), (1, 3), (1, 7)]
    _stream(w, budget, 3 * chunk + 4, 2, chunk, units=units)


@pytest.mark.parametrize("chunk,budget", [(3, 9000), (5, 9000), (16, 9008)])
def test_chunk_scan_split_over_ctas(chunk, budget):
    """Budgets above one prep item (whole chunks, a multiple of 16 slots): the
    chunk scores of a unit come from several CTAs."""
    w = small(batch=1, kv_heads=2, heads=8, budget=budget, prompt=budget + 64, decode=8)
    _stream(w, budget, 2 * chunk + 2, 3, chunk)


def test_chunk_with_threshold():
    w = small(batch=2, budget=120, prompt=240, decode=8)
    _stream(w, 120, 40, 5, 4, threshold=0.6)


def bf16_bits(a):
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def to_f64(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# (bits, budget, chunk, first slot): a chunk inside one tile; a chunk across
# tiles 339 and 340 of a unit of 375 tiles spread over every stream CTA.
@pytest.mark.parametrize("bits,budget,chunk,first", [(16, 256, 4, 76), (32, 24000, 6, 21756),
                                                     (32, 24000, 8, 21760)])
def test_dominant_chunk_is_recomputed(bits, budget, chunk, first):
    """Every slot of one chunk holds a key that is both the most Hamming-
    dissimilar to the query (all bits flipped, so the chunk scores the maximum)
    and far the largest logit: taking the chunk out of its partials by
    subtraction would cancel, so the exact recompute must run."""
    import torch
    w = small(batch=1, heads=4, kv_heads=1, budget=budget, bits=bits, prompt=2 * budget)
    D, B, G = w.head_dim, w.budget, w.group
    o = oracle.load()
    rng = np.random.default_rng(bits + chunk)
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
    cq = o.code(bf16_bits(q0)[None, :], W)[0]
    assert bin(int(cq) ^ int(o.code(kstar[None, :], W)[0])).count("1") == bits
    K = bf16_bits(rng.standard_normal((B, D)) * 0.5)
    V = bf16_bits(rng.standard_normal((B, D)))
    K[first:first + chunk] = kstar
    q = np.broadcast_to(bf16_bits(q0), (G, D)).copy()
    T = chunk  # c - 1 staged tokens, then the evicting one
    kn = bf16_bits(rng.standard_normal((T, D)))
    vn = bf16_bits(rng.standard_normal((T, D)))
    st = o.unit_fill_chunk(W, B, chunk, K, V)
    r_or = o.unit_stream(st, np.broadcast_to(q, (T, G, D)).copy(), kn, vn)
    assert r_or["evicted"].tolist() == [-1] * (T - 1) + [first]

    he = make_handle(w, chunk=chunk)
    try:
        he.fill(torch_from_host(K[None, None]), torch_from_host(V[None, None]))
        qt = torch_from_host(q[None])
        for t in range(T):
            out = he.step(qt, torch_from_host(kn[t][None, None]), torch_from_host(vn[t][None, None]))
        assert he.last_evicted().tolist() == [[first]]
        got = out.cpu().numpy()[0].astype(np.float64)
        assert he.recompute_count == 1
        Kg, Vg, codes, occ = he.state()
    finally:
        he.close()
    err = np.abs(got - r_or["out"][-1])
    assert err.max() <= MAX_ABS_TOL and err.mean() <= MEAN_ABS_TOL, (err.max(), err.mean())
    assert occ == st.occupancy == B
    assert np.array_equal(Kg[0, 0], st.K) and np.array_equal(Vg[0, 0], st.V)
    assert np.array_equal(codes[0, 0].astype(np.uint64), st.codes)


def test_heavy_chunk_is_subtracted():
    """A chunk that holds nearly all of its own partial's weight (97 %: one
    64-slot tile per stream CTA) but about a third of the unit's attention is
    taken out by subtraction (no recompute), and the output still matches."""
    import torch
    w = small(batch=1, heads=4, kv_heads=1, budget=4096, bits=32, prompt=8192)
    D, B, G, chunk, first = w.head_dim, w.budget, w.group, 8, 1608
    o = oracle.load()
    rng = np.random.default_rng(77)
    W = o.projection(w.projection_seed(), D, 32, "bf16")
    Wf = to_f64(W)
    q0 = to_f64(bf16_bits(rng.standard_normal(D)))
    s = np.sign(Wf.T @ q0)
    P = np.eye(D) - np.outer(q0, q0) / (q0 @ q0)
    A = (P @ Wf).T
    alpha = 8.0 * np.sqrt(D) / (q0 @ q0) / np.log2(np.e)  # base-2 logit 8: weight 256
    b = -alpha * (Wf.T @ q0) - s * 40.0
    r = A.T @ np.linalg.solve(A @ A.T, b)
    kstar = bf16_bits(alpha * q0 + r)
    K = bf16_bits(rng.standard_normal((B, D)) * 0.05)
    V = bf16_bits(rng.standard_normal((B, D)))
    K[first:first + chunk] = kstar
    q = np.broadcast_to(bf16_bits(q0), (G, D)).copy()
    kn = bf16_bits(rng.standard_normal((chunk, D)) * 0.05)
    vn = bf16_bits(rng.standard_normal((chunk, D)))
    st = o.unit_fill_chunk(W, B, chunk, K, V)
    r_or = o.unit_stream(st, np.broadcast_to(q, (chunk, G, D)).copy(), kn, vn)
    assert r_or["evicted"].tolist() == [-1] * (chunk - 1) + [first]
    # the chunk's share of its tile and of the whole cache, before the step
    lg = (to_f64(K) @ q0) / np.sqrt(D) * np.log2(np.e)
    wt = np.exp2(lg - lg.max())
    tile = wt[first // 64 * 64:first // 64 * 64 + 64]
    share_tile = wt[first:first + chunk].sum() / tile.sum()
    share_all = wt[first:first + chunk].sum() / wt.sum()
    assert share_tile > 0.9 and 0.1 < share_all < 0.6, (share_tile, share_all)

    he = make_handle(w, chunk=chunk)
    try:
        he.fill(torch_from_host(K[None, None]), torch_from_host(V[None, None]))
        qt = torch_from_host(q[None])
        for t in range(chunk):
            out = he.step(qt, torch_from_host(kn[t][None, None]), torch_from_host(vn[t][None, None]))
        assert he.last_evicted().tolist() == [[first]]
        got = out.cpu().numpy()[0].astype(np.float64)
        assert he.recompute_count == 0
    finally:
        he.close()
    err = np.abs(got - r_or["out"][-1])
    assert err.max() <= MAX_ABS_TOL and err.mean() <= MEAN_ABS_TOL, (err.max(), err.mean())


def test_chunk_full_llama8b_b8_sampled():
    """The benchmark's workload (batch 8, 32/8 heads, budget 4096) with c = 16
    in the launch configuration the benchmark times (296 stream CTAs, the
    two-group tile split): 40 steps (two and a half staging cycles) on sampled
    units: every eviction, outputs at the evicting steps, and the final cache."""
    w = synth.WORKLOADS["llama8b_b8"]
    steps = 40
    out_steps = [0, 14, 15, 16, 31, 39]
    g = run_gpu(w, w.budget, steps, out_steps, read_state=True, chunk=16, device_gen=True)
    units = [(0, 0), (3, 5), (7, 7)]
    orc = run_oracle_units(w, units, w.budget, steps, out_steps, chunk=16)
    compare(w, g, orc, out_steps, check_state=True)
    assert (g.evicted[15] >= 0).all() and (g.evicted[31] >= 0).all()
    assert (g.evicted[:15] == -1).all()


@pytest.mark.parametrize("chunk", [4, 16])
def test_chunk_more_units_than_sms(chunk):
    """Batch 40 x 8 KV heads = 320 units: the merge CTAs take several units
    each through staging and chunk evictions."""
    budget = 8 * chunk
    w = small(batch=40, budget=budget, prompt=4 * budget, decode=8)
    units = [(0, 0), (7, 3), (19, 7), (20, 0), (33, 5), (39, 7)]
    _stream(w, budget - 3, 3 * chunk + 6, 4, chunk, units=units)
