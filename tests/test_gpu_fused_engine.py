"""GPU parity of the single-kernel engine (he_cfg.engine = HE_ENGINE_FUSED): the
whole step in one kernel per decode step, a hash warp per CTA coding the
queries and scanning the CTA's own codes (HashEvict paper, technical framework
steps 1-4), the consumer warps streaming the attention, and the last CTA to
finish a (batch, KV head) unit merging it and overwriting the evicted slot
(step 5).

The same bar as the three-kernel engine: codes, distances, evictions and the
cache bit for bit against the CPU oracle, outputs within max-abs 1e-2 and
mean-abs 1e-3 of the fp64 oracle, on the shapes of the parity suite, and with
steps issued back to back or replayed from a captured graph (the device
eviction log)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_harness import (compare, compare_b2b, oracle_b2b, run_gpu, run_gpu_b2b,
                         run_oracle_units)

pytestmark = pytest.mark.gpu
FUSED = "fused"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_pre_attention_decode_b300 as he
    he.lib()


def small(**kw):
    return synth.WORKLOADS["llama8b_b8"].with_(**kw)


def all_units(w):
    return [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]


def stream_case(w, fill_n, steps, out_every, units=None, **opt):
    out_steps = sorted(set(range(0, steps, out_every)) | {steps - 1})
    g = run_gpu(w, fill_n, steps, out_steps, read_state=True, engine=FUSED, **opt)
    orc = run_oracle_units(w, units or all_units(w), fill_n, steps, out_steps, **opt)
    return compare(w, g, orc, out_steps, check_state=True)


@pytest.mark.parametrize("budget,fill_n", [(512, 512), (333, 300), (64, 0), (1, 1), (100, 37)])
def test_streams_ragged_budgets_and_appends(budget, fill_n):
    w = small(batch=2, budget=budget, prompt=2 * budget + 64, decode=8)
    stream_case(w, fill_n, budget - fill_n + 40, 7)


@pytest.mark.parametrize("G,D,bits", [(1, 128, 64), (2, 64, 8), (8, 128, 16), (8, 64, 32),
                                      (4, 64, 64)])
def test_group_sizes_dims_and_code_lengths(G, D, bits):
    w = small(batch=2, heads=4 * G, kv_heads=4, head_dim=D, bits=bits, budget=200, prompt=400,
              decode=8)
    stream_case(w, w.budget, 60, 11)


def test_threshold():
    w = small(batch=2, budget=300, prompt=700, decode=8)
    stream_case(w, w.budget, 50, 9, threshold=0.5)


def test_many_units_per_cta_and_many_ctas_per_unit():
    stream_case(small(batch=64, budget=40, prompt=80, decode=4), 40, 30, 9,
                units=[(0, 0), (5, 3), (31, 7), (63, 7)])
    stream_case(small(batch=1, heads=4, kv_heads=1, budget=20000, prompt=20100, decode=4), 20000,
                12, 5)


@pytest.mark.parametrize("bits", [32, 8, 64])
def test_step_distances_bit_exact(bits):
    """The distances the hash warps compute (each CTA over its own slots)."""
    import torch
    from gpu_harness import make_handle
    from lsh_pre_attention_decode_b300 import he_set_dist_log
    w = small(batch=2, bits=bits, budget=4096, prompt=4200)
    steps = 3
    with make_handle(w, engine=FUSED) as he:
        he.fill(synth.gpu_kv(w, "key", 0, w.budget), synth.gpu_kv(w, "value", 0, w.budget))
        q = synth.gpu_queries(w, w.budget, steps)
        k = synth.gpu_kv(w, "key", w.budget, steps, token_major=True)
        v = synth.gpu_kv(w, "value", w.budget, steps, token_major=True)
        dist = torch.full((steps, w.batch, w.kv_heads, w.budget), -1, dtype=torch.int32,
                          device="cuda")
        for t in range(steps):
            he_set_dist_log(he.h, dist[t])
            he.step(q[t], k[t], v[t])
        he_set_dist_log(he.h, None)
        got = dist.cpu().numpy()
    o = oracle.load()
    W = o.projection(w.projection_seed(), w.head_dim, bits, w.dtype)
    for b in range(w.batch):
        for j in range(w.kv_heads):
            st = o.unit_fill(W, w.budget, synth.host_unit_kv(w, "key", b, j, 0, w.budget),
                             synth.host_unit_kv(w, "value", b, j, 0, w.budget))
            r = o.unit_stream(st, synth.host_unit_queries(w, b, j, w.budget, steps),
                              synth.host_unit_kv(w, "key", b, j, w.budget, steps),
                              synth.host_unit_kv(w, "value", b, j, w.budget, steps),
                              dist_log=True)
            assert np.array_equal(got[:, b, j], r["dist"]), (b, j)


def check_b2b(w, fill_n, tokens, units, layers=1, graph=False, replays=2, warm=0, out_steps=(),
              check_layers=None, **opt):
    g = run_gpu_b2b(w, fill_n, tokens, out_steps, layers=layers, graph=graph, replays=replays,
                    warm=warm, engine=FUSED, **opt)
    for layer in (check_layers if check_layers is not None else range(layers)):
        orc = oracle_b2b(w, units, fill_n, g.tokens, out_steps, layer=layer, **opt)
        compare_b2b(w, g, layer, orc, out_steps)


@pytest.mark.parametrize("graph", [False, True])
def test_one_cache_back_to_back(graph):
    """Every step right behind the previous one on the same cache: the first
    tiles are fetched before the wait, the written slot (from the previous
    step's key once its hash warps have counted in) patched after it."""
    w = small(batch=2, budget=1024, prompt=2048, decode=8)
    n = 96
    outs = [0, 1, 47, 95] if not graph else [2 * n - 1, n + 5]
    check_b2b(w, w.budget, n, all_units(w), graph=graph, out_steps=outs)


def test_appends_then_evictions_back_to_back():
    w = small(batch=3, budget=333, prompt=800, decode=8)
    check_b2b(w, 300, 120, all_units(w), out_steps=[0, 20, 33, 34, 80, 119])


def test_empty_cache_back_to_back():
    w = small(batch=2, budget=70, prompt=200, decode=8)
    check_b2b(w, 0, 110, all_units(w), out_steps=[0, 1, 69, 70, 109])


def test_layer_rotation_as_benchmarked():
    """Four caches in turn, full Llama-3-8B layer shape, a graph of 64 tokens
    per layer replayed twice after 8 eager tokens."""
    w = synth.WORKLOADS["llama8b_b8"]
    units = [(0, 0), (2, 5), (5, 2), (7, 7)]
    check_b2b(w, w.budget, 64, units, layers=4, graph=True, replays=2, warm=8,
              out_steps=[8 + 64 + 63], check_layers=[0, 2])


def test_long_units_back_to_back():
    w = small(batch=1, heads=8, kv_heads=2, budget=20000, prompt=20100, decode=8)
    check_b2b(w, w.budget, 40, all_units(w), graph=True, replays=2, out_steps=[40, 79])
