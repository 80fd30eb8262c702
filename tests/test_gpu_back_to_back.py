"""GPU parity of steps issued the way a serving loop and the benchmark issue
them: back to back on one stream with no host synchronisation between steps,
eagerly and as a captured CUDA graph replayed several times in a row, over one
cache or several caches in turn (the benchmark's layer rotation).

Every step logs the slot it wrote on the device (he_set_evict_log), so the host
reads nothing until the last step has run.  In that mode the cache-streaming
kernel of a step fetches its first tiles while the previous step's merge may
still be writing the evicted row, and patches that row after its wait; these
tests check that path against the CPU oracle on the same token stream: every
eviction bit for bit, the final cache (keys, values, codes, and the value
scales or scores of the options) byte for byte, kept outputs within max-abs
1e-2 and mean-abs 1e-3 of the fp64 oracle (HashEvict paper, technical
framework steps 3-5: at every decoding step the current token replaces the
evicted one)."""
import pytest

import synth
from gpu_harness import compare_b2b, oracle_b2b, run_gpu_b2b

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_pre_attention_decode_b300 as he
    he.lib()


def small(**kw):
    return synth.WORKLOADS["llama8b_b8"].with_(**kw)


def check(w, fill_n, tokens, units, layers=1, graph=False, replays=2, warm=0, out_steps=(),
          check_layers=None, **opt):
    g = run_gpu_b2b(w, fill_n, tokens, out_steps, layers=layers, graph=graph, replays=replays,
                    warm=warm, **opt)
    for layer in (check_layers if check_layers is not None else range(layers)):
        orc = oracle_b2b(w, units, fill_n, g.tokens, out_steps, layer=layer, **opt)
        compare_b2b(w, g, layer, orc, out_steps)
    return g


def all_units(w):
    return [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]


@pytest.mark.parametrize("graph", [False, True])
def test_one_cache_back_to_back(graph):
    """One cache, every step right behind the previous one (the pre-wait fetch
    races the previous step's overwrite of the same cache)."""
    w = small(batch=2, budget=1024, prompt=2048, decode=8)
    n = 96
    outs = [0, 1, 47, 95] if not graph else [2 * n - 1, 2 * n - 2, n + 5]
    check(w, w.budget, n, all_units(w), graph=graph, out_steps=outs)


def test_graph_captured_right_after_fill_replays_consistently():
    """A graph captured on a freshly filled cache (no eager step first), replayed
    three times: each replay starts from the state the previous one left."""
    w = small(batch=2, budget=640, prompt=1400, decode=8)
    check(w, w.budget, 64, all_units(w), graph=True, replays=3, warm=0,
          out_steps=[128, 150, 191])


def test_layer_rotation_as_benchmarked():
    """Four caches in turn (layer 0, 1, 2, 3, layer 0, ...) as the benchmark
    issues them, a graph of 64 tokens per layer replayed twice after 8 eager
    tokens; full Llama-3-8B layer shape (batch 8, budget 4096 of an 8192-token
    prompt), sampled units of two layers."""
    w = synth.WORKLOADS["llama8b_b8"]
    units = [(0, 0), (1, 7), (3, 3), (4, 4), (6, 1), (7, 6)]
    outs = [8 + 64 + 63, 8 + 64 + 10]
    check(w, w.budget, 64, units, layers=4, graph=True, replays=2, warm=8, out_steps=outs,
          check_layers=[0, 3])


def test_ragged_budget_with_appends_back_to_back():
    """A cache filled below a ragged budget: appends (the pre-wait patch of the
    appended row), then evictions, all back to back."""
    w = small(batch=3, budget=333, prompt=800, decode=8)
    check(w, 300, 120, all_units(w), out_steps=[0, 20, 33, 34, 80, 119])


def test_many_ctas_per_unit_back_to_back():
    """Long units (most stream CTAs hold a part of every unit)."""
    w = small(batch=1, heads=8, kv_heads=2, budget=20000, prompt=20100, decode=8)
    check(w, w.budget, 40, all_units(w), graph=True, replays=2, out_steps=[40, 79])


@pytest.mark.parametrize("graph", [False, True])
def test_chunk_eviction_back_to_back(graph):
    """Chunks of 16 slots: a step after a chunk eviction fetches nothing before
    its wait (16 rows move); whole staging cycles per graph replay."""
    w = small(batch=2, budget=1024, prompt=2200, decode=8)
    if graph:
        check(w, w.budget, 64, all_units(w), graph=True, replays=2, chunk=16,
              out_steps=[64, 79, 80, 127])
    else:
        check(w, w.budget - 20, 100, all_units(w), chunk=16, out_steps=[0, 19, 20, 35, 36, 99])


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
@pytest.mark.parametrize("graph", [False, True])
def test_quantised_values_back_to_back(graph, fmt):
    w = small(batch=2, budget=900, prompt=1900, decode=8)
    if graph:
        check(w, w.budget, 64, all_units(w), graph=True, replays=2, v_format=fmt,
              out_steps=[64, 127])
    else:
        check(w, w.budget - 10, 80, all_units(w), v_format=fmt, out_steps=[0, 9, 10, 79])


@pytest.mark.parametrize("graph", [False, True])
def test_score_memory_back_to_back(graph):
    w = small(batch=2, budget=700, prompt=1500, decode=8)
    if graph:
        check(w, w.budget, 64, all_units(w), graph=True, replays=2, decay=0.5,
              out_steps=[64, 127])
    else:
        check(w, w.budget - 8, 80, all_units(w), decay=0.5, threshold=0.25,
              out_steps=[0, 8, 79])


@pytest.mark.parametrize("graph", [False, True])
def test_median_thresholds_back_to_back(graph):
    w = small(batch=2, budget=700, prompt=1500, decode=8)
    if graph:
        check(w, w.budget, 64, all_units(w), graph=True, replays=2, threshold="median",
              out_steps=[64, 127])
    else:
        check(w, w.budget - 8, 80, all_units(w), threshold="median", out_steps=[0, 8, 79])


def test_other_shapes_back_to_back():
    """G = 8 with D = 64 and 16-bit codes, G = 1; two caches in turn."""
    w = small(batch=2, heads=64, head_dim=64, bits=16, budget=500, prompt=1100, decode=8)
    check(w, w.budget, 64, all_units(w), layers=2, graph=True, replays=2, out_steps=[64, 127])
    w = small(batch=2, heads=8, kv_heads=8, bits=64, budget=300, prompt=700, decode=8)
    check(w, w.budget, 60, all_units(w), out_steps=[0, 59])


def test_more_units_than_sms_back_to_back():
    """320 units (several per merge CTA), a graph replayed twice."""
    w = small(batch=40, budget=200, prompt=500, decode=8)
    check(w, w.budget, 32, [(0, 0), (13, 4), (39, 7)], graph=True, replays=2,
          out_steps=[32, 63])
