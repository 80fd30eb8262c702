"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Bar: projection matrix, codes, Hamming distances, evicted-slot sequences and the
cache contents bit-exact; attention output within max-abs 1e-2 and mean-abs
1e-3 of the oracle's fp64 result on the identical retained cache.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_harness import (compare, host_from_torch, make_handle, run_gpu, run_oracle_units,
                         torch_from_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_pre_attention_decode_b300 as he
    he.lib()  # the library must load: no fallback


def small(name, **kw):
    return synth.WORKLOADS[name].with_(**kw)


# ---------------------------------------------------------------------------
# steps 1-2
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,D,bits", [("bf16", 128, 32), ("bf16", 64, 8), ("bf16", 128, 64),
                                          ("fp32", 64, 16), ("fp32", 128, 64)])
def test_projection_bit_exact(dtype, D, bits):
    w = small("llama8b_b8", batch=1, heads=4, kv_heads=4, head_dim=D, bits=bits, budget=64,
              dtype=dtype)
    with make_handle(w) as he:
        got = he.projection()
    want = oracle.load().projection(w.projection_seed(), D, bits, dtype)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype,D,bits", [("bf16", 128, 32), ("bf16", 128, 16), ("bf16", 64, 8),
                                          ("bf16", 128, 64), ("fp32", 64, 16), ("fp32", 128, 32)])
def test_codes_bit_exact(dtype, D, bits):
    import torch
    from lsh_pre_attention_decode_b300 import he_codes
    w = small("llama8b_b8", batch=1, heads=4, kv_heads=4, head_dim=D, bits=bits, budget=64,
              dtype=dtype)
    o = oracle.load()
    rng = np.random.default_rng(D * bits)
    n = 1000
    xf = rng.standard_normal((n, D)).astype(np.float32)
    xf[1] = 0.0                      # all projections exactly 0 -> code 0
    xf[2] = 1e-30                    # tiny values
    with make_handle(w) as he:
        W = he.projection()
        Wf = synth.to_float(W)
        # rows whose projection onto column j is exactly zero (two exact products cancel)
        for r, jj in ((3, 0), (4, bits - 1), (5, bits // 2)):
            xf[r] = 0.0
            xf[r, 7] = Wf[11, jj]
            xf[r, 11] = -Wf[7, jj]
        x = xf if dtype == "fp32" else (
            (xf.view(np.uint32).astype(np.uint64) + 0x7FFF + ((xf.view(np.uint32) >> 16) & 1))
            >> 16).astype(np.uint16)
        xt = torch_from_host(x)
        ct = {8: torch.uint8, 16: torch.int16, 32: torch.int32, 64: torch.int64}[bits]
        codes = torch.empty(n, dtype=ct, device="cuda")
        he_codes(he.h, xt, n, codes)
        torch.cuda.synchronize()
        got = codes.cpu().numpy().view({8: np.uint8, 16: np.uint16, 32: np.uint32,
                                        64: np.uint64}[bits]).astype(np.uint64)
        want = o.code(x, W)
    assert np.array_equal(got, want)
    if dtype == "bf16":  # bf16 products are exact, so the two terms cancel exactly
        for r, jj in ((3, 0), (4, bits - 1), (5, bits // 2)):
            assert (int(want[r]) >> jj) & 1 == 0
    assert int(want[1]) == 0


def test_scores_bit_exact():
    import torch
    from lsh_pre_attention_decode_b300 import he_scores
    w = small("llama8b_b8", batch=2, budget=300, prompt=600)
    o = oracle.load()
    with make_handle(w) as he:
        K = synth.host_kv(w, "key", 0, w.budget)
        he.fill(torch_from_host(K), torch_from_host(synth.host_kv(w, "value", 0, w.budget)))
        q = synth.host_queries(w, w.budget, 1)[0]
        dist = torch.zeros((w.batch, w.kv_heads, w.budget), dtype=torch.int32, device="cuda")
        he_scores(he.h, torch_from_host(q), dist)
        got = dist.cpu().numpy()
        W = he.projection()
    for b in range(w.batch):
        for j in range(w.kv_heads):
            cq = o.code(q[b, j * w.group:(j + 1) * w.group], W)
            ck = o.code(K[b, j], W)
            want = [o.group_distance(cq, int(c)) for c in ck]
            assert got[b, j].tolist() == want


@pytest.mark.parametrize("bits,budget,opt", [(32, 4096, {}), (8, 4096, {}), (64, 4096, {}),
                                              (16, 9000, {}), (32, 5000, {"decay": 0.5}),
                                              (32, 4096, {"threshold": 0.5}),
                                              (32, 4096, {"v_format": "int8"}),
                                              (32, 4096, {"v_format": "fp8"}),
                                              (32, 4096, {"threshold": "median"}),
                                              (64, 9000, {"threshold": "median"})])
def test_step_distances_bit_exact(bits, budget, opt):
    """The group-summed Hamming distances that the step's own scan computes
    (method step 3, the codes/eviction kernel of every step), logged on the
    device for three steps issued back to back, against the oracle's distances
    on the same token stream: Llama-3-8B-shaped units (32/8 heads, head_dim 128),
    one and several scan items per unit (budget 9000), the options."""
    import torch
    from lsh_pre_attention_decode_b300 import he_set_dist_log
    w = small("llama8b_b8", batch=2, bits=bits, budget=budget, prompt=budget + 64)
    decay, tau = opt.get("decay", 0.0), opt.get("threshold", 0.0)
    vq = opt.get("v_format", "elem")
    steps = 3
    with make_handle(w, threshold=tau, decay=decay, v_format=vq) as he:
        he.fill(synth.gpu_kv(w, "key", 0, w.budget), synth.gpu_kv(w, "value", 0, w.budget))
        q = synth.gpu_queries(w, w.budget, steps)
        k = synth.gpu_kv(w, "key", w.budget, steps, token_major=True)
        v = synth.gpu_kv(w, "value", w.budget, steps, token_major=True)
        dist = torch.full((steps, w.batch, w.kv_heads, w.budget), -1, dtype=torch.int32,
                          device="cuda")
        out = torch.empty((w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
        for t in range(steps):
            he_set_dist_log(he.h, dist[t])
            he.step(q[t], k[t], v[t], out)
        he_set_dist_log(he.h, None)
        got = dist.cpu().numpy()
    o = oracle.load()
    W = o.projection(w.projection_seed(), w.head_dim, bits, w.dtype)
    for b in range(w.batch):
        for j in range(w.kv_heads):
            st = o.unit_fill(W, w.budget, synth.host_unit_kv(w, "key", b, j, 0, w.budget),
                             synth.host_unit_kv(w, "value", b, j, 0, w.budget),
                             tau=0.0 if tau == "median" else tau, memory=decay > 0.0,
                             median=tau == "median")
            r = o.unit_stream(st, synth.host_unit_queries(w, b, j, w.budget, steps),
                              synth.host_unit_kv(w, "key", b, j, w.budget, steps),
                              synth.host_unit_kv(w, "value", b, j, w.budget, steps),
                              dist_log=True, decay=decay)
            assert np.array_equal(got[:, b, j], r["dist"]), (b, j)


def test_chunk_step_distances_bit_exact():
    """With chunk eviction the scan logs every slot's own distance (the chunks'
    sums are built from them): compared with the brute-force group distances
    of the cache before the step."""
    import torch
    from lsh_pre_attention_decode_b300 import he_set_dist_log
    w = small("llama8b_b8", batch=2, budget=4800, prompt=4900)
    c = 16
    o = oracle.load()
    with make_handle(w, chunk=c) as he:
        K = synth.host_kv(w, "key", 0, w.budget)
        he.fill(torch_from_host(K), torch_from_host(synth.host_kv(w, "value", 0, w.budget)))
        q = synth.host_queries(w, w.budget, c)
        k = synth.host_kv(w, "key", w.budget, c, token_major=True)
        v = synth.host_kv(w, "value", w.budget, c, token_major=True)
        dist = torch.full((w.batch, w.kv_heads, he.rows), -1, dtype=torch.int32, device="cuda")
        for t in range(c):  # c - 1 staged tokens, then the evicting step
            if t == c - 1:
                he_set_dist_log(he.h, dist)
            he.step(torch_from_host(q[t]), torch_from_host(k[t]), torch_from_host(v[t]))
        got = dist.cpu().numpy()
        W = he.projection()
    for b in range(w.batch):
        for j in range(w.kv_heads):
            cq = o.code(q[c - 1, b, j * w.group:(j + 1) * w.group], W)
            ck = o.code(K[b, j], W)
            want = [o.group_distance(cq, int(x)) for x in ck]
            assert got[b, j, :w.budget].tolist() == want
            assert (got[b, j, w.budget:] == -1).all()


# ---------------------------------------------------------------------------
# whole streams: method steps 1-5 + attention
# ---------------------------------------------------------------------------

def _stream_case(w, fill_n, steps, out_every=1, units=None, check_state=True, device_gen=False):
    out_steps = list(range(0, steps, out_every)) + [steps - 1]
    out_steps = sorted(set(out_steps))
    g = run_gpu(w, fill_n, steps, out_steps, read_state=check_state, device_gen=device_gen)
    if units is None:
        units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    orc = run_oracle_units(w, units, fill_n, steps, out_steps)
    return compare(w, g, orc, out_steps, check_state=check_state)


def test_tiny_fp32_full_stream():
    """batch 1, 4/4 heads, head_dim 64, fp32, 16-bit codes, budget 256: the first
    256 of 512 prompt tokens fill the cache, 256 + 64 tokens stream; every step,
    every unit, every output."""
    w = synth.WORKLOADS["tiny_fp32"]
    _stream_case(w, w.budget, w.streamed, out_every=1)


def test_llama_shape_small_budget():
    """32/8 heads, head_dim 128, bf16, 32-bit codes, outlier channels; budget 512."""
    w = small("llama8b_b8", batch=2, budget=512, prompt=1024, decode=64)
    _stream_case(w, w.budget, w.streamed, out_every=37)


@pytest.mark.parametrize("bits", [8, 16, 32, 64])
def test_code_lengths(bits):
    w = small("llama8b_32layer", batch=2, budget=320, prompt=640, decode=16, bits=bits)
    _stream_case(w, w.budget, 80, out_every=13)


@pytest.mark.parametrize("G,D,dtype", [(1, 128, "bf16"), (2, 64, "bf16"), (8, 128, "bf16"),
                                       (8, 64, "fp32"), (4, 128, "fp32"), (2, 128, "fp32")])
def test_group_sizes_and_dims(G, D, dtype):
    w = small("llama8b_b8", batch=2, heads=4 * G, kv_heads=4, head_dim=D, dtype=dtype,
              budget=200, prompt=400, decode=8, bits=32)
    _stream_case(w, w.budget, 60, out_every=11)


@pytest.mark.parametrize("budget,fill_n", [(100, 100), (33, 33), (1, 1), (70, 10), (64, 0),
                                           (31, 5), (257, 250)])
def test_ragged_budgets_and_appends(budget, fill_n):
    """Budgets that are not a multiple of the 32-slot tile, a one-slot cache, and
    caches filled below the budget (the first tokens are appended)."""
    w = small("llama8b_b8", batch=3, budget=budget, prompt=2 * budget + 8, decode=4)
    steps = budget - fill_n + 40
    _stream_case(w, fill_n, steps, out_every=7)


def test_many_units_per_cta_and_many_ctas_per_unit():
    """Tiny units (several per CTA range) and one long unit (many CTAs per unit)."""
    _stream_case(small("serving_b64", batch=64, budget=40, prompt=80, decode=4), 40, 30,
                 out_every=9, units=[(0, 0), (5, 3), (31, 7), (63, 7)])
    _stream_case(small("long_128k", batch=1, heads=4, kv_heads=1, budget=20000, prompt=40000,
                       decode=4), 20000, 12, out_every=5)


def test_units_of_many_tiles():
    """64 units of 32 tiles (budget 2048): every stream CTA covers several
    segments of up to seven tiles; every unit, outputs sampled."""
    w = small("llama8b_b8", batch=8, budget=2048, prompt=4096, decode=4)
    _stream_case(w, w.budget, 24, out_every=5)


def test_all_keys_equal_tie_goes_to_slot_zero():
    """Identical cached keys: every distance ties, so slot 0 is evicted; the new
    token (identical key) keeps the tie for the next step."""
    import torch
    w = small("llama8b_b8", batch=1, budget=96, prompt=200, decode=4)
    he = make_handle(w)
    try:
        K = np.broadcast_to(synth.host_kv(w, "key", 0, 1), (1, 8, w.budget, 128)).copy()
        V = synth.host_kv(w, "value", 0, w.budget)
        he.fill(torch_from_host(K), torch_from_host(V))
        q = torch_from_host(synth.host_queries(w, w.budget, 6))
        kk = torch_from_host(K[:, :, 0])
        v = torch_from_host(synth.host_kv(w, "value", w.budget, 6, token_major=True))
        for i in range(6):
            he.step(q[i], kk, v[i])
            assert he.last_evicted().tolist() == [[0] * 8]
    finally:
        he.close()


@pytest.mark.parametrize("opt", [
    {}, {"v_format": "int8"}, {"v_format": "fp8"}, {"chunk": 4}, {"decay": 0.5},
    {"threshold": "median"}, {"engine": "fused"}, {"dtype": "fp32"}],
    ids=["method", "int8", "fp8", "chunk4", "decay", "median", "fused", "fp32"])
def test_host_entry_point_matches_device_entry_point(opt):
    """he_step_host (host buffers, copies inside the call) gives the device
    entry point's results bit for bit, with each option."""
    import torch
    from lsh_pre_attention_decode_b300 import he_step_host
    opt = dict(opt)
    w = small("llama8b_b8", batch=2, budget=128, prompt=256, decode=4,
              dtype=opt.pop("dtype", "bf16"))
    outs = []
    for host in (False, True):
        he = make_handle(w, **opt)
        try:
            he.fill(torch_from_host(synth.host_kv(w, "key", 0, w.budget)),
                    torch_from_host(synth.host_kv(w, "value", 0, w.budget)))
            q = synth.host_queries(w, w.budget, 5)
            k = synth.host_kv(w, "key", w.budget, 5, token_major=True)
            v = synth.host_kv(w, "value", w.budget, 5, token_major=True)
            res = []
            for i in range(5):
                if host:
                    o = np.empty((w.batch, w.heads, w.head_dim), np.float32)
                    he_step_host(he.h, np.ascontiguousarray(q[i]), np.ascontiguousarray(k[i]),
                                 np.ascontiguousarray(v[i]), o)
                else:
                    o = he.step(torch_from_host(q[i]), torch_from_host(k[i]),
                                torch_from_host(v[i])).cpu().numpy()
                res.append((o, he.last_evicted()))
            outs.append(res)
        finally:
            he.close()
    for (a, ea), (b, eb) in zip(*outs):
        assert np.array_equal(a, b) and np.array_equal(ea, eb)


# ---------------------------------------------------------------------------
# full-size workloads (sampled units / steps, as the benchmark launches them)
# ---------------------------------------------------------------------------

def test_gpu_generator_matches_host_generator():
    for name in ("llama8b_b8", "tiny_fp32"):
        w = synth.WORKLOADS[name].with_(batch=2)
        assert np.array_equal(host_from_torch(synth.gpu_kv(w, "key", 100, 9)),
                              synth.host_kv(w, "key", 100, 9))
        assert np.array_equal(host_from_torch(synth.gpu_kv(w, "value", 7, 5, token_major=True)),
                              synth.host_kv(w, "value", 7, 5, token_major=True))
        assert np.array_equal(host_from_torch(synth.gpu_queries(w, 3000, 4, layer=3)),
                              synth.host_queries(w, 3000, 4, layer=3))


@pytest.mark.slow
def test_full_llama8b_b8_all_steps():
    """Llama-3-8B-shaped layer at full size (batch 8, 32/8 heads, budget 4096 of an
    8192-token prompt, 256 decode steps): all 4352 streamed steps on the GPU;
    8 units checked bit-exact on every eviction, outputs at 9 steps."""
    w = synth.WORKLOADS["llama8b_b8"]
    steps = w.streamed
    out_steps = [0, 1, 500, 1000, 2000, 3000, 4095, 4096, steps - 1]
    units = [(0, 0), (1, 7), (2, 3), (3, 4), (4, 1), (5, 6), (6, 2), (7, 5)]
    g = run_gpu(w, w.budget, steps, out_steps, device_gen=True)
    orc = run_oracle_units(w, units, w.budget, steps, out_steps)
    compare(w, g, orc, out_steps)


@pytest.mark.slow
def test_full_serving_b64_sampled():
    w = synth.WORKLOADS["serving_b64"]
    steps = 200
    out_steps = [0, 99, 199]
    units = [(0, 0), (17, 3), (42, 6), (63, 7)]
    g = run_gpu(w, w.budget, steps, out_steps, device_gen=True)
    compare(w, g, run_oracle_units(w, units, w.budget, steps, out_steps), out_steps)


@pytest.mark.slow
def test_full_long_128k_first_64_steps():
    w = synth.WORKLOADS["long_128k"]
    steps = 64
    out_steps = [0, 31, 63]
    g = run_gpu(w, w.budget, steps, out_steps, device_gen=True)
    compare(w, g, run_oracle_units(w, [(0, 0), (0, 5)], w.budget, steps, out_steps), out_steps)


@pytest.mark.slow
@pytest.mark.parametrize("bits", [8, 16, 32, 64])
def test_full_32layer_sampled_layers(bits):
    w = synth.WORKLOADS["llama8b_32layer"].with_(bits=bits)
    steps = 64
    out_steps = [0, 63]
    for layer in (0, 31):
        g = run_gpu(w, w.budget, steps, out_steps, layer=layer, device_gen=True)
        orc = run_oracle_units(w, [(0, 0), (15, 7)], w.budget, steps, out_steps, layer=layer)
        compare(w, g, orc, out_steps)
