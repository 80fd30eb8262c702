"""he_attend_noalloc — decode attention that allocates no device memory.

It serves callers that cannot let a library allocate: runtimes whose device
memory is owned by their own pool or arena, and deployments that fix every byte
of device memory up front.  It runs the same split-K attention kernel as he_step
with its scratch in a static device array that every call shares.

Checked here: against the CPU oracle's fp64 attention on the identical cache
(stream CTAs that hold several tiles of several units, n below the budget,
head_dim 64 and 128, G = 1, 2, 4 and 8), two calls in a row each time, and on
a seeded sweep of random shapes; and against he_step's own output on the cache
the step leaves.  This file is
collected last on purpose.
"""
import numpy as np
import pytest

import lsh_pre_attention_decode_b300 as pkg
import oracle
import synth
from gpu_harness import MAX_ABS_TOL, MEAN_ABS_TOL, make_handle, torch_from_host


def test_rejects_bad_arguments_without_touching_the_device():
    L = pkg.lib()
    assert L.he_attend_noalloc(0, 32, 8, 128, 64, 64, None, None, None, None, None) == -1
    assert L.he_attend_noalloc(1, 30, 8, 128, 64, 64, None, None, None, None, None) == -1
    assert L.he_attend_noalloc(1, 32, 8, 96, 64, 64, None, None, None, None, None) == -1
    assert L.he_attend_noalloc(1, 32, 8, 128, 64, 65, None, None, None, None, None) == -1
    assert L.he_attend_noalloc(1, 32, 8, 128, 64, 0, None, None, None, None, None) == -1
    assert L.he_attend_noalloc(1, 32, 8, 128, 64, 64, None, None, None, None, None) == -1


def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.lib()


@pytest.mark.gpu
@pytest.mark.parametrize("batch,heads,kv,D,budget,n", [
    (8, 32, 8, 128, 4096, 4000),   # 64 units x 63 tiles: every CTA holds several tiles
    (2, 64, 8, 64, 1000, 777),     # G = 8, head_dim 64, ragged n
    (3, 8, 8, 128, 300, 300),      # G = 1
    (1, 8, 4, 64, 9000, 8999),     # G = 2, long units over many CTAs
])
def test_matches_the_oracle_on_two_calls_in_a_row(batch, heads, kv, D, budget, n):
    import torch
    _cuda()
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=batch, heads=heads, kv_heads=kv, head_dim=D,
                                            budget=budget, prompt=budget + 8)
    K = synth.host_kv(w, "key", 0, budget)
    V = synth.host_kv(w, "value", 0, budget)
    Q = synth.host_queries(w, budget, 2)
    Kd, Vd, Qd = torch_from_host(K), torch_from_host(V), torch_from_host(Q)
    o = oracle.load()
    G = heads // kv
    for call in range(2):
        out = torch.full((batch, heads, D), float("nan"), dtype=torch.float32, device="cuda")
        pkg.he_attend_noalloc(batch, heads, kv, D, budget, n, Kd, Vd, Qd[call], out)
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        worst_max = worst_mean = 0.0
        for b in range(batch):
            for j in range(kv):
                want = o.attend(Q[call, b, j * G:(j + 1) * G], K[b, j, :n], V[b, j, :n])
                err = np.abs(got[b, j * G:(j + 1) * G] - want)
                worst_max = max(worst_max, float(err.max()))
                worst_mean = max(worst_mean, float(err.mean()))
        assert worst_max <= MAX_ABS_TOL and worst_mean <= MEAN_ABS_TOL, (call, worst_max,
                                                                          worst_mean)


def _random_shape(i):
    rng = np.random.default_rng(6300 + i)
    G = int(rng.choice([1, 2, 4, 8]))
    kv = int(rng.integers(1, 9))
    budget = int(rng.integers(16, 6000))
    return dict(batch=int(rng.integers(1, 9)), heads=G * kv, kv=kv,
                D=int(rng.choice([64, 128])), budget=budget,
                n=int(rng.choice([budget, int(rng.integers(1, budget + 1))])),
                seed=int(rng.integers(1, 1 << 30)))


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(16), ids=[
    "{i}-b{batch}-h{heads}-kv{kv}-D{D}-B{budget}-n{n}".format(i=i, **_random_shape(i))
    for i in range(16)])
def test_random_shapes_match_the_oracle(i):
    """A seeded sweep of random shapes (batch, query and KV heads, head_dim,
    budget, n from 1 to the budget) against the oracle's fp64 attention."""
    import torch
    _cuda()
    c = _random_shape(i)
    batch, heads, kv, D, budget, n = (c["batch"], c["heads"], c["kv"], c["D"], c["budget"],
                                      c["n"])
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=batch, heads=heads, kv_heads=kv, head_dim=D,
                                            budget=budget, prompt=budget + 8, seed=c["seed"])
    K = synth.host_kv(w, "key", 0, budget)
    V = synth.host_kv(w, "value", 0, budget)
    Q = synth.host_queries(w, budget, 1)[0]
    out = torch.full((batch, heads, D), float("nan"), dtype=torch.float32, device="cuda")
    pkg.he_attend_noalloc(batch, heads, kv, D, budget, n, torch_from_host(K), torch_from_host(V),
                          torch_from_host(Q), out)
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    o = oracle.load()
    G = heads // kv
    worst_max = worst_mean = 0.0
    for b in range(batch):
        for j in range(kv):
            want = o.attend(Q[b, j * G:(j + 1) * G], K[b, j, :n], V[b, j, :n])
            err = np.abs(got[b, j * G:(j + 1) * G] - want)
            worst_max = max(worst_max, float(err.max()))
            worst_mean = max(worst_mean, float(err.mean()))
    assert worst_max <= MAX_ABS_TOL and worst_mean <= MEAN_ABS_TOL, (worst_max, worst_mean)


@pytest.mark.gpu
def test_matches_the_step_on_two_calls_in_a_row():
    import torch
    _cuda()
    w = synth.WORKLOADS["llama8b_b8"].with_(batch=2, budget=300, prompt=600)
    he = make_handle(w)
    try:
        he.fill(torch_from_host(synth.host_kv(w, "key", 0, w.budget)),
                torch_from_host(synth.host_kv(w, "value", 0, w.budget)))
        q = torch_from_host(synth.host_queries(w, w.budget, 2))
        k = torch_from_host(synth.host_kv(w, "key", w.budget, 2, token_major=True))
        v = torch_from_host(synth.host_kv(w, "value", w.budget, 2, token_major=True))
        for t in range(2):
            ref = he.step(q[t], k[t], v[t])
            K, V, _, occ = he.state()  # the cache after the step
            Kd, Vd = torch_from_host(K), torch_from_host(V)
            out = torch.full_like(ref, float("nan"))
            pkg.he_attend_noalloc(w.batch, w.heads, w.kv_heads, w.head_dim, w.budget, occ, Kd, Vd,
                                  q[t], out)
            torch.cuda.synchronize()
            err = (out - ref).abs()
            assert torch.isfinite(out).all()
            assert err.max().item() <= MAX_ABS_TOL and err.mean().item() <= MEAN_ABS_TOL, (
                t, err.max().item(), err.mean().item())
    finally:
        he.close()


@pytest.mark.gpu
def test_rejects_sizes_beyond_the_scratch():
    import torch
    _cuda()
    buf = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1024, dtype=torch.float32, device="cuda")
    # 4096 (batch, KV head) units of partial records do not fit 8 MiB
    rc = pkg.lib().he_attend_noalloc(512, 32, 8, 128, 64, 64, buf.data_ptr(), buf.data_ptr(),
                                     buf.data_ptr(), out.data_ptr(), None)
    assert rc == -1
    assert np.isfinite(out.cpu().numpy()).all()
