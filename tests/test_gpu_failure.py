"""Failure paths on the GPU, without a fault: an allocation that does not fit
(a simulated device-memory cap), a bounded wait that runs out (a barrier that
nothing completes, with a short limit), and calls in the wrong order.  Each
returns its status code; the CUDA context stays usable and later handles work."""
import time

import numpy as np
import pytest

import lsh_pre_attention_decode_b300 as pkg
import synth
from gpu_harness import compare, make_handle, run_gpu, run_oracle_units, torch_from_host

pytestmark = pytest.mark.gpu

W_SMALL = synth.WORKLOADS["llama8b_b8"].with_(batch=1, budget=128, prompt=256, decode=8)


def test_allocation_cap_fails_cleanly():
    import torch
    make_handle(W_SMALL).close()  # (loads the kernels: the measurement below sees only he_create)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    pkg.he_set_alloc_limit(64 << 10)
    try:
        with pytest.raises(pkg.HashEvictError) as e:
            make_handle(W_SMALL)
        assert e.value.code == -4  # HE_ENOMEM
    finally:
        pkg.he_set_alloc_limit(0)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0  # nothing was allocated
    # without the cap the same handle is created and works
    w = W_SMALL
    g = run_gpu(w, w.budget, 6, range(6), read_state=True)
    orc = run_oracle_units(w, [(0, j) for j in range(w.kv_heads)], w.budget, 6, range(6))
    compare(w, g, orc, range(6), check_state=True)


def test_median_fill_scratch_cap_leaves_the_handle_unfilled():
    """A refill whose threshold scratch does not fit the cap fails with
    HE_ENOMEM and leaves the handle unfilled (the step is refused, not run on
    new rows with old codes); the next fill that fits restores it, with the
    oracle's thresholds and codes."""
    import torch
    import oracle
    w = W_SMALL
    K = synth.host_kv(w, "key", 0, w.budget)
    V = synth.host_kv(w, "value", 0, w.budget)
    q = torch_from_host(synth.host_queries(w, w.budget, 1)[0])
    k = torch_from_host(synth.host_kv(w, "key", w.budget, 1, token_major=True)[0])
    v = torch_from_host(synth.host_kv(w, "value", w.budget, 1, token_major=True)[0])
    with make_handle(w, threshold="median") as he:
        he.fill(torch_from_host(K), torch_from_host(V))
        pkg.he_set_alloc_limit(1024)  # (the scratch: bits x budget floats per unit)
        try:
            with pytest.raises(pkg.HashEvictError) as e:
                he.fill(torch_from_host(K), torch_from_host(V))
            assert e.value.code == -4  # HE_ENOMEM
        finally:
            pkg.he_set_alloc_limit(0)
        with pytest.raises(pkg.HashEvictError) as e:
            he.step(q, k, v)
        assert e.value.code == -2  # HE_ENOTFILLED
        he.fill(torch_from_host(K), torch_from_host(V))
        he.step(q, k, v)
        o = oracle.load()
        W = o.projection(w.projection_seed(), w.head_dim, w.bits, w.dtype)
        tv = he.thresholds()
        for j in range(w.kv_heads):
            assert np.array_equal(tv[0, j], o.median_thresholds(K[0, j], W))


def test_bounded_wait_gives_up_and_reports():
    import torch
    w = W_SMALL
    he = make_handle(w)
    other = make_handle(w, layer=1)
    try:
        K = torch_from_host(synth.host_kv(w, "key", 0, w.budget))
        V = torch_from_host(synth.host_kv(w, "value", 0, w.budget))
        he.fill(K, V)
        q = torch_from_host(synth.host_queries(w, w.budget, 1))[0]
        k = torch_from_host(synth.host_kv(w, "key", w.budget, 1, token_major=True))[0]
        v = torch_from_host(synth.host_kv(w, "value", w.budget, 1, token_major=True))[0]
        he.step(q, k, v)
        assert (he.last_evicted() >= 0).all()
        t0 = time.perf_counter()
        pkg.he_wait_probe(he.h, 20000)  # 20 ms
        with pytest.raises(pkg.HashEvictError) as e:
            he.last_evicted()  # synchronises: the kernel has given up and exited
        elapsed = time.perf_counter() - t0
        assert e.value.code == -5  # HE_EDEVICE
        assert 0.015 < elapsed < 5.0, elapsed
        # the handle now refuses work
        with pytest.raises(pkg.HashEvictError) as e:
            he.step(q, k, v)
        assert e.value.code == -5
        # another handle on the same context is unaffected
        other.fill(K, V)
        other.step(q, k, v)
        assert other.last_evicted().shape == (w.batch, w.kv_heads)
    finally:
        he.close()
        other.close()
    torch.cuda.synchronize()


def test_calls_out_of_order_are_refused():
    import torch
    w = W_SMALL
    he = make_handle(w)
    try:
        q = torch.zeros((w.batch, w.heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
        k = torch.zeros((w.batch, w.kv_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(pkg.HashEvictError) as e:
            he.step(q, k, k)  # before he_fill
        assert e.value.code == -2  # HE_ENOTFILLED
        too_many = torch.zeros((w.batch, w.kv_heads, w.budget + 1, w.head_dim),
                               dtype=torch.bfloat16, device="cuda")
        with pytest.raises(pkg.HashEvictError) as e:
            he.fill(too_many, too_many)
        assert e.value.code == -1  # HE_EINVAL
        with pytest.raises(pkg.HashEvictError):
            pkg.he_wait_probe(he.h, 0)
        # the handle is still usable
        he.fill(None, None)
        he.step(q, k, k)
        assert (he.last_evicted() == -1).all()
    finally:
        he.close()
