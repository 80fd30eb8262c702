"""The synthetic workload generator (host build): determinism, layouts,
distribution shape.  CPU only."""
import numpy as np
import pytest
import torch

import synth


W2 = synth.WORKLOADS["llama8b_b8"].with_(batch=2, budget=64, prompt=128)
W1 = synth.WORKLOADS["tiny_fp32"]


def test_deterministic_and_seeded():
    a = synth.host_kv(W2, "key", 0, 16)
    b = synth.host_kv(W2, "key", 0, 16)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, synth.host_kv(W2, "key", 0, 16, layer=1))
    assert not np.array_equal(a, synth.host_kv(W2.with_(seed=7), "key", 0, 16))
    assert not np.array_equal(a, synth.host_kv(W2, "value", 0, 16))


def test_layouts_agree():
    cache = synth.host_kv(W2, "key", 5, 9)
    step = synth.host_kv(W2, "key", 5, 9, token_major=True)
    assert np.array_equal(cache.transpose(2, 0, 1, 3), step)
    for b in range(W2.batch):
        for j in range(W2.kv_heads):
            assert np.array_equal(synth.host_unit_kv(W2, "key", b, j, 5, 9), cache[b, j])
    q = synth.host_queries(W2, 3, 4)
    for j in range(W2.kv_heads):
        u = synth.host_unit_queries(W2, 1, j, 3, 4)
        assert np.array_equal(u, q[:, 1, j * W2.group:(j + 1) * W2.group])


def test_key_value_distribution():
    K = synth.to_float(synth.host_kv(W2, "key", 0, 512))
    V = synth.to_float(synth.host_kv(W2, "value", 0, 512))
    outl = list(W2.cfg().outliers)
    assert len(set(outl)) == 4 and all(0 <= c < W2.head_dim for c in outl)
    normal = [d for d in range(W2.head_dim) if d not in outl]
    assert abs(K[..., normal].std() - 1.0) < 0.02
    assert abs(K[..., outl].std() - 8.0) < 0.3
    assert abs(V.std() - 1.0) < 0.02 and abs(V.mean()) < 0.02
    assert np.abs(V).max() <= 6.0


def test_query_mixes_a_past_key():
    lib = synth._host_lib()
    cfg = W2.cfg()
    q = synth.to_float(synth.host_queries(W2, 0, 40))
    K = synth.to_float(synth.host_kv(W2, "key", 0, 40))
    resid = []
    for t in range(1, 40):
        for h in (0, 5, 31):
            tau = lib.synth_host_query_past(cfg, 0, h, t)
            assert 0 <= tau < t
            resid.append(q[t, 0, h] - 0.5 * K[0, h // W2.group, tau])
    r = np.concatenate(resid)
    assert abs(r.std() - 1.0) < 0.08  # the N(0,1) noise, up to bf16 rounding


def test_fp32_mode_is_iid():
    K = synth.host_kv(W1, "key", 0, 256)
    assert K.dtype == np.float32
    assert abs(K.std() - 1.0) < 0.03
    q = synth.host_queries(W1, 0, 64)
    assert abs(q.std() - 1.0) < 0.03


def test_bf16_rounding_matches_torch():
    lib = synth._host_lib()
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32) * 3
    ours = np.array([lib.synth_host_bf16(float(v)) for v in x], np.uint16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_normal_is_exact_irwin_hall():
    lib = synth._host_lib()
    vals = np.array([lib.synth_host_normal(12345, d) for d in range(20000)])
    assert np.all(np.abs(vals) <= 6.0)
    assert np.array_equal(vals * 65536, np.round(vals * 65536))  # multiples of 2^-16
    assert abs(vals.mean()) < 0.03 and abs(vals.std() - 1.0) < 0.02
