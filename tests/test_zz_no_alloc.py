"""he_attend_noalloc — decode attention that allocates no device memory.

It serves callers that cannot let a library allocate: work recorded under CUDA
graph capture (allocation cannot be captured), runtimes whose device memory is
owned by their own pool or arena, and deployments that fix every byte of device
memory up front.  It runs the same split-K attention kernel as he_step with its
scratch in a static device array.

he_step attends over the cache as it stands after the step, so he_attend_noalloc
on that cache with the same queries must give he_step's output, within the
tolerance of the parity tests.  This file is collected last on purpose.
"""
import numpy as np
import pytest

import lsh_pre_attention_decode_b300 as pkg
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


@pytest.mark.gpu
def test_matches_the_step_on_two_calls_in_a_row():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
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
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    buf = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1024, dtype=torch.float32, device="cuda")
    # 4096 (batch, KV head) units of partial records do not fit 8 MiB
    rc = pkg.lib().he_attend_noalloc(512, 32, 8, 128, 64, 64, buf.data_ptr(), buf.data_ptr(),
                                     buf.data_ptr(), out.data_ptr(), None)
    assert rc == -1
    assert np.isfinite(out.cpu().numpy()).all()
