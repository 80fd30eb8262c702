"""The C ABI library without a GPU: it builds for sm_103a, loads, exports every
entry point declared in include/hashevict.h, and rejects bad arguments before
touching the device.  CPU only."""
import ctypes
import os
import re

import pytest

import lsh_pre_attention_decode_b300 as pkg
from lsh_pre_attention_decode_b300 import _binding, _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hashevict.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return pkg.lib()


def declared_entry_points():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(he_\w+)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("he_create", "he_fill", "he_step", "he_destroy", "he_step_host", "he_last_evicted",
              "he_read_state", "he_get_projection", "he_codes", "he_scores", "he_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_entry_points():
        assert hasattr(L, n), n


def test_python_binding_has_the_same_names():
    for n in declared_entry_points():
        assert hasattr(pkg, n), n


def test_strerror(L):
    assert pkg.he_strerror(0) == "ok"
    for c in (-1, -2, -3, -4, -5):
        assert pkg.he_strerror(c) != "unknown error code"
    assert pkg.he_strerror(-99) == "unknown error code"


def cfg(**kw):
    d = dict(batch=1, heads=32, kv_heads=8, head_dim=128, bits=32, budget=256, dtype=0,
             threshold=0.0, seed=1, decay=0.0, v_format=0, chunk=0)
    d.update(kw)
    return pkg.HeCfg(**d)


@pytest.mark.parametrize("bad", [dict(batch=0), dict(heads=30), dict(kv_heads=0), dict(bits=12),
                                 dict(bits=128), dict(budget=0), dict(budget=(1 << 24) + 1),
                                 dict(head_dim=96), dict(head_dim=256), dict(dtype=2),
                                 dict(heads=64, kv_heads=4), dict(v_format=3),
                                 dict(v_format=-1), dict(v_format=1, dtype=1),
                                 dict(v_format=2, dtype=1),
                                 dict(batch=70000), dict(decay=-0.5), dict(decay=1.5),
                                 dict(decay=float("nan")), dict(threshold=float("inf")),
                                 dict(threshold=float("nan")), dict(chunk=-1), dict(chunk=17),
                                 dict(chunk=3), dict(chunk=2, dtype=1),
                                 dict(chunk=2, v_format=1), dict(chunk=2, v_format=2),
                                 dict(chunk=2, decay=0.5),
                                 dict(engine=2), dict(engine=-1), dict(engine=1, dtype=1),
                                 dict(engine=1, decay=0.5), dict(engine=1, v_format=1),
                                 dict(engine=1, v_format=2),
                                 dict(engine=1, chunk=4, budget=256), dict(tau_mode=2),
                                 dict(tau_mode=-1)])
def test_create_rejects_bad_configs(L, bad):
    h = ctypes.c_void_p()
    assert L.he_create(ctypes.byref(cfg(**bad)), ctypes.byref(h)) == -1
    assert not h.value


def test_null_arguments_are_rejected(L):
    assert L.he_create(None, None) == -1
    assert L.he_destroy(None) == 0
    assert L.he_fill(None, None, None, 0, None) == -1
    assert L.he_step(None, None, None, None, None, None) == -1
    assert L.he_step_host(None, None, None, None, None, None) == -1
    assert L.he_last_evicted(None, None) == -1
    assert L.he_read_state(None, None, None, None, None) == -1
    assert L.he_get_projection(None, None) == -1
    assert L.he_codes(None, None, 0, None, None) == -1
    assert L.he_scores(None, None, None, None) == -1
    assert L.he_occupancy(None, None) == -1
    assert L.he_step_bytes(None, None) == -1
    assert L.he_launch_info(None, None, None, None, None) == -1
    assert L.he_recompute_count(None, None) == -1
    assert L.he_read_scores(None, None) == -1
    assert L.he_read_vscales(None, None) == -1
    assert L.he_wait_probe(None, 1000, None) == -1
    assert L.he_set_evict_log(None, None, None, 0) == -1
    assert L.he_set_dist_log(None, None) == -1
    assert L.he_set_alloc_limit(0) == 0


def test_python_errors_raise(L):
    with pytest.raises(pkg.HashEvictError) as e:
        pkg.he_create(cfg(bits=7))
    assert e.value.code == -1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_binding, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(ImportError):
        _binding.lib()
