"""Seeded synthetic workloads for the HashEvict decode step (inputs only).

Shared by the tests, the benchmark and the smoke check; holds none of the
method's arithmetic.  The generator itself is ``synth_core.h`` (plain source),
built twice: for the host with gcc (``libsynth_host.so``) and for the GPU with
nvcc (``libsynth_gpu.so``).  Both builds produce bit-identical tensors.

bf16 tensors on the host are ``numpy.uint16`` bit patterns; fp32 tensors are
``numpy.float32``.  Device tensors are torch tensors (bf16 or fp32).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libsynth_host.so")
GPU_LIB = os.path.join(HERE, "libsynth_gpu.so")
_SRCS_HOST = [os.path.join(HERE, f) for f in ("synth_core.h", "synth_host.c")]
_SRCS_GPU = [os.path.join(HERE, f) for f in ("synth_core.h", "synth_gpu.cu")]

MODE_LLAMA_BF16 = 0
MODE_IID_F32 = 1


class SynthCfg(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("layer", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("outliers", ctypes.c_int32 * 4)]


def _stale(out: str, srcs: list[str]) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(s) for s in srcs)


def build_host() -> str:
    if _stale(HOST_LIB, _SRCS_HOST):
        subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fPIC", "-shared",
                        "-o", HOST_LIB, os.path.join(HERE, "synth_host.c")], check=True)
    return HOST_LIB


def build_gpu() -> str:
    if _stale(GPU_LIB, _SRCS_GPU):
        subprocess.run(["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-o", GPU_LIB,
                        os.path.join(HERE, "synth_gpu.cu")], check=True)
    return GPU_LIB


def build() -> None:
    build_host()
    build_gpu()


_host = None
_gpu = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        P = ctypes.POINTER(SynthCfg)
        i32, vp = ctypes.c_int32, ctypes.c_void_p
        lib.synth_host_init.argtypes = [P]
        lib.synth_host_kv.argtypes = [P, ctypes.c_int, i32, i32, ctypes.c_int, vp]
        lib.synth_host_queries.argtypes = [P, i32, i32, vp]
        lib.synth_host_unit_kv.argtypes = [P, ctypes.c_int, i32, i32, i32, i32, vp]
        lib.synth_host_unit_queries.argtypes = [P, i32, i32, i32, i32, vp]
        lib.synth_host_mix64.argtypes = [ctypes.c_uint64]
        lib.synth_host_mix64.restype = ctypes.c_uint64
        lib.synth_host_normal.argtypes = [ctypes.c_uint64, i32]
        lib.synth_host_normal.restype = ctypes.c_float
        lib.synth_host_bf16.argtypes = [ctypes.c_float]
        lib.synth_host_bf16.restype = ctypes.c_uint16
        lib.synth_host_query_past.argtypes = [P, i32, i32, i32]
        lib.synth_host_query_past.restype = i32
        _host = lib
    return _host


def _gpu_lib():
    global _gpu
    if _gpu is None:
        lib = ctypes.CDLL(build_gpu())
        P = ctypes.POINTER(SynthCfg)
        i32, vp = ctypes.c_int32, ctypes.c_void_p
        lib.synth_gpu_kv.argtypes = [P, ctypes.c_int, i32, i32, ctypes.c_int, vp, vp]
        lib.synth_gpu_queries.argtypes = [P, i32, i32, vp, vp]
        _gpu = lib
    return _gpu


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """One HashEvict decode workload: head shapes, code length, cache budget,
    prompt length P (the first `budget` prompt tokens fill the cache, the rest
    stream through the step) and T decode steps."""
    name: str
    batch: int
    heads: int
    kv_heads: int
    head_dim: int
    bits: int
    budget: int
    dtype: str  # "bf16" | "fp32"
    prompt: int
    decode: int
    layers: int = 1
    seed: int = 1234
    description: str = ""

    @property
    def group(self) -> int:
        return self.heads // self.kv_heads

    @property
    def mode(self) -> int:
        return MODE_IID_F32 if self.dtype == "fp32" else MODE_LLAMA_BF16

    @property
    def streamed(self) -> int:
        """Tokens that go through the step: P - budget prompt tokens + T."""
        return self.prompt - self.budget + self.decode

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "fp32" else 2

    def with_(self, **kw) -> "Workload":
        d = {k: getattr(self, k) for k in self.__dataclass_fields__}
        d.update(kw)
        return Workload(**d)

    def projection_seed(self, layer: int = 0) -> int:
        """Seed of the projection matrix of a layer (one matrix per layer)."""
        return (self.seed * 0x9E3779B1 + 0x5EED + layer) & 0xFFFFFFFFFFFFFFFF

    def cfg(self, layer: int = 0) -> SynthCfg:
        c = SynthCfg(seed=self.seed, layer=layer, batch=self.batch, heads=self.heads,
                     kv_heads=self.kv_heads, head_dim=self.head_dim, mode=self.mode)
        _host_lib().synth_host_init(ctypes.byref(c))
        return c


WORKLOADS: dict[str, Workload] = {w.name: w for w in [
    Workload("tiny_fp32", 1, 4, 4, 64, 16, 256, "fp32", 512, 64, seed=1235,
             description="batch 1, 4/4 heads, head_dim 64, fp32, 16-bit codes, budget 256, "
                         "prompt 512, 64 decode steps"),
    Workload("llama8b_b8", 8, 32, 8, 128, 32, 4096, "bf16", 8192, 256, seed=1236,
             description="Llama-3-8B-shaped layer: batch 8, 32/8 heads, head_dim 128, bf16, "
                         "32-bit codes, prompt 8192, budget 4096, 256 decode steps"),
    Workload("long_128k", 1, 32, 8, 128, 32, 65536, "bf16", 131072, 512, seed=1237,
             description="batch 1, 32/8 heads, head_dim 128, bf16, 32-bit codes, prompt 131072, "
                         "budget 65536, 512 decode steps"),
    Workload("serving_b64", 64, 32, 8, 128, 16, 2816, "bf16", 4096, 128, seed=1238,
             description="batch 64, 32/8 heads, head_dim 128, bf16, 16-bit codes, prompt 4096, "
                         "budget 2816, 128 decode steps"),
    Workload("llama8b_32layer", 16, 32, 8, 128, 32, 9728, "bf16", 32768, 64, layers=32,
             seed=1239,
             description="32 attention layers: batch 16, 32/8 heads, head_dim 128, bf16, "
                         "prompt 32768, budget 9728, 64 decode steps, code length 8/16/32/64"),
]}


# ---------------------------------------------------------------------------
# Host generation (numpy)
# ---------------------------------------------------------------------------

def _np_dtype(w: Workload):
    return np.float32 if w.dtype == "fp32" else np.uint16


def host_kv(w: Workload, which: str, t0: int, nt: int, layer: int = 0,
            token_major: bool = False) -> np.ndarray:
    """Keys or values of tokens [t0, t0+nt): cache layout [batch][kv][nt][D]
    or, with token_major, step layout [nt][batch][kv][D]."""
    c = w.cfg(layer)
    shape = (nt, w.batch, w.kv_heads, w.head_dim) if token_major else (
        w.batch, w.kv_heads, nt, w.head_dim)
    out = np.empty(shape, _np_dtype(w))
    _host_lib().synth_host_kv(ctypes.byref(c), 0 if which == "key" else 1, t0, nt,
                              int(token_major), out.ctypes.data_as(ctypes.c_void_p))
    return out


def host_queries(w: Workload, t0: int, nt: int, layer: int = 0) -> np.ndarray:
    """Queries of tokens [t0, t0+nt): [nt][batch][heads][D]."""
    c = w.cfg(layer)
    out = np.empty((nt, w.batch, w.heads, w.head_dim), _np_dtype(w))
    _host_lib().synth_host_queries(ctypes.byref(c), t0, nt, out.ctypes.data_as(ctypes.c_void_p))
    return out


def host_unit_kv(w: Workload, which: str, b: int, j: int, t0: int, nt: int,
                 layer: int = 0) -> np.ndarray:
    """Keys or values of one (batch b, KV head j) unit: [nt][D]."""
    c = w.cfg(layer)
    out = np.empty((nt, w.head_dim), _np_dtype(w))
    _host_lib().synth_host_unit_kv(ctypes.byref(c), 0 if which == "key" else 1, b, j, t0, nt,
                                   out.ctypes.data_as(ctypes.c_void_p))
    return out


def host_unit_queries(w: Workload, b: int, j: int, t0: int, nt: int, layer: int = 0) -> np.ndarray:
    """Queries of the G heads of KV group j: [nt][G][D]."""
    c = w.cfg(layer)
    out = np.empty((nt, w.group, w.head_dim), _np_dtype(w))
    _host_lib().synth_host_unit_queries(ctypes.byref(c), b, j, t0, nt,
                                        out.ctypes.data_as(ctypes.c_void_p))
    return out


# ---------------------------------------------------------------------------
# Device generation (torch tensors on the current CUDA device)
# ---------------------------------------------------------------------------

def _torch_dtype(w: Workload):
    import torch
    return torch.float32 if w.dtype == "fp32" else torch.bfloat16


def gpu_kv(w: Workload, which: str, t0: int, nt: int, layer: int = 0, token_major: bool = False,
           out=None, stream=None):
    import torch
    c = w.cfg(layer)
    shape = (nt, w.batch, w.kv_heads, w.head_dim) if token_major else (
        w.batch, w.kv_heads, nt, w.head_dim)
    if out is None:
        out = torch.empty(shape, dtype=_torch_dtype(w), device="cuda")
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _gpu_lib().synth_gpu_kv(ctypes.byref(c), 0 if which == "key" else 1, t0, nt,
                                 int(token_major), ctypes.c_void_p(out.data_ptr()),
                                 ctypes.c_void_p(s))
    if rc != 0:
        raise RuntimeError(f"synth_gpu_kv failed: CUDA error {rc}")
    return out


def gpu_queries(w: Workload, t0: int, nt: int, layer: int = 0, out=None, stream=None):
    import torch
    c = w.cfg(layer)
    if out is None:
        out = torch.empty((nt, w.batch, w.heads, w.head_dim), dtype=_torch_dtype(w), device="cuda")
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _gpu_lib().synth_gpu_queries(ctypes.byref(c), t0, nt, ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(s))
    if rc != 0:
        raise RuntimeError(f"synth_gpu_queries failed: CUDA error {rc}")
    return out


def to_float(a: np.ndarray) -> np.ndarray:
    """Exact float64 values of a bf16-bits (uint16) or fp32 array."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)
