"""ctypes binding of libhashevict.so, one Python function per C entry point
(same names), plus a small handle class.  Tensors are passed by data_ptr();
streams default to torch's current CUDA stream."""
from __future__ import annotations

import ctypes
import os

from ._build import LIB

HE_DTYPE_BF16 = 0
HE_DTYPE_FP32 = 1
HE_VFMT_ELEM = 0
HE_VFMT_INT8 = 1
HE_VFMT_FP8 = 2
HE_TAU_FIXED = 0
HE_TAU_MEDIAN = 1
HE_ENGINE_PIPELINE = 0
HE_ENGINE_FUSED = 1

_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


class HeCfg(ctypes.Structure):
    _fields_ = [("batch", _i32), ("heads", _i32), ("kv_heads", _i32), ("head_dim", _i32),
                ("bits", _i32), ("budget", _i32), ("dtype", _i32), ("threshold", ctypes.c_float),
                ("seed", ctypes.c_uint64), ("decay", ctypes.c_float), ("v_format", _i32),
                ("chunk", _i32), ("engine", _i32), ("tau_mode", _i32)]


class HashEvictError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {code} ({he_strerror(code)})")
        self.code = code


_lib = None


def lib_path() -> str:
    return LIB


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"libhashevict.so is not built ({LIB}); run "
                              "`python -m lsh_pre_attention_decode_b300._build`")
        L = ctypes.CDLL(LIB)
        P = ctypes.POINTER
        L.he_create.argtypes = [P(HeCfg), P(_vp)]
        L.he_fill.argtypes = [_vp, _vp, _vp, _i32, _vp]
        L.he_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp]
        L.he_step_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp]
        L.he_destroy.argtypes = [_vp]
        L.he_last_evicted.argtypes = [_vp, _vp]
        L.he_read_state.argtypes = [_vp, _vp, _vp, _vp, _vp]
        L.he_get_projection.argtypes = [_vp, _vp]
        L.he_codes.argtypes = [_vp, _vp, _i32, _vp, _vp]
        L.he_scores.argtypes = [_vp, _vp, _vp, _vp]
        L.he_occupancy.argtypes = [_vp, P(_i32)]
        L.he_step_bytes.argtypes = [_vp, P(ctypes.c_uint64)]
        L.he_launch_info.argtypes = [_vp, P(_i32), P(_i32), P(_i32), P(_i32)]
        L.he_recompute_count.argtypes = [_vp, P(ctypes.c_int64)]
        L.he_attend_noalloc.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp]
        L.he_read_scores.argtypes = [_vp, _vp]
        L.he_read_vscales.argtypes = [_vp, _vp]
        L.he_read_thresholds.argtypes = [_vp, _vp]
        L.he_set_alloc_limit.argtypes = [ctypes.c_uint64]
        L.he_wait_probe.argtypes = [_vp, ctypes.c_uint32, _vp]
        L.he_profile_start.argtypes = [_vp, _i32]
        L.he_profile_stop.argtypes = [_vp, P(ctypes.c_float), P(_i32)]
        L.he_set_evict_log.argtypes = [_vp, _vp, _vp, _i32]
        L.he_set_dist_log.argtypes = [_vp, _vp]
        L.he_strerror.argtypes = [ctypes.c_int]
        L.he_strerror.restype = ctypes.c_char_p
        for n in ("he_create", "he_fill", "he_step", "he_step_host", "he_destroy",
                  "he_last_evicted", "he_read_state", "he_get_projection", "he_codes", "he_scores",
                  "he_occupancy", "he_step_bytes", "he_launch_info", "he_recompute_count",
                  "he_attend_noalloc", "he_profile_start", "he_profile_stop", "he_read_scores",
                  "he_read_vscales", "he_set_alloc_limit", "he_wait_probe", "he_set_evict_log",
                  "he_set_dist_log", "he_read_thresholds"):
            getattr(L, n).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise HashEvictError(fn, rc)


def _ptr(x) -> int | None:
    """Device or host address of a torch tensor / numpy array / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def he_strerror(code: int) -> str:
    return lib().he_strerror(code).decode()


def he_create(cfg: HeCfg) -> int:
    h = _vp()
    _check("he_create", lib().he_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def he_fill(h: int, K, V, n: int, stream=None) -> None:
    _check("he_fill", lib().he_fill(h, _ptr(K), _ptr(V), n, _stream(stream)))


def he_step(h: int, q, k, v, out, stream=None) -> None:
    _check("he_step", lib().he_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _stream(stream)))


def he_step_host(h: int, q, k, v, out, stream=None) -> None:
    _check("he_step_host",
           lib().he_step_host(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _stream(stream)))


def he_destroy(h: int) -> None:
    _check("he_destroy", lib().he_destroy(h))


def he_last_evicted(h: int, host_slots) -> None:
    _check("he_last_evicted", lib().he_last_evicted(h, _ptr(host_slots)))


def he_read_state(h: int, K=None, V=None, codes=None, occupancy=None) -> None:
    _check("he_read_state", lib().he_read_state(h, _ptr(K), _ptr(V), _ptr(codes),
                                                _ptr(occupancy)))


def he_get_projection(h: int, host_W) -> None:
    _check("he_get_projection", lib().he_get_projection(h, _ptr(host_W)))


def he_codes(h: int, x, n: int, codes, stream=None) -> None:
    _check("he_codes", lib().he_codes(h, _ptr(x), n, _ptr(codes), _stream(stream)))


def he_scores(h: int, q, dist, stream=None) -> None:
    _check("he_scores", lib().he_scores(h, _ptr(q), _ptr(dist), _stream(stream)))


def he_occupancy(h: int) -> int:
    o = _i32()
    _check("he_occupancy", lib().he_occupancy(h, ctypes.byref(o)))
    return o.value


def he_set_alloc_limit(nbytes: int) -> None:
    _check("he_set_alloc_limit", lib().he_set_alloc_limit(nbytes))


def he_wait_probe(h: int, limit_us: int, stream=None) -> None:
    _check("he_wait_probe", lib().he_wait_probe(h, limit_us, _stream(stream)))


def he_read_vscales(h: int, host_scales) -> None:
    _check("he_read_vscales", lib().he_read_vscales(h, _ptr(host_scales)))


def he_read_thresholds(h: int, host_tau) -> None:
    _check("he_read_thresholds", lib().he_read_thresholds(h, _ptr(host_tau)))


def he_read_scores(h: int, host_scores) -> None:
    _check("he_read_scores", lib().he_read_scores(h, _ptr(host_scores)))


def he_step_bytes(h: int) -> int:
    b = ctypes.c_uint64()
    _check("he_step_bytes", lib().he_step_bytes(h, ctypes.byref(b)))
    return b.value


def he_recompute_count(h: int) -> int:
    t = ctypes.c_int64()
    _check("he_recompute_count", lib().he_recompute_count(h, ctypes.byref(t)))
    return t.value


def he_profile_start(h: int, max_steps: int) -> None:
    _check("he_profile_start", lib().he_profile_start(h, max_steps))


def he_profile_stop(h: int) -> dict:
    """Summed event times (ms) of the steps recorded since he_profile_start."""
    ms = (ctypes.c_float * 4)()
    n = _i32()
    _check("he_profile_stop", lib().he_profile_stop(h, ms, ctypes.byref(n)))
    return {"stream_ms": ms[0], "prep_ms": ms[1], "merge_ms": ms[2], "step_ms": ms[3],
            "steps": n.value}


def he_attend_noalloc(batch: int, heads: int, kv_heads: int, head_dim: int, budget: int, n: int,
                      K, V, q, out, stream=None) -> None:
    _check("he_attend_noalloc",
           lib().he_attend_noalloc(batch, heads, kv_heads, head_dim, budget, n, _ptr(K), _ptr(V),
                                   _ptr(q), _ptr(out), _stream(stream)))


def he_set_evict_log(h: int, log, count, capacity: int) -> None:
    _check("he_set_evict_log", lib().he_set_evict_log(h, _ptr(log), _ptr(count), capacity))


def he_set_dist_log(h: int, dist) -> None:
    _check("he_set_dist_log", lib().he_set_dist_log(h, _ptr(dist)))


def he_launch_info(h: int) -> dict:
    a, b, c, d = _i32(), _i32(), _i32(), _i32()
    _check("he_launch_info", lib().he_launch_info(h, ctypes.byref(a), ctypes.byref(b),
                                                  ctypes.byref(c), ctypes.byref(d)))
    return {"ctas": a.value, "ctas_per_sm": b.value, "tiles": c.value, "stages": d.value}


class HashEvict:
    """One layer's HashEvict cache on the current CUDA device (torch tensors)."""

    def __init__(self, batch: int, heads: int, kv_heads: int, head_dim: int, bits: int,
                 budget: int, dtype: str = "bf16", seed: int = 0, threshold: float = 0.0,
                 decay: float = 0.0, v_format: str = "elem", chunk: int = 1,
                 engine: str = "pipeline", tau_mode: str = "fixed"):
        self.cfg = HeCfg(batch=batch, heads=heads, kv_heads=kv_heads, head_dim=head_dim,
                         bits=bits, budget=budget,
                         dtype=HE_DTYPE_FP32 if dtype == "fp32" else HE_DTYPE_BF16,
                         threshold=threshold, seed=seed, decay=decay,
                         v_format={"elem": HE_VFMT_ELEM, "int8": HE_VFMT_INT8,
                                   "fp8": HE_VFMT_FP8}[v_format], chunk=chunk,
                         engine={"pipeline": HE_ENGINE_PIPELINE,
                                 "fused": HE_ENGINE_FUSED}[engine],
                         tau_mode={"fixed": HE_TAU_FIXED, "median": HE_TAU_MEDIAN}[tau_mode])
        self.v_format = v_format
        # rows per unit: the budget, plus chunk - 1 staging rows with chunk eviction
        self.rows = budget + max(chunk, 1) - 1
        self.dtype = dtype
        self.h = he_create(self.cfg)

    def close(self) -> None:
        if self.h:
            he_destroy(self.h)
            self.h = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    @property
    def torch_dtype(self):
        import torch
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def fill(self, K, V, stream=None) -> None:
        """K, V: [batch][kv_heads][n][head_dim] device tensors."""
        n = 0 if K is None else K.shape[2]
        he_fill(self.h, K, V, n, stream)

    def step(self, q, k, v, out=None, stream=None):
        import torch
        c = self.cfg
        if out is None:
            out = torch.empty((c.batch, c.heads, c.head_dim), dtype=torch.float32, device=q.device)
        he_step(self.h, q, k, v, out, stream)
        return out

    def last_evicted(self):
        import numpy as np
        a = np.empty((self.cfg.batch, self.cfg.kv_heads), np.int32)
        he_last_evicted(self.h, a)
        return a

    def state(self):
        """Host snapshot: K, V [batch][kv][rows][D] (uint16 bf16 bits or float32;
        V int8 or uint8 E4M3 codes with a quantised value cache), codes
        [batch][kv][rows] (uint8/16/32/64), occupancy."""
        import numpy as np
        c = self.cfg
        et = np.float32 if self.dtype == "fp32" else np.uint16
        ct = {8: np.uint8, 16: np.uint16, 32: np.uint32, 64: np.uint64}[c.bits]
        K = np.empty((c.batch, c.kv_heads, self.rows, c.head_dim), et)
        V = np.empty(K.shape, {"int8": np.int8, "fp8": np.uint8}.get(self.v_format, et))
        codes = np.empty((c.batch, c.kv_heads, self.rows), ct)
        occ = np.zeros(1, np.int32)
        he_read_state(self.h, K, V, codes, occ)
        return K, V, codes, int(occ[0])

    def thresholds(self):
        """Binarisation thresholds [batch][kv_heads][bits] (per-bit medians with
        tau_mode "median", else the threshold in every entry)."""
        import numpy as np
        c = self.cfg
        a = np.empty((c.batch, c.kv_heads, c.bits), np.float32)
        he_read_thresholds(self.h, a)
        return a

    def vscales(self):
        """Per-slot value scales [batch][kv_heads][budget] (quantised value cache only)."""
        import numpy as np
        c = self.cfg
        a = np.empty((c.batch, c.kv_heads, self.rows), np.float32)
        he_read_vscales(self.h, a)
        return a

    def scores(self):
        """Per-slot eviction scores [batch][kv_heads][budget] (score memory only)."""
        import numpy as np
        c = self.cfg
        a = np.empty((c.batch, c.kv_heads, self.rows), np.float32)
        he_read_scores(self.h, a)
        return a

    def projection(self):
        import numpy as np
        c = self.cfg
        W = np.empty((c.head_dim, c.bits), np.float32 if self.dtype == "fp32" else np.uint16)
        he_get_projection(self.h, W)
        return W

    @property
    def occupancy(self) -> int:
        return he_occupancy(self.h)

    @property
    def step_bytes(self) -> int:
        return he_step_bytes(self.h)

    def launch_info(self) -> dict:
        return he_launch_info(self.h)

    @property
    def recompute_count(self) -> int:
        return he_recompute_count(self.h)

    def profile_start(self, max_steps: int) -> None:
        he_profile_start(self.h, max_steps)

    def profile_stop(self) -> dict:
        return he_profile_stop(self.h)
