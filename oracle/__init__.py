"""CPU oracle of the HashEvict decode step — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path (``lsh_pre_attention_decode_b300``)
never does: it shares no code with the oracle.

The arithmetic lives in ``hashevict_oracle.c`` (plain C, compiled with gcc,
``-ffp-contract=off`` so that only the fused multiply-adds the code spells out
are fused).  This module only marshals numpy arrays:

* bf16 tensors are ``numpy.uint16`` arrays of bf16 bit patterns (dtype code 0),
* fp32 tensors are ``numpy.float32`` arrays (dtype code 1),
* codes are ``numpy.uint64`` (bit j of the code = bit j of the word).

Method: "HashEvict: A Pre-Attention KV Cache Eviction Strategy using
Locality-Sensitive Hashing" (arXiv 2412.16187), abstract and technical
framework steps 1-5; attention over the retained cache per the TTKV page's
introduction (each decode step attends the whole cache).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hashevict_oracle.c")
LIB = os.path.join(HERE, "libhashevict_oracle.so")

_i32 = ctypes.c_int32
_u64 = ctypes.c_uint64
_vp = ctypes.c_void_p


def build(out: str = LIB, mutant: int = 0) -> str:
    """Compile the oracle with gcc.  ``mutant`` > 0 plants one known mistake
    (see the ORACLE_MUTANT blocks in the C file); only the pin tests use that."""
    src_m = os.path.getmtime(SRC)
    if os.path.exists(out) and os.path.getmtime(out) >= src_m and mutant == 0:
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fPIC", "-shared",
           f"-DORACLE_MUTANT={int(mutant)}", "-o", out, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return 0
    if a.dtype == np.float32:
        return 1
    raise TypeError(f"oracle tensors are uint16 (bf16 bits) or float32, got {a.dtype}")


def _vfmt(fmt: str) -> int:
    """Byte format code of a quantised value cache: 1 int8, 2 fp8 (E4M3)."""
    try:
        return {"int8": 1, "fp8": 2}[fmt]
    except KeyError:
        raise ValueError(f"value format is 'int8' or 'fp8', got {fmt!r}") from None


def _tauv(tau, bits: int):
    """A per-bit threshold array (fp32 [bits]) from tau, or None for a scalar."""
    if np.ndim(tau) == 0:
        return None
    tv = np.ascontiguousarray(tau, np.float32)
    if tv.shape != (bits,):
        raise ValueError(f"per-bit thresholds must have shape ({bits},), got {tv.shape}")
    return tv


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_vp)


@dataclass
class UnitState:
    """Cache of one (batch, KV head) unit: K, V [budget][D], codes [budget]; with
    score memory, the per-slot scores A [budget] (fp32); tau: binarisation
    threshold of every code of this unit, or tauv [bits] (fp32): one threshold
    per bit (e.g. the per-bit medians of the filled keys' projections)."""
    W: np.ndarray
    bits: int
    budget: int
    K: np.ndarray
    V: np.ndarray
    codes: np.ndarray
    occupancy: int
    tau: float = 0.0
    score: np.ndarray | None = None
    Vq: np.ndarray | None = None     # quantised value cache: bytes [budget][D] (int8, or
    Vs: np.ndarray | None = None     # E4M3 codes as uint8) and one fp32 scale per row
                                     # (then V is unused)
    chunk: int = 1                   # chunk eviction: K, V, codes hold budget + chunk - 1 rows
    chunked: bool = False            # filled by unit_fill_chunk: streams run the chunk routine
    tauv: np.ndarray | None = None   # per-bit thresholds (then tau is unused)


class Oracle:
    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.orc_projection.argtypes = [_u64, _i32, _i32, _i32, _vp]
        lib.orc_projection.restype = None
        lib.orc_code.argtypes = [_vp, _i32, _i32, _vp, _i32]
        lib.orc_code.restype = _u64
        lib.orc_code_many.argtypes = [_vp, _i32, _i32, _i32, _vp, _i32, _vp]
        lib.orc_code_many.restype = None
        lib.orc_code_many_tau.argtypes = [_vp, _i32, _i32, _i32, _vp, _i32, ctypes.c_float, _vp,
                                          _vp]
        lib.orc_median_thresholds.argtypes = [_vp, _i32, _i32, _i32, _vp, _i32, _vp]
        lib.orc_median_thresholds.restype = None
        lib.orc_code_many_tau.restype = None
        lib.orc_most_dissimilar_score.argtypes = [_vp, _i32]
        lib.orc_most_dissimilar_score.restype = _i32
        lib.orc_unit_fill_tau.argtypes = [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _i32,
                                          ctypes.c_float, _vp, _vp, _vp, _vp, _vp]
        lib.orc_unit_fill_tau.restype = None
        lib.orc_unit_stream_ext.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                            _vp, _vp, _i32, _vp, _vp, _vp, ctypes.c_float, _vp,
                                            ctypes.c_float, _vp, _vp, _vp, _vp, _vp]
        lib.orc_unit_stream_ext.restype = None
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_quantize_row.argtypes = [_vp, _i32, _i32, _i32, _vp, _vp]
        lib.orc_quantize_row.restype = None
        lib.orc_attend_vq.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp]
        lib.orc_attend_vq.restype = None
        lib.orc_unit_fill_vq.argtypes = [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _i32,
                                         ctypes.c_float, _vp, _i32, _vp, _vp, _vp, _vp, _vp]
        lib.orc_unit_fill_vq.restype = None
        lib.orc_unit_stream_vq.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp,
                                           _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp,
                                           ctypes.c_float, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]
        lib.orc_unit_stream_vq.restype = None
        lib.orc_unit_stream_chunk.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp,
                                              _vp, _vp, _i32, _vp, _vp, _vp, ctypes.c_float, _vp, _vp,
                                              _vp, _vp, _vp]
        lib.orc_unit_stream_chunk.restype = None
        lib.orc_group_distance.argtypes = [_vp, _i32, _u64]
        lib.orc_group_distance.restype = _i32
        lib.orc_most_dissimilar.argtypes = [_vp, _i32]
        lib.orc_most_dissimilar.restype = _i32
        lib.orc_attend.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp]
        lib.orc_attend.restype = None
        lib.orc_unit_fill.argtypes = [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp,
                                      _vp, _vp]
        lib.orc_unit_fill.restype = None
        lib.orc_unit_stream.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                                        _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        lib.orc_unit_stream.restype = None
        self.lib = lib

    # -- steps 1-2 -----------------------------------------------------------
    def projection(self, seed: int, head_dim: int, bits: int, dtype: str) -> np.ndarray:
        """W[head_dim][bits], drawn from ``seed`` (bf16 bits or fp32)."""
        W = np.empty((head_dim, bits), np.uint16 if dtype == "bf16" else np.float32)
        self.lib.orc_projection(seed, head_dim, bits, _dtype_code(W), _ptr(W))
        return W

    def code(self, x: np.ndarray, W: np.ndarray, tau=0.0) -> np.ndarray:
        """Codes of the rows of x [n][D] (or one vector [D]) -> uint64 [n];
        bit j = (projection > tau), or (projection_j > tau[j]) for an array of
        one threshold per bit."""
        x2 = np.ascontiguousarray(x.reshape(-1, x.shape[-1]))
        Wc = np.ascontiguousarray(W)
        if _dtype_code(x2) != _dtype_code(Wc):
            raise TypeError("x and W must have the same element type")
        out = np.empty(x2.shape[0], np.uint64)
        tv = _tauv(tau, Wc.shape[1])
        if tv is None and float(tau) == 0.0:
            self.lib.orc_code_many(_ptr(x2), x2.shape[0], _dtype_code(x2), x2.shape[1], _ptr(Wc),
                                   Wc.shape[1], _ptr(out))
        else:
            self.lib.orc_code_many_tau(_ptr(x2), x2.shape[0], _dtype_code(x2), x2.shape[1],
                                       _ptr(Wc), Wc.shape[1], 0.0 if tv is not None else float(tau),
                                       _ptr(tv), _ptr(out))
        return out

    def median_thresholds(self, K: np.ndarray, W: np.ndarray) -> np.ndarray:
        """Per-bit thresholds [bits] (fp32): the lower median of the rows'
        projections onto each column of W (0 for no rows)."""
        K2 = np.ascontiguousarray(K.reshape(-1, K.shape[-1]))
        Wc = np.ascontiguousarray(W)
        tau = np.empty(Wc.shape[1], np.float32)
        self.lib.orc_median_thresholds(_ptr(K2), K2.shape[0], _dtype_code(K2), K2.shape[1],
                                       _ptr(Wc), Wc.shape[1], _ptr(tau))
        return tau

    # -- steps 3-4 -----------------------------------------------------------
    def group_distance(self, code_q: np.ndarray, code_slot: int) -> int:
        cq = np.ascontiguousarray(code_q, np.uint64)
        return int(self.lib.orc_group_distance(_ptr(cq), cq.size, int(code_slot)))

    def most_dissimilar(self, dist: np.ndarray) -> int:
        d = np.ascontiguousarray(dist, np.int32)
        return int(self.lib.orc_most_dissimilar(_ptr(d), d.size))

    def most_dissimilar_score(self, score: np.ndarray) -> int:
        a = np.ascontiguousarray(score, np.float32)
        return int(self.lib.orc_most_dissimilar_score(_ptr(a), a.size))

    # -- quantised values ----------------------------------------------------
    def e4m3_decode(self, c) -> np.ndarray:
        """The values of E4M3 codes (fp64, exact)."""
        c2 = np.asarray(c, np.uint8)
        return np.array([self.lib.orc_e4m3_decode(int(x)) for x in c2.ravel()],
                        np.float64).reshape(c2.shape)

    def e4m3_encode(self, x) -> np.ndarray:
        """The E4M3 codes nearest to fp32 values x (ties to even, saturating)."""
        x2 = np.asarray(x, np.float32)
        return np.array([self.lib.orc_e4m3_encode(float(v)) for v in x2.ravel()],
                        np.uint8).reshape(x2.shape)

    def quantize_rows(self, v: np.ndarray, fmt: str = "int8"):
        """Byte rows and fp32 scales of v [n][D] (bf16 bits or fp32): int8
        values (numpy int8) or E4M3 codes (``fmt="fp8"``, numpy uint8)."""
        f = _vfmt(fmt)
        v2 = np.ascontiguousarray(v.reshape(-1, v.shape[-1]))
        n, D = v2.shape
        q = np.empty((n, D), np.uint8 if f == 2 else np.int8)
        sc = np.empty(n, np.float32)
        row = D * v2.itemsize
        for i in range(n):
            self.lib.orc_quantize_row(ctypes.c_void_p(v2.ctypes.data + i * row), _dtype_code(v2), D,
                                      f, ctypes.c_void_p(q.ctypes.data + i * D),
                                      ctypes.c_void_p(sc.ctypes.data + 4 * i))
        return q, sc

    def dequantize_rows(self, q: np.ndarray, sc: np.ndarray) -> np.ndarray:
        """fp64 values decode(q) * s of byte rows from ``quantize_rows``."""
        deq = self.e4m3_decode(q) if q.dtype == np.uint8 else q.astype(np.float64)
        return deq * np.asarray(sc, np.float64)[..., None]

    def attend_vq(self, q: np.ndarray, K: np.ndarray, Vq: np.ndarray, Vs: np.ndarray) -> np.ndarray:
        """Attention over byte rows Vq (int8 values, or E4M3 codes as uint8)."""
        q2 = np.ascontiguousarray(q.reshape(-1, q.shape[-1]))
        K2, Vq2, Vs2 = (np.ascontiguousarray(a) for a in (K, Vq, Vs))
        G, D = q2.shape
        out = np.empty((G, D), np.float64)
        self.lib.orc_attend_vq(_ptr(q2), _ptr(K2), _ptr(Vq2), _ptr(Vs2), K2.shape[0], D, G,
                               _dtype_code(q2), 2 if Vq2.dtype == np.uint8 else 1, _ptr(out))
        return out

    # -- attention -----------------------------------------------------------
    def attend(self, q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
        """fp64 softmax(q K^T / sqrt(D)) V for q [G][D], K, V [n][D]."""
        q2 = np.ascontiguousarray(q.reshape(-1, q.shape[-1]))
        K2 = np.ascontiguousarray(K)
        V2 = np.ascontiguousarray(V)
        G, D = q2.shape
        out = np.empty((G, D), np.float64)
        self.lib.orc_attend(_ptr(q2), _ptr(K2), _ptr(V2), K2.shape[0], D, G, _dtype_code(q2),
                            _ptr(out))
        return out

    # -- one (batch, KV head) unit -----------------------------------------
    def unit_fill_chunk(self, W: np.ndarray, budget: int, chunk: int, Kin: np.ndarray,
                        Vin: np.ndarray, tau: float = 0.0, median: bool = False) -> UnitState:
        """A unit for chunk eviction: room for budget + chunk - 1 rows."""
        if budget % chunk:
            raise ValueError("the budget must be a whole number of chunks")
        st = self.unit_fill(W, budget + chunk - 1, Kin, Vin, tau=tau, median=median)
        st.budget = budget
        st.chunk = chunk
        st.chunked = True  # (c = 1 too: then the chunk routine must give the method)
        return st

    def unit_fill(self, W: np.ndarray, budget: int, Kin: np.ndarray, Vin: np.ndarray,
                  tau: float = 0.0, memory: bool = False, vq=False,
                  median: bool = False) -> UnitState:
        """A unit filled with the rows of Kin, Vin.  ``memory``: keep per-slot
        scores (zero after the fill) for streams with score memory.  ``vq``:
        a quantised value cache, one byte per value and one fp32 scale per row:
        ``True`` or ``"int8"`` (int8 values), ``"fp8"`` (E4M3 codes).
        ``median``: one threshold per bit, the lower median of the filled
        keys' projections (fixed for the unit's later steps; tau unused)."""
        n, D = Kin.shape
        if n > budget:
            raise ValueError("more fill tokens than the budget")
        tv = self.median_thresholds(Kin, W) if median else None
        if tv is not None:
            tau = 0.0
        if vq:
            f = _vfmt("int8" if vq is True else vq)
            K = np.zeros((budget, D), Kin.dtype)
            Vq = np.zeros((budget, D), np.uint8 if f == 2 else np.int8)
            Vs = np.zeros(budget, np.float32)
            codes = np.zeros(budget, np.uint64)
            occ = np.zeros(1, np.int32)
            Kc, Vc, Wc = (np.ascontiguousarray(a) for a in (Kin, Vin, W))
            self.lib.orc_unit_fill_vq(_ptr(Wc), D, Wc.shape[1], _dtype_code(Kc), budget, _ptr(Kc),
                                      _ptr(Vc), n, float(tau), _ptr(tv), f, _ptr(K), _ptr(Vq),
                                      _ptr(Vs), _ptr(codes), _ptr(occ))
            score = np.zeros(budget, np.float32) if memory else None
            return UnitState(Wc, Wc.shape[1], budget, K, None, codes, int(occ[0]), float(tau),
                             score, Vq, Vs, tauv=tv)
        K = np.zeros((budget, D), Kin.dtype)
        V = np.zeros((budget, D), Kin.dtype)
        codes = np.zeros(budget, np.uint64)
        occ = np.zeros(1, np.int32)
        Kc, Vc, Wc = (np.ascontiguousarray(a) for a in (Kin, Vin, W))
        if tau == 0.0 and tv is None:
            self.lib.orc_unit_fill(_ptr(Wc), D, Wc.shape[1], _dtype_code(Kc), budget, _ptr(Kc),
                                   _ptr(Vc), n, _ptr(K), _ptr(V), _ptr(codes), _ptr(occ))
        else:
            self.lib.orc_unit_fill_tau(_ptr(Wc), D, Wc.shape[1], _dtype_code(Kc), budget,
                                       _ptr(Kc), _ptr(Vc), n, float(tau), _ptr(tv), _ptr(K),
                                       _ptr(V), _ptr(codes), _ptr(occ))
        score = np.zeros(budget, np.float32) if memory else None
        return UnitState(Wc, Wc.shape[1], budget, K, V, codes, int(occ[0]), float(tau), score,
                         tauv=tv)

    def unit_stream(self, st: UnitState, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                    want_out: np.ndarray | None = None, dist_log: bool = False,
                    decay: float = 0.0) -> dict:
        """Run tokens q [T][G][D], k, v [T][D] through the step (state updated
        in place).  Returns evicted [T] (-1 = appended), written [T], out
        [n_wanted][G][D] fp64 and, if asked, dist [T][budget].  A unit filled
        with ``memory`` evicts by scores with memory ``decay`` (the unit's tau
        applies to every code)."""
        T, G, D = q.shape
        qc, kc, vc = (np.ascontiguousarray(a) for a in (q, k, v))
        evicted = np.empty(T, np.int32)
        written = np.empty(T, np.int32)
        if want_out is None:
            n_out = T
            wo = None
        else:
            wo = np.ascontiguousarray(want_out, np.uint8)
            n_out = int(wo.astype(bool).sum())
        out = np.empty((n_out, G, D), np.float64)
        dl = np.empty((T, st.budget), np.int32) if dist_log else None
        occ = np.array([st.occupancy], np.int32)
        if st.chunked:
            if decay != 0.0 or st.score is not None or st.Vq is not None or dist_log:
                raise ValueError("chunk eviction takes neither score memory nor int8 values")
            self.lib.orc_unit_stream_chunk(_ptr(st.W), D, G, st.bits, _dtype_code(qc), st.budget,
                                           st.chunk, _ptr(st.K), _ptr(st.V), _ptr(st.codes),
                                           _ptr(occ), T, _ptr(qc), _ptr(kc), _ptr(vc),
                                           float(st.tau), _ptr(st.tauv), _ptr(evicted),
                                           _ptr(written), _ptr(wo), _ptr(out))
        elif st.Vq is not None:
            if st.score is None and decay != 0.0:
                raise ValueError("score memory needs a unit filled with memory=True")
            self.lib.orc_unit_stream_vq(_ptr(st.W), D, G, st.bits, _dtype_code(qc), st.budget,
                                        2 if st.Vq.dtype == np.uint8 else 1, _ptr(st.K),
                                        _ptr(st.Vq), _ptr(st.Vs), _ptr(st.codes),
                                        _ptr(st.score), _ptr(occ), T, _ptr(qc), _ptr(kc),
                                        _ptr(vc), float(st.tau), _ptr(st.tauv), float(decay),
                                        _ptr(evicted), _ptr(written), _ptr(wo), _ptr(out))
            if dist_log:
                raise ValueError("no distance log for the quantised value cache")
        elif st.score is None and st.tau == 0.0 and st.tauv is None:
            if decay != 0.0:
                raise ValueError("score memory needs a unit filled with memory=True")
            self.lib.orc_unit_stream(_ptr(st.W), D, G, st.bits, _dtype_code(qc), st.budget,
                                     _ptr(st.K), _ptr(st.V), _ptr(st.codes), _ptr(occ), T,
                                     _ptr(qc), _ptr(kc), _ptr(vc), _ptr(evicted), _ptr(written),
                                     _ptr(wo), _ptr(out), _ptr(dl))
        else:
            if st.score is None and decay != 0.0:
                raise ValueError("score memory needs a unit filled with memory=True")
            self.lib.orc_unit_stream_ext(_ptr(st.W), D, G, st.bits, _dtype_code(qc), st.budget,
                                         _ptr(st.K), _ptr(st.V), _ptr(st.codes), _ptr(st.score),
                                         _ptr(occ), T, _ptr(qc), _ptr(kc), _ptr(vc),
                                         float(st.tau), _ptr(st.tauv), float(decay),
                                         _ptr(evicted), _ptr(written), _ptr(wo), _ptr(out),
                                         _ptr(dl))
        st.occupancy = int(occ[0])
        res = {"evicted": evicted, "written": written, "out": out}
        if dist_log:
            res["dist"] = dl
        return res


_cache: dict[int, Oracle] = {}


def load(mutant: int = 0, build_dir: str | None = None) -> Oracle:
    """The oracle library (built on first use).  Mutants are built into
    ``build_dir`` (required for mutant > 0)."""
    if mutant in _cache:
        return _cache[mutant]
    if mutant == 0:
        path = build()
    else:
        if build_dir is None:
            raise ValueError("mutant builds need a build_dir")
        path = build(os.path.join(build_dir, f"liboracle_mutant{mutant}.so"), mutant)
    o = Oracle(path)
    _cache[mutant] = o
    return o
