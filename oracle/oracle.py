"""ctypes wrapper of the plain CPU oracle in ``cgo.c``.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline / reference arm.  The product path never imports
this module, and it imports nothing from the product package.

Every function takes and returns numpy arrays; fp16 values travel as their
uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as ct
import dataclasses
import os
import subprocess
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cgo.c")
_LIB = os.path.join(_HERE, "libcgoracle.so")

OK, ERR_INVALID_ARG, ERR_NONFINITE, ERR_RANGE, ERR_CORRUPT = 0, 1, 2, 3, 4
ERR_NOMEM = 7
LANES = 32
ESC = 255
M = 65536


def build(force: bool = False) -> str:
    """Compile cgo.c into libcgoracle.so (IEEE fp32: no fast-math, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lpthread", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ct.Structure):
    _fields_ = [("L", ct.c_uint32), ("T", ct.c_uint32), ("C", ct.c_uint32), ("G", ct.c_uint32),
                ("chunk_tokens", ct.c_uint32), ("tokens_per_stream", ct.c_uint32),
                ("step", ct.POINTER(ct.c_float))]


class _Enc(ct.Structure):
    _fields_ = [("anchors", ct.c_void_p), ("scales", ct.c_void_p), ("tables", ct.c_void_p),
                ("table_off", ct.c_void_p), ("payload", ct.c_void_p), ("stream_off", ct.c_void_p),
                ("escapes", ct.c_void_p), ("esc_off", ct.c_void_p),
                ("tables_cap", ct.c_uint64), ("payload_cap", ct.c_uint64), ("escapes_cap", ct.c_uint64)]


class _Sizes(ct.Structure):
    _fields_ = [("payload_bytes", ct.c_uint64), ("tables_bytes", ct.c_uint64),
                ("n_escapes", ct.c_uint64), ("total_bytes", ct.c_uint64)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ct.CDLL(build())
        P = ct.c_void_p
        _lib.cgo_f16_to_f32.restype = ct.c_float
        _lib.cgo_f16_to_f32.argtypes = [ct.c_uint16]
        _lib.cgo_f32_to_f16.restype = ct.c_uint16
        _lib.cgo_f32_to_f16.argtypes = [ct.c_float]
        _lib.cgo_f32_to_f16_array.argtypes = [P, P, ct.c_uint64]
        _lib.cgo_f16_to_f32_array.argtypes = [P, P, ct.c_uint64]
        _lib.cgo_geometry.argtypes = [ct.POINTER(_Cfg), P]
        _lib.cgo_normalize.argtypes = [P, P, ct.POINTER(ct.c_int32), ct.POINTER(ct.c_int32)]
        _lib.cgo_rans_encode.argtypes = [ct.c_uint32, ct.c_uint32, P, P, P, ct.c_uint64, ct.POINTER(ct.c_uint64)]
        _lib.cgo_rans_decode.argtypes = [ct.c_uint32, ct.c_uint32, P, ct.c_uint64, P, P, P, P,
                                         ct.POINTER(ct.c_uint64)]
        _lib.cgo_encode.argtypes = [ct.POINTER(_Cfg), P, ct.POINTER(_Enc), ct.POINTER(_Sizes), ct.c_int]
        _lib.cgo_decode.argtypes = [ct.POINTER(_Cfg), ct.POINTER(_Enc), P, ct.c_int]
        _lib.cgo_anchor_scales.argtypes = [ct.POINTER(_Cfg), P, P]
        _lib.cgo_quantize.argtypes = [ct.POINTER(_Cfg), P, P, P, P]
        _lib.cgo_histograms.argtypes = [ct.POINTER(_Cfg), P, P]
        _lib.cgo_is_anchor.argtypes = [ct.POINTER(_Cfg), ct.c_uint32]
        _lib.cgo_layer_steps.argtypes = [ct.c_uint32, P, ct.c_float, P]
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def _check(code: int, what: str) -> None:
    if code != OK:
        raise OracleError(code, what)


@dataclasses.dataclass
class Config:
    L: int
    T: int
    C: int
    G: int
    chunk_tokens: int
    tokens_per_stream: int
    step: np.ndarray  # float32 [L]

    def c(self) -> _Cfg:
        self._step = np.ascontiguousarray(self.step, dtype=np.float32)
        return _Cfg(self.L, self.T, self.C, self.G, self.chunk_tokens, self.tokens_per_stream,
                    self._step.ctypes.data_as(ct.POINTER(ct.c_float)))


def layer_steps(L: int, base: Sequence[float] = (0.5, 1.0, 1.5), mult: float = 1.0) -> np.ndarray:
    """Per-layer step: base[floor(3 l / L)] * mult (layer thirds)."""
    b = np.asarray(base, dtype=np.float32)
    out = np.empty(L, dtype=np.float32)
    lib().cgo_layer_steps(L, _p(b), ct.c_float(mult), _p(out))
    return out


def geometry(cfg: Config) -> dict:
    out = np.zeros(7, dtype=np.uint64)
    _check(lib().cgo_geometry(ct.byref(cfg.c()), _p(out)), "geometry")
    keys = ["A", "spans_total", "n_streams", "n_tables", "tables_max_bytes", "payload_max_bytes",
            "escapes_max_count"]
    return {k: int(v) for k, v in zip(keys, out)}


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().cgo_f16_to_f32_array(_p(h), _p(out), h.size)
    return out


def f32_to_f16(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    lib().cgo_f32_to_f16_array(_p(f), _p(out), f.size)
    return out


def normalize(counts: np.ndarray) -> Tuple[np.ndarray, int, int]:
    n = np.ascontiguousarray(counts, dtype=np.uint32)
    assert n.shape == (256,)
    f = np.zeros(256, dtype=np.uint32)
    lo, hi = ct.c_int32(), ct.c_int32()
    _check(lib().cgo_normalize(_p(n), _p(f), ct.byref(lo), ct.byref(hi)), "normalize")
    return f, lo.value, hi.value


def rans_encode(sym: np.ndarray, freq: np.ndarray) -> np.ndarray:
    """sym [steps][lanes] uint8, freq [lanes][256] -> uint16 words."""
    sym = np.ascontiguousarray(sym, dtype=np.uint8)
    steps, lanes = sym.shape
    freq = np.ascontiguousarray(freq, dtype=np.uint32)
    assert freq.shape == (lanes, 256)
    cap = (steps + 2) * lanes
    out = np.zeros(max(cap, 1), dtype=np.uint16)
    n = ct.c_uint64()
    _check(lib().cgo_rans_encode(lanes, steps, _p(sym), _p(freq), _p(out), cap, ct.byref(n)), "rans_encode")
    return out[: n.value].copy()


def rans_decode(words: np.ndarray, steps: int, freq: np.ndarray, lo=None, hi=None) -> Tuple[np.ndarray, int]:
    words = np.ascontiguousarray(words, dtype=np.uint16)
    freq = np.ascontiguousarray(freq, dtype=np.uint32)
    lanes = freq.shape[0]
    if lo is None:
        lo = np.array([int(np.nonzero(f)[0].min()) if f.any() else 1 for f in freq], dtype=np.int32)
        hi = np.array([int(np.nonzero(f)[0].max()) if f.any() else 0 for f in freq], dtype=np.int32)
    lo = np.ascontiguousarray(lo, dtype=np.int32)
    hi = np.ascontiguousarray(hi, dtype=np.int32)
    sym = np.zeros((max(steps, 1), lanes), dtype=np.uint8)
    used = ct.c_uint64()
    wp = _p(words) if words.size else 0
    _check(lib().cgo_rans_decode(lanes, steps, wp, words.size, _p(freq), _p(lo), _p(hi), _p(sym),
                                 ct.byref(used)), "rans_decode")
    return sym[:steps], used.value


@dataclasses.dataclass
class Encoded:
    anchors: np.ndarray     # int8, chunk-major [chunk][L][2][anchor rows of the chunk][C]
                            # (the array is shaped [L][2][A][C] only for its size)
    scales: np.ndarray      # float32 [L][2][C]
    tables: np.ndarray      # uint8 [tables_bytes]
    table_off: np.ndarray   # uint32 [n_tables + 1]
    payload: np.ndarray     # uint8 [payload_bytes]
    stream_off: np.ndarray  # uint64 [n_streams + 1]
    escapes: np.ndarray     # int32 [n_escapes]
    esc_off: np.ndarray     # uint32 [n_streams + 1]
    total_bytes: int = 0

    def _c(self) -> _Enc:
        def ptr(a):
            return _p(a) if a.size else _p(np.zeros(1, dtype=a.dtype))
        self._keep = [self.escapes if self.escapes.size else np.zeros(1, np.int32),
                      self.payload if self.payload.size else np.zeros(16, np.uint8)]
        return _Enc(_p(self.anchors), _p(self.scales), _p(self.tables), _p(self.table_off),
                    _p(self._keep[1]), _p(self.stream_off), _p(self._keep[0]),
                    _p(self.esc_off), self.tables.size, self.payload.size, self.escapes.size)


def encode(cfg: Config, kv: np.ndarray, nthreads: int = 1) -> Encoded:
    """Encode kv [L][2][T][C] (uint16 fp16 bits)."""
    kv = np.ascontiguousarray(kv)
    if kv.dtype == np.float16:
        kv = kv.view(np.uint16)
    assert kv.dtype == np.uint16 and kv.shape == (cfg.L, 2, cfg.T, cfg.C)
    geo = geometry(cfg)
    A = geo["A"]
    anchors = np.zeros((cfg.L, 2, A, cfg.C), dtype=np.int8)
    scales = np.zeros((cfg.L, 2, cfg.C), dtype=np.float32)
    tables = np.zeros(geo["tables_max_bytes"], dtype=np.uint8)
    table_off = np.zeros(geo["n_tables"] + 1, dtype=np.uint32)
    payload = np.zeros(max(geo["payload_max_bytes"], 16), dtype=np.uint8)
    stream_off = np.zeros(geo["n_streams"] + 1, dtype=np.uint64)
    esc_off = np.zeros(geo["n_streams"] + 1, dtype=np.uint32)
    esc_cap = min(geo["escapes_max_count"], cfg.L * 2 * cfg.T * cfg.C // 64 + 4096)
    cc = cfg.c()
    for attempt in range(2):
        escapes = np.zeros(max(esc_cap, 1), dtype=np.int32)
        enc = _Enc(_p(anchors), _p(scales), _p(tables), _p(table_off), _p(payload), _p(stream_off),
                   _p(escapes), _p(esc_off), tables.size, payload.size, esc_cap)
        sz = _Sizes()
        code = lib().cgo_encode(ct.byref(cc), _p(kv), ct.byref(enc), ct.byref(sz), nthreads)
        if code == ERR_RANGE and attempt == 0:
            esc_cap = geo["escapes_max_count"]
            continue
        _check(code, "encode")
        break
    return Encoded(anchors, scales, tables[: sz.tables_bytes].copy(), table_off,
                   payload[: sz.payload_bytes].copy(), stream_off, escapes[: sz.n_escapes].copy(), esc_off,
                   int(sz.total_bytes))


def decode(cfg: Config, enc: Encoded, nthreads: int = 1) -> np.ndarray:
    out = np.zeros((cfg.L, 2, cfg.T, cfg.C), dtype=np.uint16)
    cc = cfg.c()
    e = enc._c()
    _check(lib().cgo_decode(ct.byref(cc), ct.byref(e), _p(out), nthreads), "decode")
    return out


def anchor_scales(cfg: Config, kv: np.ndarray) -> np.ndarray:
    kv = np.ascontiguousarray(kv).view(np.uint16)
    out = np.zeros((cfg.L, 2, cfg.C), dtype=np.float32)
    _check(lib().cgo_anchor_scales(ct.byref(cfg.c()), _p(kv), _p(out)), "anchor_scales")
    return out


def quantize(cfg: Config, kv: np.ndarray, scales: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    kv = np.ascontiguousarray(kv).view(np.uint16)
    A = geometry(cfg)["A"]
    anchors = np.zeros((cfg.L, 2, A, cfg.C), dtype=np.int8)
    q = np.zeros((cfg.L, 2, cfg.T, cfg.C), dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    _check(lib().cgo_quantize(ct.byref(cfg.c()), _p(kv), _p(scales), _p(anchors), _p(q)), "quantize")
    return anchors, q


def histograms(cfg: Config, q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int32)
    out = np.zeros((cfg.L * 2 * cfg.C, 256), dtype=np.uint32)
    _check(lib().cgo_histograms(ct.byref(cfg.c()), _p(q), _p(out)), "histograms")
    return out


def anchor_mask(cfg: Config) -> np.ndarray:
    cc = cfg.c()
    return np.array([bool(lib().cgo_is_anchor(ct.byref(cc), t)) for t in range(cfg.T)])


def parse_tables(enc: Encoded, n_tables: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Compact tables -> (freq [n][256] uint32, lo [n], hi [n])."""
    freq = np.zeros((n_tables, 256), dtype=np.uint32)
    lo = np.zeros(n_tables, dtype=np.int32)
    hi = np.zeros(n_tables, dtype=np.int32)
    for i in range(n_tables):
        b, e = int(enc.table_off[i]), int(enc.table_off[i + 1])
        lo[i], hi[i] = int(enc.tables[b]), int(enc.tables[b + 1])
        if lo[i] <= hi[i]:
            fm1 = enc.tables[b + 2: e].view(np.uint16).astype(np.uint32)
            freq[i, lo[i]: hi[i] + 1] = fm1 + 1
    return freq, lo, hi
