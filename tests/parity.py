"""Helpers shared by the parity tests: build matching configs for the CUDA
path and the oracle (each from its own layer-step function), move encoded
objects between the two representations, and cut a layer range out of an
encoded object using the documented chunk-major layout."""
from __future__ import annotations

import math
import os

import numpy as np
import torch

from oracle import oracle as O

FIELDS = ["anchors", "scales", "tables", "table_off", "payload", "stream_off", "escapes", "esc_off"]
NP_DT = {"anchors": np.int8, "scales": np.float32, "tables": np.uint8, "table_off": np.uint32,
         "payload": np.uint8, "stream_off": np.uint64, "escapes": np.int32, "esc_off": np.uint32}


def nthreads() -> int:
    return max(1, os.cpu_count() or 1)


def configs(L, T, C, G=10, chunk=0, tps=1536, mult=1.0):
    """(product Config, oracle Config) for the same workload."""
    from kv_cache_compression_decode_gb300 import codec as Cd
    chunk = chunk or T
    return (Cd.Config(L, T, C, G, chunk, tps, Cd.layer_steps(L, mult=mult)),
            O.Config(L, T, C, G, chunk, tps, O.layer_steps(L, mult=mult)))


def gpu_to_np(enc) -> dict:
    """Product Encoded (device or host tensors, trimmed) -> flat numpy arrays."""
    out = {}
    for f in FIELDS:
        t = getattr(enc, f).detach().cpu().contiguous()
        out[f] = t.numpy().view(NP_DT[f]).reshape(-1)
    return out


def oracle_to_np(oenc: O.Encoded) -> dict:
    return {f: np.ascontiguousarray(getattr(oenc, f)).view(NP_DT[f]).reshape(-1) for f in FIELDS}


def upload(oenc: O.Encoded, device="cuda"):
    """Oracle object -> product Encoded of device tensors (payload 16-aligned)."""
    from kv_cache_compression_decode_gb300 import codec as Cd
    d = oracle_to_np(oenc)
    ts = []
    for f in FIELDS:
        a = d[f]
        view_dt = {np.uint32: np.int32, np.uint64: np.int64}.get(a.dtype.type, a.dtype.type)
        ts.append(torch.from_numpy(np.ascontiguousarray(a).view(view_dt).copy()).to(device))
    return Cd.Encoded(*ts, sizes={"payload_bytes": d["payload"].size, "tables_bytes": d["tables"].size,
                                  "n_escapes": d["escapes"].size, "total_bytes": oenc.total_bytes})


def assert_same_object(got: dict, exp: dict, what=""):
    for f in FIELDS:
        a, b = got[f], exp[f]
        assert a.shape == b.shape, f"{what} {f}: size {a.shape} vs {b.shape}"
        if not np.array_equal(a, b):
            bad = np.nonzero(a != b)[0]
            raise AssertionError(f"{what} {f}: {bad.size} differing entries, first at {bad[0]}: "
                                 f"{a[bad[0]]} vs {b[bad[0]]}")


class Geo:
    """Layout of an encoded object (chunk-major per-chunk sections)."""

    def __init__(self, L, T, C, G, chunk, tps):
        self.L, self.T, self.C, self.G = L, T, C, G
        self.chunk = min(chunk or T, T)
        self.tps = min(tps, self.chunk)
        self.n_chunks = math.ceil(T / self.chunk)
        self.lens = [min(self.chunk, T - ch * self.chunk) for ch in range(self.n_chunks)]
        self.apc = [math.ceil(n / G) for n in self.lens]
        self.spc = [math.ceil(n / self.tps) for n in self.lens]
        self.NG = C // 32
        self.S = 2 * L

    def row0(self, ch):
        return sum(self.apc[:ch]) * self.S

    def stream0(self, ch):
        return sum(self.spc[:ch]) * self.S * self.NG


def cut_layers(obj: dict, geo: Geo, l0: int, l1: int) -> dict:
    """Sections of layers [l0, l1) of an object, re-based as a standalone
    object of l1 - l0 layers."""
    C, NG, S = geo.C, geo.NG, geo.S
    s0, s1 = 2 * l0, 2 * l1
    anch = obj["anchors"]
    a_parts, p_parts, e_parts, so, eo = [], [], [], [0], [0]
    for ch in range(geo.n_chunks):
        base = geo.row0(ch)
        a_parts.append(anch[(base + s0 * geo.apc[ch]) * C:(base + s1 * geo.apc[ch]) * C])
        k0 = geo.stream0(ch) + s0 * geo.spc[ch] * NG
        k1 = geo.stream0(ch) + s1 * geo.spc[ch] * NG
        for k in range(k0, k1):
            b, e = int(obj["stream_off"][k]), int(obj["stream_off"][k + 1])
            p_parts.append(obj["payload"][b:e])
            so.append(so[-1] + (e - b))
            b, e = int(obj["esc_off"][k]), int(obj["esc_off"][k + 1])
            e_parts.append(obj["escapes"][b:e])
            eo.append(eo[-1] + (e - b))
    t0, t1 = s0 * C, s1 * C
    tb, te = int(obj["table_off"][t0]), int(obj["table_off"][t1])
    cat = lambda parts, dt: np.concatenate(parts).astype(dt) if parts else np.zeros(0, dt)
    return {"anchors": cat(a_parts, np.int8), "scales": obj["scales"][t0:t1].copy(),
            "tables": obj["tables"][tb:te].copy(),
            "table_off": (obj["table_off"][t0:t1 + 1] - np.uint32(tb)).astype(np.uint32),
            "payload": cat(p_parts, np.uint8), "stream_off": np.array(so, dtype=np.uint64),
            "escapes": cat(e_parts, np.int32), "esc_off": np.array(eo, dtype=np.uint32)}
