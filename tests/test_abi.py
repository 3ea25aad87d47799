"""Host-side checks of the C ABI (no GPU, no kernel launch)."""
import ctypes as ct
import os
import re

import numpy as np
import pytest
import torch

from oracle import oracle as O
from kv_cache_compression_decode_gb300 import codec as C
from tests import parity as P

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "cg.h")


def declared_functions():
    text = open(HDR).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cg_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 11
    lib = C.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(C.EXPORTS)


CASES = [(4, 256, 1024, 10, 0, 1536), (2, 300, 64, 10, 128, 64), (1, 1, 32, 10, 1, 1), (2, 57, 96, 1, 57, 20),
         (3, 1000, 128, 7, 333, 100), (80, 16384, 1024, 10, 0, 1536), (32, 16384, 1024, 10, 1536, 1536),
         (2, 4100, 64, 10, 0, 1536)]


@pytest.mark.parametrize("L,T,Cc,G,chunk,tps", CASES)
def test_bounds_match_oracle_geometry(L, T, Cc, G, chunk, tps):
    pc, oc = P.configs(L, T, Cc, G, chunk, tps)
    b = C.cg_encode_bounds(pc)
    g = O.geometry(oc)
    assert b["A"] == g["A"]
    assert b["spans_total"] == g["spans_total"]
    assert b["n_streams"] == g["n_streams"]
    assert b["n_tables"] == g["n_tables"]
    assert b["tables_max_bytes"] == g["tables_max_bytes"]
    assert b["payload_max_bytes"] == g["payload_max_bytes"]
    assert b["escapes_max_count"] == g["escapes_max_count"]
    assert b["anchors_bytes"] == 2 * L * g["A"] * Cc


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 32, 48, 80, 1024])
@pytest.mark.parametrize("mult", [1.0, 2.0, 4.0])
def test_layer_steps_product_matches_oracle(L, mult):
    assert np.array_equal(C.layer_steps(L, mult=mult), O.layer_steps(L, mult=mult))


def _cfg(**kw):
    d = dict(L=2, T=100, C=64, group_size=10, chunk_tokens=100, tokens_per_stream=50)
    d.update(kw)
    step = np.array(kw.pop("step", [0.5] * d["L"]), dtype=np.float32)
    d.pop("step", None)
    return C.Config(d["L"], d["T"], d["C"], d["group_size"], d["chunk_tokens"], d["tokens_per_stream"], step)


@pytest.mark.parametrize("kw", [dict(C=48), dict(C=0), dict(T=0), dict(group_size=0), dict(tokens_per_stream=0),
                                dict(step=[0.5, 2.0 ** -10]), dict(step=[0.5, float("nan")]),
                                dict(step=[0.5, float("inf")]), dict(step=[0.5, -1.0])])
def test_invalid_config_rejected_on_host(kw):
    cfg = _cfg(**kw)
    b = C.cg_bounds()
    assert C.lib().cg_encode_bounds(ct.byref(cfg.c()), ct.byref(b)) == C.CG_ERR_INVALID_ARG
    enc = C.cg_encoded()
    sz = C.cg_sizes()
    # rejected before any CUDA call: no GPU is needed to get the status back
    assert C.lib().cg_encode(ct.byref(cfg.c()), 1, 256, 1 << 20, ct.byref(enc), ct.byref(sz), 0, None) \
        == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_decode(ct.byref(cfg.c()), ct.byref(enc), 1, 0, None) == C.CG_ERR_INVALID_ARG


def test_too_many_layers_rejected():
    cfg = _cfg(L=1025, step=[0.5] * 1025)
    b = C.cg_bounds()
    assert C.lib().cg_encode_bounds(ct.byref(cfg.c()), ct.byref(b)) == C.CG_ERR_INVALID_ARG


def test_null_buffers_rejected():
    cfg = _cfg()
    enc = C.cg_encoded()
    sz = C.cg_sizes()
    assert C.lib().cg_encode(ct.byref(cfg.c()), None, 256, 1 << 20, ct.byref(enc), ct.byref(sz), 0, None) \
        == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_decode(ct.byref(cfg.c()), ct.byref(enc), 0, 0, None) == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_test_decode_timeout(ct.byref(cfg.c()), ct.byref(enc), 0, 0, None) == C.CG_ERR_INVALID_ARG
    n = ct.c_size_t()
    assert C.lib().cg_decode_chunks_ws_bytes(None, 0, ct.byref(n)) == C.CG_ERR_INVALID_ARG


_SECTIONS = ["anchors", "scales", "tables", "table_off", "payload", "stream_off", "escapes", "esc_off"]
_ALIGN = {"scales": 4, "tables": 2, "table_off": 4, "payload": 16, "stream_off": 8, "escapes": 4, "esc_off": 4}


def _fake_object(shift=None):
    """A cg_encoded of made-up, never dereferenced addresses (each 4 KiB
    apart), optionally with one section moved off its alignment."""
    ptrs = {f: (1 << 24) + 4096 * i for i, f in enumerate(_SECTIONS)}
    if shift:
        ptrs[shift[0]] += shift[1]
    return C.cg_encoded(*[ptrs[f] for f in _SECTIONS], 1 << 16, 1 << 20, 1 << 16)


@pytest.mark.parametrize("field,off", [(f, o) for f, a in _ALIGN.items() for o in sorted({1, a // 2})])
def test_misaligned_sections_refused_on_host(field, off):
    """Each section sits at an address aligned to its element type (the
    payload to 16 bytes).  A misaligned one is refused before anything is
    enqueued.  Controls with every section aligned show that the refusal
    comes from the alignment: the encoder then stops at its workspace-size
    check (RANGE, still on the host), and the chunk planner, which runs on
    the host alone, accepts the object."""
    cfg = _cfg(L=2, T=100, C=64, chunk_tokens=50, tokens_per_stream=50)
    sz = C.cg_sizes()
    kv = ws = dst = 1 << 30
    ok, bad = _fake_object(), _fake_object((field, off))
    assert C.lib().cg_encode(ct.byref(cfg.c()), kv, ws, 1, ct.byref(ok), ct.byref(sz), 0, None) == C.CG_ERR_RANGE
    assert C.lib().cg_encode(ct.byref(cfg.c()), kv, ws, 1, ct.byref(bad), ct.byref(sz), 0, None) \
        == C.CG_ERR_INVALID_ARG
    n = ct.c_size_t()
    for enc, want in ((ok, C.CG_OK), (bad, C.CG_ERR_INVALID_ARG)):
        ref = (C.cg_chunk_ref * 1)(C.cg_chunk_ref(ct.pointer(cfg.c()), ct.pointer(enc), 1, dst, 100, 50))
        assert C.lib().cg_decode_chunks_ws_bytes(ref, 1, ct.byref(n)) == want
    # cg_decode has no host-only control: with every section aligned it would launch
    assert C.lib().cg_decode(ct.byref(cfg.c()), ct.byref(bad), dst, 0, None) == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_test_decode_timeout(ct.byref(cfg.c()), ct.byref(bad), dst, 0, None) == C.CG_ERR_INVALID_ARG


def test_cache_source_host_checks():
    """cg_cache_source refuses null arguments; without a usable device the
    pointer query itself fails (CUDA error), and nothing is reported usable."""
    mt, view = ct.c_int(7), ct.c_void_p(1)
    assert C.lib().cg_cache_source(None, ct.byref(mt), ct.byref(view)) == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_cache_source(256, None, ct.byref(view)) == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_cache_source(256, ct.byref(mt), None) == C.CG_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        code = C.lib().cg_cache_source(256, ct.byref(mt), ct.byref(view))
        assert code == C.CG_ERR_CUDA and view.value is None


def test_status_strings_and_flags():
    for code in range(7):
        assert C.cg_status_string(code)
    assert C.cg_status_string(99) == "unknown status"
    assert C.cg_status_from_flags(0) == C.CG_OK
    assert C.cg_status_from_flags(1 << C.CG_ERR_CORRUPT) == C.CG_ERR_CORRUPT
    assert C.cg_status_from_flags((1 << C.CG_ERR_CORRUPT) | (1 << C.CG_ERR_NONFINITE)) == C.CG_ERR_NONFINITE


def _host_encoded(d, oenc):
    def t(a):
        view = {np.uint32: np.int32, np.uint64: np.int64}.get(a.dtype.type, a.dtype.type)
        return torch.from_numpy(np.ascontiguousarray(a).view(view).copy())
    return C.Encoded(*[t(d[f]) for f in P.FIELDS],
                     sizes={"payload_bytes": d["payload"].size, "tables_bytes": d["tables"].size,
                            "n_escapes": d["escapes"].size, "total_bytes": oenc.total_bytes})


def test_serialize_round_trip_of_an_oracle_object():
    from kv_cache_compression_decode_gb300 import synth
    L, T, Cc = 2, 333, 64
    pc, oc = P.configs(L, T, Cc, 10, 100, 64)
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=3).numpy()
    x[0, 0, 7, 3] = 300.0  # an escape
    oenc = O.encode(oc, x)
    d = P.oracle_to_np(oenc)
    host = _host_encoded(d, oenc)
    buf = C.cg_serialize(pc, host)
    assert buf[:4] == b"CGKV"
    cfg2, back = C.cg_deserialize(buf)
    assert (cfg2.L, cfg2.T, cfg2.C, cfg2.group_size, cfg2.chunk_tokens, cfg2.tokens_per_stream) == \
        (L, T, Cc, 10, 100, 64)
    assert np.array_equal(cfg2.step, pc.step)
    P.assert_same_object(P.gpu_to_np(back), d, "deserialized")
    bad = bytearray(buf)
    bad[0] = ord("X")
    with pytest.raises(C.CodecError) as e:
        C.cg_deserialize(bytes(bad))
    assert e.value.code == C.CG_ERR_CORRUPT
    with pytest.raises(C.CodecError):
        C.cg_deserialize(buf[: len(buf) // 2])


def test_chunk_ranges_partition_the_sections():
    from kv_cache_compression_decode_gb300 import synth
    L, T, Cc, chunk, tps = 3, 1000, 64, 300, 128
    pc, oc = P.configs(L, T, Cc, 10, chunk, tps)
    x = synth.ar1_kv(L, T, Cc, 0.9, 1, seed=5).numpy()
    oenc = O.encode(oc, x)
    geo = P.Geo(L, T, Cc, 10, chunk, tps)
    prev = None
    for ch in range(geo.n_chunks):
        r = C.cg_chunk_ranges(pc, ch, oenc.stream_off, oenc.esc_off)
        assert r["stream_begin"] == geo.stream0(ch)
        assert r["anchor_begin"] == geo.row0(ch) * Cc
        assert r["anchor_end"] - r["anchor_begin"] == 2 * L * geo.apc[ch] * Cc
        if prev:
            for k in ("stream", "payload", "escape", "anchor"):
                assert r[k + "_begin"] == prev[k + "_end"]
        prev = r
    assert prev["payload_end"] == oenc.payload.size
    assert prev["anchor_end"] == oenc.anchors.size
    assert prev["stream_end"] == oenc.stream_off.size - 1


def test_decode_chunks_plan_sizes_on_host():
    pc, _ = P.configs(2, 1000, 64, 10, 300, 128)
    enc = C.alloc_encoded(pc, device="cpu")
    dst = torch.empty((2, 2, 1000, 64), dtype=torch.float16)
    refs = [C.ChunkRef(pc, enc, ch, dst, ch * 300) for ch in range(4)]
    assert C.cg_decode_chunks_ws_bytes(refs) > 0
    with pytest.raises(C.CodecError):  # chunk out of range
        C.cg_decode_chunks_ws_bytes([C.ChunkRef(pc, enc, 4, dst, 0)])
    with pytest.raises(C.CodecError):  # destination too short for the chunk
        C.cg_decode_chunks_ws_bytes([C.ChunkRef(pc, enc, 0, dst, 800)])


@pytest.mark.parametrize("bt,nb", [(12, 100), (8, 200), (16, 62), (0, 100)])
def test_paged_decode_rejects_bad_layouts_on_host(bt, nb):
    """block_tokens must be a power of two >= group_size and the blocks must
    cover T; checked before anything is enqueued (no GPU needed)."""
    pc, _ = P.configs(2, 1000, 64, 10, 0, 128)
    enc = C.alloc_encoded(pc, device="cpu")
    pool = torch.empty(1 << 16, dtype=torch.float16)
    table = torch.zeros(nb, dtype=torch.int32)
    with pytest.raises(C.CodecError) as e:
        C.cg_decode_paged(pc, enc, pool, table, bt, 0, 0, 0, 64, torch.zeros(1, dtype=torch.int32))
    assert e.value.code == C.CG_ERR_INVALID_ARG


def test_multi_level_encode_host_checks():
    pc, _ = P.configs(2, 1000, 64, 10, 0, 128)
    one = C.cg_encode_levels_ws_bytes(pc, 1)
    assert one == C.cg_encode_bounds(pc)["workspace_bytes"]
    assert one < C.cg_encode_levels_ws_bytes(pc, 2) < C.cg_encode_levels_ws_bytes(pc, 4)
    for bad in (0, 5):
        with pytest.raises(C.CodecError):
            C.cg_encode_levels_ws_bytes(pc, bad)
    # a level whose steps would fall to 2^-10 or below is rejected before any work
    outs = [C.alloc_encoded(pc, device="cpu") for _ in range(2)]
    arr = (C.cg_encoded * 2)(*[o.c() for o in outs])
    sizes = (C.cg_sizes * 2)()
    mult = np.array([1.0, 1e-4], np.float32)
    code = C.lib().cg_encode_levels(ct.byref(pc.c()), 2, mult.ctypes.data, 256, 256, 1 << 30, arr,
                                    ct.addressof(sizes), 0, None)
    assert code == C.CG_ERR_INVALID_ARG
    # the cache is read in 16-byte pieces: with every other argument valid,
    # a cache that is only 2-byte aligned is refused before any CUDA call
    mult = np.array([1.0, 2.0], np.float32)
    for kv in (258, 264):
        code = C.lib().cg_encode_levels(ct.byref(pc.c()), 2, mult.ctypes.data, kv, 256, 1 << 30, arr,
                                        ct.addressof(sizes), 0, None)
        assert code == C.CG_ERR_INVALID_ARG
        code = C.lib().cg_encode(ct.byref(pc.c()), kv, 256, 1 << 30, ct.byref(arr[0]), ct.byref(sizes[0]), 0, None)
        assert code == C.CG_ERR_INVALID_ARG


def test_ablation_host_checks():
    """cg_ablation sizes its workspace and rejects bad arguments before any
    GPU work (no GPU needed)."""
    pc, _ = P.configs(2, 1000, 64, 10, 0, 128)
    n = ct.c_size_t()
    assert C.lib().cg_ablation_ws_bytes(ct.byref(pc.c()), ct.byref(n)) == C.CG_OK
    assert n.value >= C.cg_encode_bounds(pc)["workspace_bytes"]
    assert C.lib().cg_ablation_ws_bytes(ct.byref(pc.c()), None) == C.CG_ERR_INVALID_ARG
    ws = 256
    # null cache, null output, misaligned workspace, too small a workspace
    assert C.lib().cg_ablation(ct.byref(pc.c()), None, ws, n.value, 256, 0, None) == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_ablation(ct.byref(pc.c()), 256, ws, n.value, None, 0, None) == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_ablation(ct.byref(pc.c()), 256, ws + 8, n.value, 256, 0, None) == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_ablation(ct.byref(pc.c()), 264, ws, n.value, 256, 0, None) == C.CG_ERR_INVALID_ARG
    assert C.lib().cg_ablation(ct.byref(pc.c()), 256, ws, n.value - 1, 256, 0, None) == C.CG_ERR_RANGE
