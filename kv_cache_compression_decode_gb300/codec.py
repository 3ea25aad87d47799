"""Python binding of libcg (the codec's C ABI in include/cg.h).

Argument marshalling only: every step of the codec runs in libcg's CUDA
kernels.  PyTorch supplies device memory, pinned host memory and streams.
The functions keep the C names (cg_encode, cg_decode, ...); a few helpers
(`alloc_encoded`, `encode`, `decode`) only size and allocate buffers around
those calls.  There is no CPU fallback: if libcg.so cannot be built or loaded,
every call raises.
"""
from __future__ import annotations

import ctypes as ct
import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import build as _build

CG_OK, CG_ERR_INVALID_ARG, CG_ERR_NONFINITE, CG_ERR_RANGE = 0, 1, 2, 3
CG_ERR_CORRUPT, CG_ERR_TIMEOUT, CG_ERR_CUDA = 4, 5, 6
CG_MAX_LAYERS = 1024

# Step per layer third: shallow / middle / deep ("CacheGen vs 传统量化KV缓存压缩
# 技术深度对比与性能测试", §1 and §2.1, layer-sensitive quantization).
LAYER_BASE_STEPS = (0.5, 1.0, 1.5)


def layer_steps(L: int, base: Sequence[float] = LAYER_BASE_STEPS, mult: float = 1.0) -> np.ndarray:
    """Quantization step of each layer: base[floor(3 l / L)] * mult, fp32."""
    b = np.asarray(base, dtype=np.float32)
    return np.array([b[(3 * l) // L] * np.float32(mult) for l in range(L)], dtype=np.float32)


class cg_config(ct.Structure):
    _fields_ = [("L", ct.c_uint32), ("T", ct.c_uint32), ("C", ct.c_uint32), ("group_size", ct.c_uint32),
                ("chunk_tokens", ct.c_uint32), ("tokens_per_stream", ct.c_uint32),
                ("step", ct.POINTER(ct.c_float))]


class cg_bounds(ct.Structure):
    _fields_ = [(n, ct.c_uint64) for n in (
        "A", "n_chunks", "spans_total", "n_streams", "n_tables", "anchors_bytes", "scales_bytes",
        "table_off_bytes", "tables_max_bytes", "stream_off_bytes", "payload_max_bytes", "esc_off_bytes",
        "escapes_max_count", "workspace_bytes")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class cg_encoded(ct.Structure):
    _fields_ = [("anchors", ct.c_void_p), ("scales", ct.c_void_p), ("tables", ct.c_void_p),
                ("table_off", ct.c_void_p), ("payload", ct.c_void_p), ("stream_off", ct.c_void_p),
                ("escapes", ct.c_void_p), ("esc_off", ct.c_void_p), ("tables_cap", ct.c_uint64),
                ("payload_cap", ct.c_uint64), ("escapes_cap", ct.c_uint64)]


class cg_sizes(ct.Structure):
    _fields_ = [("payload_bytes", ct.c_uint64), ("tables_bytes", ct.c_uint64), ("n_escapes", ct.c_uint64),
                ("total_bytes", ct.c_uint64)]


class cg_chunk_ref(ct.Structure):
    _fields_ = [("cfg", ct.POINTER(cg_config)), ("enc", ct.POINTER(cg_encoded)), ("chunk", ct.c_uint32),
                ("dst", ct.c_void_p), ("dst_tokens", ct.c_uint32), ("dst_token0", ct.c_uint32)]


class cg_chunk_range(ct.Structure):
    _fields_ = [(n, ct.c_uint64) for n in (
        "stream_begin", "stream_end", "payload_begin", "payload_end", "escape_begin", "escape_end",
        "anchor_begin", "anchor_end")]


class cg_paged_kv(ct.Structure):
    _fields_ = [("pool", ct.c_void_p), ("block_table", ct.c_void_p), ("n_blocks", ct.c_uint32),
                ("n_pool_blocks", ct.c_uint32), ("block_tokens", ct.c_uint32), ("layer_stride", ct.c_uint64),
                ("kv_stride", ct.c_uint64), ("block_stride", ct.c_uint64), ("token_stride", ct.c_uint64)]


ABLATION_FIELDS = ("values", "delta_bits_channel", "delta_bits_slice", "delta_bits_global", "escape_bits",
                   "anchor_bits_raw", "anchor_bits_channel")


class cg_level_plan(ct.Structure):
    _fields_ = [("n_chunks", ct.c_uint32), ("n_levels", ct.c_uint32), ("bytes", ct.c_void_p),
                ("decode_s", ct.c_void_p), ("bw", ct.c_void_p), ("n_slots", ct.c_uint32), ("slot_s", ct.c_double),
                ("slo_s", ct.c_double)]


class cg_chunk_time(ct.Structure):
    _fields_ = [("arrive_s", ct.c_double), ("done_s", ct.c_double)]


# Every symbol libcg exports (the declarations of include/cg.h).
EXPORTS = ("cg_status_string", "cg_status_from_flags", "cg_encode_bounds", "cg_encode", "cg_decode",
           "cg_decode_chunks_ws_bytes", "cg_decode_chunks", "cg_decode_chunks_noalloc", "cg_chunk_ranges",
           "cg_serialize",
           "cg_deserialize_header", "cg_deserialize", "cg_plan_levels", "cg_decode_paged",
           "cg_encode_levels_ws_bytes", "cg_encode_levels", "cg_ablation_ws_bytes", "cg_ablation",
           "cg_cache_source", "cg_test_decode_timeout")

_lib = None


def lib() -> ct.CDLL:
    """Load libcg.so (building it first if its sources are newer)."""
    global _lib
    if _lib is None:
        L = ct.CDLL(_build.build())
        P, U32, U64 = ct.c_void_p, ct.c_uint32, ct.c_uint64
        L.cg_status_string.restype = ct.c_char_p
        L.cg_status_string.argtypes = [ct.c_int]
        L.cg_status_from_flags.argtypes = [U32]
        L.cg_encode_bounds.argtypes = [ct.POINTER(cg_config), ct.POINTER(cg_bounds)]
        L.cg_encode.argtypes = [ct.POINTER(cg_config), P, P, ct.c_size_t, ct.POINTER(cg_encoded),
                                ct.POINTER(cg_sizes), P, P]
        L.cg_decode.argtypes = [ct.POINTER(cg_config), ct.POINTER(cg_encoded), P, P, P]
        L.cg_test_decode_timeout.argtypes = [ct.POINTER(cg_config), ct.POINTER(cg_encoded), P, P, P]
        L.cg_decode_chunks_ws_bytes.argtypes = [ct.POINTER(cg_chunk_ref), U32, ct.POINTER(ct.c_size_t)]
        L.cg_decode_chunks.argtypes = [ct.POINTER(cg_chunk_ref), U32, P, ct.c_size_t, P, P]
        L.cg_decode_chunks_noalloc.argtypes = [ct.POINTER(cg_chunk_ref), U32, P, P]
        L.cg_chunk_ranges.argtypes = [ct.POINTER(cg_config), U32, P, P, ct.POINTER(cg_chunk_range)]
        L.cg_serialize.argtypes = [ct.POINTER(cg_config), ct.POINTER(cg_encoded), ct.POINTER(cg_sizes), P,
                                   ct.POINTER(ct.c_size_t)]
        L.cg_deserialize_header.argtypes = [P, ct.c_size_t, ct.POINTER(cg_config), P, ct.POINTER(cg_sizes)]
        L.cg_deserialize.argtypes = [P, ct.c_size_t, ct.POINTER(cg_encoded)]
        L.cg_plan_levels.argtypes = [ct.POINTER(cg_level_plan), P, P, ct.POINTER(ct.c_double)]
        L.cg_encode_levels_ws_bytes.argtypes = [ct.POINTER(cg_config), U32, ct.POINTER(ct.c_size_t)]
        L.cg_ablation_ws_bytes.argtypes = [ct.POINTER(cg_config), ct.POINTER(ct.c_size_t)]
        L.cg_ablation.argtypes = [ct.POINTER(cg_config), P, P, ct.c_size_t, P, P, P]
        L.cg_encode_levels.argtypes = [ct.POINTER(cg_config), U32, P, P, P, ct.c_size_t, P, P, P, P]
        L.cg_decode_paged.argtypes = [ct.POINTER(cg_config), ct.POINTER(cg_encoded), ct.POINTER(cg_paged_kv), P, P]
        L.cg_cache_source.argtypes = [P, ct.POINTER(ct.c_int), ct.POINTER(ct.c_void_p)]
        for name in EXPORTS:
            if name not in ("cg_status_string",):
                getattr(L, name).restype = ct.c_int
        _lib = L
    return _lib


class CodecError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {cg_status_string(code)} ({code})")
        self.code = code


def cg_status_string(code: int) -> str:
    return lib().cg_status_string(int(code)).decode()


def cg_status_from_flags(flags: int) -> int:
    return int(lib().cg_status_from_flags(int(flags) & 0xFFFFFFFF))


def _check(code: int, what: str) -> None:
    if code != CG_OK:
        raise CodecError(code, what)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


@dataclasses.dataclass
class Config:
    """Codec configuration (mirrors cg_config); `step` is the per-layer step."""
    L: int
    T: int
    C: int
    group_size: int = 10
    chunk_tokens: int = 0          # 0: one chunk covering all T tokens
    tokens_per_stream: int = 1536
    step: Optional[np.ndarray] = None

    def __post_init__(self):
        if self.step is None:
            self.step = layer_steps(self.L)
        self.step = np.ascontiguousarray(self.step, dtype=np.float32)
        if not self.chunk_tokens:
            self.chunk_tokens = self.T
        self._c = cg_config(self.L, self.T, self.C, self.group_size, self.chunk_tokens, self.tokens_per_stream,
                            self.step.ctypes.data_as(ct.POINTER(ct.c_float)))

    def c(self) -> cg_config:
        return self._c


def cg_encode_bounds(cfg: Config) -> dict:
    b = cg_bounds()
    _check(lib().cg_encode_bounds(ct.byref(cfg.c()), ct.byref(b)), "cg_encode_bounds")
    return b.as_dict()


@dataclasses.dataclass
class Encoded:
    """The sections of an encoded object as torch tensors (device or host)."""
    anchors: torch.Tensor     # int8
    scales: torch.Tensor      # float32
    tables: torch.Tensor      # uint8
    table_off: torch.Tensor   # int32 (u32 bits)
    payload: torch.Tensor     # uint8
    stream_off: torch.Tensor  # int64 (u64 bits)
    escapes: torch.Tensor     # int32
    esc_off: torch.Tensor     # int32 (u32 bits)
    sizes: Optional[dict] = None

    def c(self) -> cg_encoded:
        def ptr(t):
            return t.data_ptr() if t.numel() else None
        self._c = cg_encoded(ptr(self.anchors), ptr(self.scales), ptr(self.tables), ptr(self.table_off),
                             ptr(self.payload), ptr(self.stream_off), ptr(self.escapes), ptr(self.esc_off),
                             self.tables.numel(), self.payload.numel(), self.escapes.numel())
        return self._c

    def fields(self):
        return ["anchors", "scales", "tables", "table_off", "payload", "stream_off", "escapes", "esc_off"]

    def to(self, device, non_blocking=False) -> "Encoded":
        kw = dict(device=device, non_blocking=non_blocking)
        e = Encoded(*[getattr(self, f).to(**kw) for f in self.fields()], sizes=self.sizes)
        return e

    def trimmed(self) -> "Encoded":
        """Views cut to the actual sizes (after an encode has completed)."""
        s = self.sizes
        return Encoded(self.anchors, self.scales, self.tables[: s["tables_bytes"]], self.table_off,
                       self.payload[: s["payload_bytes"]], self.stream_off, self.escapes[: s["n_escapes"]],
                       self.esc_off, sizes=s)


@dataclasses.dataclass
class RawEncoded:
    """An encoded object given as raw device addresses and capacities (a
    cg_encoded as such).  Used to point the per-chunk sections at a staging
    buffer that holds only some chunks: the section base is the staging
    address minus the chunk range's start, so that base + offset lands in
    the staged bytes, and the capacity is the range's end."""
    anchors: int
    scales: int
    tables: int
    table_off: int
    payload: int
    stream_off: int
    escapes: int
    esc_off: int
    tables_cap: int
    payload_cap: int
    escapes_cap: int

    def c(self) -> cg_encoded:
        self._c = cg_encoded(self.anchors, self.scales, self.tables, self.table_off, self.payload, self.stream_off,
                             self.escapes or None, self.esc_off, self.tables_cap, self.payload_cap, self.escapes_cap)
        return self._c


def alloc_encoded(cfg: Config, device="cuda", escapes_cap: Optional[int] = None, pin: bool = False) -> Encoded:
    """Allocate output sections for cg_encode with worst-case capacities
    (escapes default to one per 64 delta values plus 4096; cg_encode flags
    CG_ERR_RANGE if that is not enough)."""
    b = cg_encode_bounds(cfg)
    if escapes_cap is None:
        escapes_cap = min(b["escapes_max_count"], b["escapes_max_count"] // 64 + 4096)
    kw = dict(device=device, pin_memory=pin) if device == "cpu" else dict(device=device)

    def e(n, dt):
        return torch.empty(int(n), dtype=dt, **kw)
    return Encoded(e(b["anchors_bytes"], torch.int8), e(b["scales_bytes"] // 4, torch.float32),
                   e(max(b["tables_max_bytes"], 1), torch.uint8), e(b["n_tables"] + 1, torch.int32),
                   e(max(b["payload_max_bytes"], 16), torch.uint8), e(b["n_streams"] + 1, torch.int64),
                   e(max(escapes_cap, 1), torch.int32), e(b["n_streams"] + 1, torch.int32))


def cache_source(kv: torch.Tensor):
    """(status, CUDA memory type, address the encoder's kernels read) for a
    cache tensor: device memory, or pinned host memory read over the host link."""
    mt, view = ct.c_int(0), ct.c_void_p(None)
    code = lib().cg_cache_source(kv.data_ptr(), ct.byref(mt), ct.byref(view))
    return code, mt.value, view.value


def cg_encode(cfg: Config, kv: torch.Tensor, ws: torch.Tensor, out: Encoded, sizes_host: ct.Structure,
              status: torch.Tensor, stream=None) -> None:
    """Enqueue cg_encode.  kv: fp16 [L][2][T][C] on the device, or in pinned
    host memory (the kernels then read it over the host link); ws: device uint8
    workspace; sizes_host: a cg_sizes in (ideally pinned) host memory;
    status: device int32[1] cleared by the caller."""
    assert (kv.is_cuda or kv.is_pinned()) and kv.dtype == torch.float16 and kv.is_contiguous()
    assert tuple(kv.shape) == (cfg.L, 2, cfg.T, cfg.C)
    code = lib().cg_encode(ct.byref(cfg.c()), kv.data_ptr(), ws.data_ptr(), ws.numel(), ct.byref(out.c()),
                           ct.byref(sizes_host), status.data_ptr(), _stream_ptr(stream))
    _check(code, "cg_encode")


def cg_decode(cfg: Config, enc: Encoded, kv_out: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    """Enqueue cg_decode of a whole object into kv_out (device fp16 [L][2][T][C])."""
    assert kv_out.is_cuda and kv_out.dtype == torch.float16 and kv_out.is_contiguous()
    assert tuple(kv_out.shape) == (cfg.L, 2, cfg.T, cfg.C)
    code = lib().cg_decode(ct.byref(cfg.c()), ct.byref(enc.c()), kv_out.data_ptr(), status.data_ptr(),
                           _stream_ptr(stream))
    _check(code, "cg_decode")


def cg_test_decode_timeout(cfg: Config, enc: Encoded, kv_out: torch.Tensor, status: torch.Tensor,
                           stream=None) -> None:
    """Enqueue the decoder's time-out test kernel (a withheld ring segment and
    short waits: every stream longer than 256 bytes reports CG_ERR_TIMEOUT)."""
    assert kv_out.is_cuda and kv_out.dtype == torch.float16 and kv_out.is_contiguous()
    assert tuple(kv_out.shape) == (cfg.L, 2, cfg.T, cfg.C)
    code = lib().cg_test_decode_timeout(ct.byref(cfg.c()), ct.byref(enc.c()), kv_out.data_ptr(), status.data_ptr(),
                                        _stream_ptr(stream))
    _check(code, "cg_test_decode_timeout")


def cg_decode_paged(cfg: Config, enc, pool: torch.Tensor, block_table: torch.Tensor, block_tokens: int,
                    layer_stride: int, kv_stride: int, block_stride: int, token_stride: int,
                    status: torch.Tensor, stream=None, n_pool_blocks: Optional[int] = None) -> None:
    """Enqueue a decode whose token rows go to the blocks of a paged pool
    (fp16); block_table is a device int32/uint32 tensor of logical -> physical
    blocks.  Strides are in fp16 elements."""
    assert pool.dtype == torch.float16 and block_table.dtype in (torch.int32, torch.uint32)
    assert block_table.is_contiguous()
    if n_pool_blocks is None:
        n_pool_blocks = (pool.numel() - 1) // max(block_stride, 1) + 1
    d = cg_paged_kv(pool.data_ptr(), block_table.data_ptr(), block_table.numel(), n_pool_blocks, block_tokens,
                    layer_stride, kv_stride, block_stride, token_stride)
    code = lib().cg_decode_paged(ct.byref(cfg.c()), ct.byref(enc.c()), ct.byref(d), status.data_ptr(),
                                 _stream_ptr(stream) if pool.is_cuda else None)
    _check(code, "cg_decode_paged")


@dataclasses.dataclass
class ChunkRef:
    cfg: Config
    enc: Encoded
    chunk: int
    dst: torch.Tensor      # device fp16 [L][2][dst_tokens][C]
    dst_token0: int


def _refs(refs: Sequence[ChunkRef]):
    encs = {}
    arr = (cg_chunk_ref * len(refs))()
    keep = []
    for i, r in enumerate(refs):
        key = id(r.enc)
        if key not in encs:
            encs[key] = r.enc.c()
            keep.append(encs[key])
        keep.append(r.cfg.c())
        arr[i] = cg_chunk_ref(ct.pointer(r.cfg.c()), ct.pointer(encs[key]), r.chunk, r.dst.data_ptr(),
                              r.dst.shape[2], r.dst_token0)
    return arr, keep


def cg_decode_chunks_ws_bytes(refs: Sequence[ChunkRef]) -> int:
    arr, keep = _refs(refs)
    n = ct.c_size_t()
    _check(lib().cg_decode_chunks_ws_bytes(arr, len(refs), ct.byref(n)), "cg_decode_chunks_ws_bytes")
    return int(n.value)


def cg_decode_chunks(refs: Sequence[ChunkRef], ws: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    arr, keep = _refs(refs)
    code = lib().cg_decode_chunks(arr, len(refs), ws.data_ptr(), ws.numel(), status.data_ptr(),
                                  _stream_ptr(stream))
    _check(code, "cg_decode_chunks")


CG_NOALLOC_DESC_BYTES = 4 << 20


def cg_decode_chunks_noalloc(refs: Sequence[ChunkRef], status: torch.Tensor, stream=None) -> None:
    """cg_decode_chunks without a workspace: for callers that may not allocate
    device memory (the descriptors go to a fixed array inside libcg; calls that
    overlap on the GPU race, so keep them on one stream)."""
    arr, keep = _refs(refs)
    code = lib().cg_decode_chunks_noalloc(arr, len(refs), status.data_ptr(), _stream_ptr(stream))
    _check(code, "cg_decode_chunks_noalloc")


def cg_chunk_ranges(cfg: Config, chunk: int, stream_off: np.ndarray, esc_off: np.ndarray) -> dict:
    so = np.ascontiguousarray(stream_off, dtype=np.uint64)
    eo = np.ascontiguousarray(esc_off, dtype=np.uint32)
    r = cg_chunk_range()
    _check(lib().cg_chunk_ranges(ct.byref(cfg.c()), chunk, so.ctypes.data, eo.ctypes.data, ct.byref(r)),
           "cg_chunk_ranges")
    return {n: int(getattr(r, n)) for n, _ in r._fields_}


@dataclasses.dataclass
class LevelPlan:
    levels: np.ndarray   # [n_chunks] chosen level (0 = highest quality)
    arrive_s: np.ndarray  # [n_chunks] last byte received
    done_s: np.ndarray    # [n_chunks] decode finished
    finish_s: float


def cg_plan_levels(bytes_: np.ndarray, decode_s: np.ndarray, bw: np.ndarray, slot_s: float,
                   slo_s: float) -> LevelPlan:
    """Quality level per chunk for a bandwidth trace and a deadline.
    bytes_ / decode_s: [n_chunks][n_levels]; bw: bytes/s per trace slot."""
    b = np.ascontiguousarray(bytes_, dtype=np.uint64)
    d = np.ascontiguousarray(decode_s, dtype=np.float64)
    w = np.ascontiguousarray(bw, dtype=np.float64)
    assert b.ndim == 2 and d.shape == b.shape and w.ndim == 1
    n, q = b.shape
    p = cg_level_plan(n, q, b.ctypes.data, d.ctypes.data, w.ctypes.data, len(w), float(slot_s), float(slo_s))
    lv = np.zeros(n, dtype=np.uint32)
    tm = (cg_chunk_time * max(n, 1))()
    fin = ct.c_double()
    _check(lib().cg_plan_levels(ct.byref(p), lv.ctypes.data, ct.addressof(tm), ct.byref(fin)), "cg_plan_levels")
    return LevelPlan(lv, np.array([t.arrive_s for t in tm[:n]]), np.array([t.done_s for t in tm[:n]]),
                     float(fin.value))


def cg_serialize(cfg: Config, host: Encoded) -> bytes:
    s = host.sizes
    sz = cg_sizes(s["payload_bytes"], s["tables_bytes"], s["n_escapes"], s["total_bytes"])
    n = ct.c_size_t()
    _check(lib().cg_serialize(ct.byref(cfg.c()), None, ct.byref(sz), None, ct.byref(n)), "cg_serialize")
    buf = ct.create_string_buffer(n.value)
    _check(lib().cg_serialize(ct.byref(cfg.c()), ct.byref(host.c()), ct.byref(sz), buf, ct.byref(n)),
           "cg_serialize")
    return buf.raw[: n.value]


def cg_deserialize(buf: bytes) -> Tuple[Config, Encoded]:
    c = cg_config()
    step = (ct.c_float * CG_MAX_LAYERS)()
    sz = cg_sizes()
    _check(lib().cg_deserialize_header(buf, len(buf), ct.byref(c), step, ct.byref(sz)), "cg_deserialize_header")
    cfg = Config(c.L, c.T, c.C, c.group_size, c.chunk_tokens, c.tokens_per_stream,
                 np.array(step[: c.L], dtype=np.float32))
    b = cg_encode_bounds(cfg)
    e = lambda n, dt: torch.empty(int(n), dtype=dt)
    host = Encoded(e(b["anchors_bytes"], torch.int8), e(b["scales_bytes"] // 4, torch.float32),
                   e(sz.tables_bytes, torch.uint8), e(b["n_tables"] + 1, torch.int32),
                   e(sz.payload_bytes, torch.uint8), e(b["n_streams"] + 1, torch.int64),
                   e(sz.n_escapes, torch.int32), e(b["n_streams"] + 1, torch.int32),
                   sizes={"payload_bytes": sz.payload_bytes, "tables_bytes": sz.tables_bytes,
                          "n_escapes": sz.n_escapes, "total_bytes": sz.total_bytes})
    _check(lib().cg_deserialize(buf, len(buf), ct.byref(host.c())), "cg_deserialize")
    return cfg, host


# ---------------------------------------------------------------------------
# Allocation helpers around the calls above (sizing and plumbing only)
# ---------------------------------------------------------------------------

def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def read_status(status: torch.Tensor) -> int:
    return cg_status_from_flags(int(status.item()))


class Encoder:
    """Holds the workspace, output buffers and pinned sizes for one config."""

    def __init__(self, cfg: Config, device="cuda", escapes_cap: Optional[int] = None):
        self.cfg = cfg
        self.bounds = cg_encode_bounds(cfg)
        self.ws = torch.empty(self.bounds["workspace_bytes"], dtype=torch.uint8, device=device)
        self.out = alloc_encoded(cfg, device, escapes_cap)
        self.sizes_buf = torch.zeros(4, dtype=torch.int64, pin_memory=True)
        self.sizes = cg_sizes.from_address(self.sizes_buf.data_ptr())
        self.status = new_status(device)

    def launch(self, kv: torch.Tensor, stream=None) -> None:
        cg_encode(self.cfg, kv, self.ws, self.out, self.sizes, self.status, stream)

    def result(self) -> Encoded:
        """After the stream has completed: the sizes and trimmed sections."""
        self.out.sizes = {"payload_bytes": int(self.sizes.payload_bytes), "tables_bytes": int(self.sizes.tables_bytes),
                          "n_escapes": int(self.sizes.n_escapes), "total_bytes": int(self.sizes.total_bytes)}
        return self.out.trimmed()


def _cuda_device_of(kv: torch.Tensor) -> torch.device:
    """The device that encodes kv: its own, or the current one for pinned host memory."""
    return kv.device if kv.is_cuda else torch.device("cuda", torch.cuda.current_device())


def encode(cfg: Config, kv: torch.Tensor, stream=None) -> Encoded:
    """Encode a cache (device or pinned host memory) and wait for it; raises
    on any device status."""
    dev = _cuda_device_of(kv)
    enc = Encoder(cfg, dev)
    enc.launch(kv, stream)
    torch.cuda.synchronize(dev)
    st = read_status(enc.status)
    if st == CG_ERR_RANGE and enc.sizes.n_escapes > enc.out.escapes.numel():
        enc = Encoder(cfg, dev, escapes_cap=int(enc.sizes.n_escapes))
        enc.launch(kv, stream)
        torch.cuda.synchronize(dev)
        st = read_status(enc.status)
    _check(st, "cg_encode (device)")
    return enc.result()


def cg_encode_levels_ws_bytes(cfg: Config, n_levels: int) -> int:
    n = ct.c_size_t()
    _check(lib().cg_encode_levels_ws_bytes(ct.byref(cfg.c()), n_levels, ct.byref(n)), "cg_encode_levels_ws_bytes")
    return int(n.value)


def encode_levels(cfg: Config, kv: torch.Tensor, mults: Sequence[float], share_anchors: bool = True,
                  stream=None) -> List[Tuple[Config, Encoded]]:
    """Encode a cache (device or pinned host memory) at len(mults) quality levels with one call (one
    statistics pass over the cache); level l uses cfg.step * mults[l].
    Returns (level config, trimmed object) per level; each object equals
    encode() with that level's steps.  With share_anchors the levels' objects
    share one anchors and one scales buffer."""
    dev = _cuda_device_of(kv)
    n = len(mults)
    m32 = np.ascontiguousarray(mults, dtype=np.float32)
    cfgs = [Config(cfg.L, cfg.T, cfg.C, cfg.group_size, cfg.chunk_tokens, cfg.tokens_per_stream,
                   (np.asarray(cfg.step, np.float32) * m).astype(np.float32)) for m in m32]
    ws = torch.empty(cg_encode_levels_ws_bytes(cfg, n), dtype=torch.uint8, device=dev)
    sizes_buf = torch.zeros(4 * n, dtype=torch.int64, pin_memory=True)
    sizes = (cg_sizes * n).from_address(sizes_buf.data_ptr())
    esc_cap = None
    for _ in range(2):
        outs = [alloc_encoded(cfg, dev, esc_cap) for _ in range(n)]
        if share_anchors:
            for o in outs[1:]:
                o.anchors, o.scales = outs[0].anchors, outs[0].scales
        arr = (cg_encoded * n)(*[o.c() for o in outs])
        status = new_status(dev)
        code = lib().cg_encode_levels(ct.byref(cfg.c()), n, m32.ctypes.data, kv.data_ptr(), ws.data_ptr(), ws.numel(),
                                      arr, ct.addressof(sizes), status.data_ptr(), _stream_ptr(stream))
        _check(code, "cg_encode_levels")
        torch.cuda.synchronize(dev)
        st = read_status(status)
        need = max(int(sz.n_escapes) for sz in sizes)
        if st == CG_ERR_RANGE and need > outs[0].escapes.numel():
            esc_cap = need
            continue
        _check(st, "cg_encode_levels (device)")
        break
    res = []
    for c, o, sz in zip(cfgs, outs, sizes):
        o.sizes = {"payload_bytes": int(sz.payload_bytes), "tables_bytes": int(sz.tables_bytes),
                   "n_escapes": int(sz.n_escapes), "total_bytes": int(sz.total_bytes)}
        res.append((c, o.trimmed()))
    return res


class LevelEncoder:
    """Holds the workspace, per-level outputs and pinned sizes of
    cg_encode_levels for one config and set of step multipliers, so that the
    call can be launched repeatedly without allocating (the levels share one
    anchors and one scales buffer)."""

    def __init__(self, cfg: Config, mults: Sequence[float], device="cuda", escapes_cap: Optional[int] = None):
        self.cfg = cfg
        self.n = len(mults)
        self.mults = np.ascontiguousarray(mults, dtype=np.float32)
        self.cfgs = [Config(cfg.L, cfg.T, cfg.C, cfg.group_size, cfg.chunk_tokens, cfg.tokens_per_stream,
                            (np.asarray(cfg.step, np.float32) * m).astype(np.float32)) for m in self.mults]
        self.ws = torch.empty(cg_encode_levels_ws_bytes(cfg, self.n), dtype=torch.uint8, device=device)
        self.outs = [alloc_encoded(cfg, device, escapes_cap) for _ in range(self.n)]
        for o in self.outs[1:]:
            o.anchors, o.scales = self.outs[0].anchors, self.outs[0].scales
        self.arr = (cg_encoded * self.n)(*[o.c() for o in self.outs])
        self.sizes_buf = torch.zeros(4 * self.n, dtype=torch.int64, pin_memory=True)
        self.sizes = (cg_sizes * self.n).from_address(self.sizes_buf.data_ptr())
        self.status = new_status(device)

    def launch(self, kv: torch.Tensor, stream=None) -> None:
        code = lib().cg_encode_levels(ct.byref(self.cfg.c()), self.n, self.mults.ctypes.data, kv.data_ptr(),
                                      self.ws.data_ptr(), self.ws.numel(), self.arr, ct.addressof(self.sizes),
                                      self.status.data_ptr(), _stream_ptr(stream))
        _check(code, "cg_encode_levels")

    def results(self) -> List[Tuple[Config, Encoded]]:
        """After the stream has completed: (level config, trimmed object) per level."""
        res = []
        for c, o, sz in zip(self.cfgs, self.outs, self.sizes):
            o.sizes = {"payload_bytes": int(sz.payload_bytes), "tables_bytes": int(sz.tables_bytes),
                       "n_escapes": int(sz.n_escapes), "total_bytes": int(sz.total_bytes)}
            res.append((c, o.trimmed()))
        return res


def ablation(cfg: Config, kv: torch.Tensor, stream=None) -> dict:
    """Ideal coded bits of the cache's delta symbols with one table per
    (layer, K/V, channel), per (layer, K/V) or for the whole cache, and of the
    anchors raw or entropy-coded (cg_ablation); adds bits/value per variant."""
    dev = _cuda_device_of(kv)
    n = ct.c_size_t()
    _check(lib().cg_ablation_ws_bytes(ct.byref(cfg.c()), ct.byref(n)), "cg_ablation_ws_bytes")
    ws = torch.empty(n.value, dtype=torch.uint8, device=dev)
    out = torch.zeros(len(ABLATION_FIELDS), dtype=torch.float64, device=dev)
    status = new_status(dev)
    _check(lib().cg_ablation(ct.byref(cfg.c()), kv.data_ptr(), ws.data_ptr(), ws.numel(), out.data_ptr(),
                             status.data_ptr(), _stream_ptr(stream)), "cg_ablation")
    torch.cuda.synchronize(dev)
    _check(read_status(status), "cg_ablation (device)")
    r = dict(zip(ABLATION_FIELDS, out.cpu().tolist()))
    v, e = r["values"], r["escape_bits"]
    r["bits_per_value"] = {
        "channel_tables": (r["delta_bits_channel"] + e + r["anchor_bits_raw"]) / v,
        "layer_tables": (r["delta_bits_slice"] + e + r["anchor_bits_raw"]) / v,
        "one_table": (r["delta_bits_global"] + e + r["anchor_bits_raw"]) / v,
        "channel_tables_coded_anchors": (r["delta_bits_channel"] + e + r["anchor_bits_channel"]) / v,
    }
    return r


def decode(cfg: Config, enc: Encoded, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode a device object and wait for it; raises on any device status."""
    dev = enc.payload.device
    if out is None:
        out = torch.empty((cfg.L, 2, cfg.T, cfg.C), dtype=torch.float16, device=dev)
    status = new_status(dev)
    cg_decode(cfg, enc, out, status, stream)
    torch.cuda.synchronize(dev)
    _check(read_status(status), "cg_decode (device)")
    return out
