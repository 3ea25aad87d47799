"""Decode pipelined against chunked host-to-device copies.

The CacheGen pages have the receiver decode chunks on the GPU while later
chunks are still arriving (gptget.net page, method details: GPU decoding
kept in step with the transfer by pipelining; "CacheGen vs 传统量化KV缓存压缩
技术深度对比与性能测试", §2.2: ~1.5K-token chunks as the streaming unit).
Here the "network" is pinned host memory and the transfer is the GPU's copy
engine:

  copy stream:    wait(slot free) -> H2D of the stage's payload, escape and
                  anchor ranges (each one contiguous range thanks to the
                  chunk-major layout) into staging slot i % N -> record ready_i
  compute stream: wait(ready_i) -> cg_decode_chunks(stage i) -> record free_i

A context's small per-object sections (tables, offsets, scales) go up once,
before its first stage.  All decoding happens in libcg's kernels; this module
only schedules copies and launches.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Sequence

import torch

from . import codec as C


@dataclasses.dataclass
class HostObject:
    """A compressed context held in pinned host memory (the chunk store)."""
    cfg: C.Config
    enc: C.Encoded  # host tensors (pinned), trimmed to the actual sizes
    ranges: List[dict]

    @staticmethod
    def from_device(cfg: C.Config, enc: C.Encoded) -> "HostObject":
        host = C.Encoded(*[torch.empty(getattr(enc, f).shape, dtype=getattr(enc, f).dtype, pin_memory=True)
                           for f in enc.fields()], sizes=enc.sizes)
        for f in enc.fields():
            getattr(host, f).copy_(getattr(enc, f))
        so = host.stream_off.numpy().view("uint64")
        eo = host.esc_off.numpy().view("uint32")
        n_chunks = C.cg_encode_bounds(cfg)["n_chunks"]
        ranges = [C.cg_chunk_ranges(cfg, ch, so, eo) for ch in range(n_chunks)]
        return HostObject(cfg, host, ranges)

    @property
    def n_chunks(self) -> int:
        return len(self.ranges)


class PipelineError(RuntimeError):
    pass


def _span(ranges: Sequence[dict], key: str):
    return ranges[0][key + "_begin"], ranges[-1][key + "_end"]


class StreamedDecoder:
    """Decodes a sequence of compressed contexts, `chunks_per_stage` chunks
    at a time, with H2D copies on one stream and decode on another.

    A context is one HostObject, or -- with `levels` -- one HostObject per
    quality level (the same cache encoded with different steps) together
    with the level of each of its chunks (levels[j][c]), as chosen for
    instance by codec.cg_plan_levels; every chunk is then copied from, and
    decoded with the tables of, its own level."""

    def __init__(self, contexts: Sequence, device="cuda", slots: int = 3, chunks_per_stage: int = 1,
                 copy_fn: Optional[Callable[[torch.Tensor, torch.Tensor], None]] = None,
                 outputs: Optional[Sequence[torch.Tensor]] = None,
                 levels: Optional[Sequence[Sequence[int]]] = None):
        """outputs: optional device fp16 tensor [L][2][T][C] per context;
        without it two buffers alternate between contexts (the decoded
        context is overwritten two contexts later)."""
        if levels is None:
            self.objs = [[h] for h in contexts]
            self.lv = [[0] * h.n_chunks for h in contexts]
        else:
            self.objs = [list(h) for h in contexts]
            self.lv = [list(map(int, l)) for l in levels]
            for j, (os_, lv) in enumerate(zip(self.objs, self.lv)):
                g = [(o.cfg.L, o.cfg.T, o.cfg.C, o.cfg.group_size, o.cfg.chunk_tokens, o.cfg.tokens_per_stream)
                     for o in os_]
                if len(set(g)) != 1 or len(lv) != os_[0].n_chunks or not all(0 <= q < len(os_) for q in lv):
                    raise ValueError(f"context {j}: levels do not match its objects")
        self.ctx = [os_[0] for os_ in self.objs]  # geometry of each context
        self.outputs = list(outputs) if outputs is not None else None
        self.dev = torch.device(device)
        self.N = slots
        self.cps = chunks_per_stage
        self.copy_fn = copy_fn or (lambda dst, src: dst.copy_(src, non_blocking=True))
        # stages: (context index, first chunk, last chunk + 1)
        self.stages = []
        for j, h in enumerate(self.ctx):
            for c0 in range(0, h.n_chunks, self.cps):
                self.stages.append((j, c0, min(c0 + self.cps, h.n_chunks)))
        mx = {"payload": 16, "escape": 1, "anchor": 1}
        for j, c0, c1 in self.stages:
            for k in mx:
                mx[k] = max(mx[k], sum(self._len(j, c, k) for c in range(c0, c1)))
        u8, i32 = torch.uint8, torch.int32
        self.slot_payload = [torch.empty(mx["payload"], dtype=u8, device=self.dev) for _ in range(self.N)]
        self.slot_esc = [torch.empty(mx["escape"], dtype=i32, device=self.dev) for _ in range(self.N)]
        self.slot_anc = [torch.empty(mx["anchor"], dtype=torch.int8, device=self.dev) for _ in range(self.N)]
        # two sets of device headers (one per level) and two output buffers, alternating by context
        hdr_fields = ["scales", "tables", "table_off", "stream_off", "esc_off"]
        self.hdr_fields = hdr_fields
        nlev = max(len(os_) for os_ in self.objs)
        mxh = {f: max(getattr(o.enc, f).numel() for os_ in self.objs for o in os_) for f in hdr_fields}
        dts = {f: getattr(self.ctx[0].enc, f).dtype for f in hdr_fields}
        self.hdr = [[{f: torch.empty(max(mxh[f], 1), dtype=dts[f], device=self.dev) for f in hdr_fields}
                     for _ in range(nlev)] for _ in range(2)]
        mxo = max(h.cfg.L * 2 * h.cfg.T * h.cfg.C for h in self.ctx) if outputs is None else 1
        self.out_buf = [torch.empty(mxo, dtype=torch.float16, device=self.dev) for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(self.dev)
        self.compute_stream = torch.cuda.Stream(self.dev)
        self.status = C.new_status(self.dev)
        # descriptor workspace per slot
        ws = 256
        for j, c0, c1 in self.stages:
            ws = max(ws, C.cg_decode_chunks_ws_bytes(self._refs(j, c0, c1, 0, self._place(j, c0, c1))))
        self.ws = [torch.empty(ws, dtype=torch.uint8, device=self.dev) for _ in range(self.N)]
        self.stats = {}

    def _len(self, j: int, c: int, key: str) -> int:
        r = self.objs[j][self.lv[j][c]].ranges[c]
        return r[key + "_end"] - r[key + "_begin"]

    def _place(self, j: int, c0: int, c1: int):
        """Offsets of each chunk's payload / escape / anchor ranges in a slot.
        Consecutive chunks of one level are one contiguous range (chunk-major
        sections), so they are copied together."""
        place, off = [], {"payload": 0, "escape": 0, "anchor": 0}
        for c in range(c0, c1):
            place.append(dict(off))
            for k in off:
                off[k] += self._len(j, c, k)
        return place

    def out_view(self, j: int) -> torch.Tensor:
        if self.outputs is not None:
            return self.outputs[j]
        cfg = self.ctx[j].cfg
        return self.out_buf[j % 2][: cfg.L * 2 * cfg.T * cfg.C].view(cfg.L, 2, cfg.T, cfg.C)

    def _refs(self, j, c0, c1, slot, place):
        """Chunk refs of a stage.  A run of consecutive chunks at one level
        lies contiguously in the slot and in its object's sections, so the
        run shares one view of the object (and one set of decode blocks)."""
        sp, se, sa = self.slot_payload[slot], self.slot_esc[slot], self.slot_anc[slot]
        dst = self.out_view(j)
        refs = []
        c = c0
        while c < c1:
            q = self.lv[j][c]
            e = c
            while e + 1 < c1 and self.lv[j][e + 1] == q:
                e += 1
            h, hdr, pl = self.objs[j][q], self.hdr[j % 2][q], place[c - c0]
            rb, re_ = h.ranges[c], h.ranges[e]
            raw = C.RawEncoded(anchors=sa.data_ptr() + pl["anchor"] - rb["anchor_begin"],
                               scales=hdr["scales"].data_ptr(), tables=hdr["tables"].data_ptr(),
                               table_off=hdr["table_off"].data_ptr(),
                               payload=sp.data_ptr() + pl["payload"] - rb["payload_begin"],
                               stream_off=hdr["stream_off"].data_ptr(),
                               escapes=se.data_ptr() + 4 * (pl["escape"] - rb["escape_begin"]),
                               esc_off=hdr["esc_off"].data_ptr(), tables_cap=h.enc.tables.numel(),
                               payload_cap=re_["payload_end"], escapes_cap=re_["escape_end"])
            refs += [C.ChunkRef(h.cfg, raw, k, dst, k * h.cfg.chunk_tokens) for k in range(c, e + 1)]
            c = e + 1
        return refs

    def run(self, timing: bool = True) -> dict:
        """Stream every stage through the pipeline; returns timing stats."""
        N = self.N
        ready = [torch.cuda.Event() for _ in self.stages]
        free = [torch.cuda.Event() for _ in self.stages]
        hdr_free = {}
        ev = lambda: torch.cuda.Event(enable_timing=True)
        t0, t1 = ev(), ev()
        copy_ev = [(ev(), ev()) for _ in self.stages] if timing else None
        dec_ev = [(ev(), ev()) for _ in self.stages] if timing else None
        self.status.zero_()
        torch.cuda.synchronize(self.dev)
        t0.record(self.copy_stream)
        self.compute_stream.wait_stream(self.copy_stream)
        h2d_bytes = 0
        error = None
        for i, (j, c0, c1) in enumerate(self.stages):
            slot = i % N
            place = self._place(j, c0, c1)
            try:
                with torch.cuda.stream(self.copy_stream):
                    if i >= N:
                        self.copy_stream.wait_event(free[i - N])
                    if timing:
                        copy_ev[i][0].record(self.copy_stream)
                    if c0 == 0:  # the context's headers (one per level used) into header set j % 2
                        if j >= 2:
                            self.copy_stream.wait_event(hdr_free[j - 2])
                        for q in sorted(set(self.lv[j])):
                            for f in self.hdr_fields:
                                src = getattr(self.objs[j][q].enc, f)
                                if src.numel():
                                    self.copy_fn(self.hdr[j % 2][q][f][: src.numel()], src)
                                    h2d_bytes += src.numel() * src.element_size()
                    # runs of consecutive chunks at one level: one copy per section
                    c = c0
                    while c < c1:
                        q = self.lv[j][c]
                        e = c
                        while e + 1 < c1 and self.lv[j][e + 1] == q:
                            e += 1
                        h = self.objs[j][q]
                        for key, dst, src in (("payload", self.slot_payload[slot], h.enc.payload),
                                              ("escape", self.slot_esc[slot], h.enc.escapes),
                                              ("anchor", self.slot_anc[slot], h.enc.anchors)):
                            b, en = h.ranges[c][key + "_begin"], h.ranges[e][key + "_end"]
                            o = place[c - c0][key]
                            if en > b:
                                self.copy_fn(dst[o: o + en - b], src[b:en])
                                h2d_bytes += (en - b) * src.element_size()
                        c = e + 1
                    if timing:
                        copy_ev[i][1].record(self.copy_stream)
                    ready[i].record(self.copy_stream)
            except Exception as exc:  # a failed transfer: stop issuing, drain what is in flight
                error = exc
                break
            with torch.cuda.stream(self.compute_stream):
                self.compute_stream.wait_event(ready[i])
                if timing:
                    dec_ev[i][0].record(self.compute_stream)
                refs = self._refs(j, c0, c1, slot, place)
                C.cg_decode_chunks(refs, self.ws[slot], self.status, self.compute_stream)
                if timing:
                    dec_ev[i][1].record(self.compute_stream)
                free[i].record(self.compute_stream)
                if c1 == self.ctx[j].n_chunks:
                    hdr_free[j] = torch.cuda.Event()
                    hdr_free[j].record(self.compute_stream)
        self.copy_stream.wait_stream(self.compute_stream)
        t1.record(self.copy_stream)
        torch.cuda.synchronize(self.dev)
        if error is not None:
            raise PipelineError(f"transfer of stage {i} failed: {error}") from error
        st = C.read_status(self.status)
        if st != C.CG_OK:
            raise C.CodecError(st, "streamed decode")
        done = len(self.stages)
        total_ms = t0.elapsed_time(t1)
        fp16 = sum(h.cfg.L * 2 * h.cfg.T * h.cfg.C * 2 for h in self.ctx)
        stats = {"total_ms": total_ms, "stages": done, "h2d_bytes": h2d_bytes, "fp16_bytes": fp16,
                 "fp16_gbs": fp16 / (total_ms * 1e-3) / 1e9}
        if timing:
            t_h2d = sum(a.elapsed_time(b) for a, b in copy_ev[:done])
            t_dec = sum(a.elapsed_time(b) for a, b in dec_ev[:done])
            stats.update({"h2d_ms": t_h2d, "decode_ms": t_dec, "h2d_gbs": h2d_bytes / (t_h2d * 1e-3) / 1e9,
                          "overlap_efficiency": max(t_h2d, t_dec) / total_ms})
        self.stats = stats
        return stats
