"""Streamed decode: H2D copies of compressed chunks from pinned host memory
overlapped with cg_decode_chunks on a second stream, checked against the
oracle; a failed transfer is injected on the host (no GPU fault)."""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from kv_cache_compression_decode_gb300 import codec as C
from kv_cache_compression_decode_gb300 import pipeline as PL
from kv_cache_compression_decode_gb300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu
needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _contexts(lens, L=2, Cc=64, chunk=256, tps=256):
    ctx, expect = [], []
    for j, T in enumerate(lens):
        x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=1 + j)
        pc, oc = P.configs(L, T, Cc, 10, chunk, tps)
        enc = C.encode(pc, x.cuda())
        ctx.append(PL.HostObject.from_device(pc, enc))
        oenc = O.encode(oc, x.numpy().view(np.uint16))
        P.assert_same_object(P.gpu_to_np(enc), P.oracle_to_np(oenc), f"context {j}")
        expect.append(O.decode(oc, oenc))
    return ctx, expect


@needs_gpu
@pytest.mark.parametrize("slots,cps", [(2, 1), (3, 2), (1, 3)])
def test_streamed_decode_matches_oracle(slots, cps):
    ctx, expect = _contexts([700, 1500, 333, 256])
    outs = [torch.full((h.cfg.L, 2, h.cfg.T, h.cfg.C), float("nan"), dtype=torch.float16, device="cuda")
            for h in ctx]
    sd = PL.StreamedDecoder(ctx, "cuda", slots=slots, chunks_per_stage=cps, outputs=outs)
    stats = sd.run()
    assert stats["stages"] == len(sd.stages)
    for j, (o, e) in enumerate(zip(outs, expect)):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), e), f"context {j}"
    # the pipeline moved exactly the compressed bytes (plus each context's header)
    comp = sum(h.enc.payload.numel() + 4 * h.enc.escapes.numel() + h.enc.anchors.numel() for h in ctx)
    hdr = sum(sum(getattr(h.enc, f).numel() * getattr(h.enc, f).element_size() for f in sd.hdr_fields)
              for h in ctx)
    assert stats["h2d_bytes"] == comp + hdr


@needs_gpu
def test_streamed_decode_alternating_buffers_last_contexts():
    ctx, expect = _contexts([512, 900, 300])
    sd = PL.StreamedDecoder(ctx, "cuda", slots=2, chunks_per_stage=1)
    sd.run()
    # without per-context outputs the last two contexts are still in their buffers
    for j in (1, 2):
        assert np.array_equal(sd.out_view(j).cpu().numpy().view(np.uint16), expect[j])


@needs_gpu
def test_transfer_failure_is_reported_and_context_survives():
    ctx, expect = _contexts([700, 600])
    calls = {"n": 0}

    def flaky(dst, src):
        calls["n"] += 1
        if calls["n"] == 9:
            raise IOError("injected transfer failure")
        dst.copy_(src, non_blocking=True)

    sd = PL.StreamedDecoder(ctx, "cuda", slots=2, chunks_per_stage=1, copy_fn=flaky)
    with pytest.raises(PL.PipelineError):
        sd.run()
    # the same decoder, with working transfers, still produces the right output
    sd.copy_fn = lambda d, s: d.copy_(s, non_blocking=True)
    outs = [torch.empty((h.cfg.L, 2, h.cfg.T, h.cfg.C), dtype=torch.float16, device="cuda") for h in ctx]
    sd2 = PL.StreamedDecoder(ctx, "cuda", slots=2, chunks_per_stage=1, outputs=outs)
    sd2.run()
    for o, e in zip(outs, expect):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), e)


@needs_gpu
def test_planned_levels_drive_the_stream():
    """cg_plan_levels picks a quality level per chunk for a deadline between
    the all-lowest and the all-highest transfer times; the streamed decode
    then fetches every chunk from, and decodes it with, its level's object."""
    L, Cc, chunk, tps = 2, 64, 128, 128
    objs_all, odecs_all, levels = [], [], []
    for j, T in enumerate([700, 450]):
        x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=40 + j)
        objs, odecs = [], []
        for m in synth.LEVEL_MULTIPLIERS:
            pc, oc = P.configs(L, T, Cc, 10, chunk, tps, m)
            objs.append(PL.HostObject.from_device(pc, C.encode(pc, x.cuda())))
            odecs.append(O.decode(oc, O.encode(oc, x.numpy().view(np.uint16))))
        n = objs[0].n_chunks
        size = lambda h, c: sum((h.ranges[c][k + "_end"] - h.ranges[c][k + "_begin"]) * w
                                for k, w in (("payload", 1), ("anchor", 1), ("escape", 4)))
        nbytes = np.array([[size(h, c) for h in objs] for c in range(n)], dtype=np.uint64)
        dec = np.full(nbytes.shape, 1e-6)
        bw = np.array([1e6])
        hi = C.cg_plan_levels(nbytes, dec, bw, 1.0, 1e9).finish_s
        lo = C.cg_plan_levels(nbytes, dec, bw, 1.0, 0.0).finish_s
        plan = C.cg_plan_levels(nbytes, dec, bw, 1.0, 0.5 * (hi + lo))
        assert plan.finish_s <= 0.5 * (hi + lo)
        assert len(set(plan.levels.tolist())) > 1, plan.levels
        objs_all.append(objs)
        odecs_all.append(odecs)
        levels.append(plan.levels)
    outs = [torch.full((L, 2, h[0].cfg.T, Cc), float("nan"), dtype=torch.float16, device="cuda") for h in objs_all]
    sd = PL.StreamedDecoder(objs_all, "cuda", slots=2, chunks_per_stage=2, outputs=outs, levels=levels)
    sd.run()
    for j, (o, lv) in enumerate(zip(outs, levels)):
        got = o.cpu().numpy().view(np.uint16)
        T = got.shape[2]
        for c, q in enumerate(lv):
            sl = slice(c * chunk, min(T, (c + 1) * chunk))
            assert np.array_equal(got[:, :, sl], odecs_all[j][q][:, :, sl]), f"context {j} chunk {c} level {q}"


def _oracle_layers(x_layers, layers, T):
    """Oracle encode + decode of some layers of a streamed-workload context,
    each layer as a one-layer object with that layer's step."""
    L, Cc, chunk = synth.STREAM_L, synth.STREAM_C, synth.STREAM_CHUNK
    steps = O.layer_steps(L)
    res = []
    for i, l in enumerate(layers):
        oc = O.Config(1, T, Cc, 10, chunk, 512, steps[l:l + 1])
        oenc = O.encode(oc, np.ascontiguousarray(x_layers[i:i + 1]), nthreads=2)
        res.append((P.oracle_to_np(oenc), O.decode(oc, oenc, nthreads=2)))
    return res


@needs_gpu
def test_streamed_workload_matches_oracle():
    """The streamed workload as the benchmark builds it: 64 contexts of a
    Llama-34B-shaped cache (48 layers x 1024 channels) at their drawn lengths
    (1.4K-16K tokens), generated on the device with seeds 1 + j, encoded with
    1536-token chunks and 512-token streams, held in pinned host memory, and
    streamed through StreamedDecoder with the benchmark's settings (4 chunks
    per stage, 3 slots), 8 contexts per run.  The first 8 contexts are
    compared with the oracle in full: every object section byte for byte and
    the streamed output bit for bit.  Every other context is compared on two
    layers (layer 0 and a seeded one): the object's layer cut byte for byte
    with the oracle's one-layer object, and the streamed rows bit for bit
    with the oracle's decode."""
    import concurrent.futures as cf

    L, Cc, chunk, tps = synth.STREAM_L, synth.STREAM_C, synth.STREAM_CHUNK, 512
    lens = synth.stream_context_lengths()
    assert len(lens) == synth.STREAM_CONTEXTS == 64
    pick = synth.seeded_ints(123, 1, L - 1, len(lens))
    workers = max(1, (os.cpu_count() or 1) // 2)
    full = 8
    for b0 in range(0, len(lens), 8):
        ctx, host_x, layers = [], [], []
        for j in range(b0, min(b0 + 8, len(lens))):
            T = lens[j]
            x = synth.stream_context(j, T, device="cuda")
            cfg = C.Config(L, T, Cc, 10, chunk, tps, C.layer_steps(L))
            ctx.append(PL.HostObject.from_device(cfg, C.encode(cfg, x)))
            ls = list(range(L)) if j < full else [0, pick[j]]
            layers.append(ls)
            host_x.append(x.cpu().numpy().view(np.uint16) if j < full else x[ls].cpu().numpy().view(np.uint16))
            del x
        outs = [torch.empty((L, 2, h.cfg.T, Cc), dtype=torch.float16, device="cuda") for h in ctx]
        PL.StreamedDecoder(ctx, "cuda", slots=3, chunks_per_stage=4, outputs=outs).run(timing=False)
        got = [o.cpu().numpy().view(np.uint16) for o in outs]
        del outs
        for i, j in enumerate(range(b0, b0 + len(ctx))):
            h, T = ctx[i], lens[j]
            if j < full:
                oc = O.Config(L, T, Cc, 10, chunk, tps, O.layer_steps(L))
                oenc = O.encode(oc, host_x[i], nthreads=P.nthreads())
                P.assert_same_object(P.gpu_to_np(h.enc), P.oracle_to_np(oenc), f"context {j}")
                assert np.array_equal(got[i], O.decode(oc, oenc, nthreads=P.nthreads())), f"context {j}"
        partial = [(i, j) for i, j in enumerate(range(b0, b0 + len(ctx))) if j >= full]
        with cf.ThreadPoolExecutor(workers) as ex:
            res = list(ex.map(lambda ij: _oracle_layers(host_x[ij[0]], layers[ij[0]], lens[ij[1]]), partial))
        for (i, j), per_layer in zip(partial, res):
            geo = P.Geo(L, lens[j], Cc, 10, chunk, tps)
            obj = P.gpu_to_np(ctx[i].enc)
            for l, (oobj, odec) in zip(layers[i], per_layer):
                P.assert_same_object(P.cut_layers(obj, geo, l, l + 1), oobj, f"context {j} layer {l}")
                assert np.array_equal(got[i][l:l + 1], odec), f"context {j} layer {l}"
        del ctx, host_x, got
