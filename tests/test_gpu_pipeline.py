"""Streamed decode: H2D copies of compressed chunks from pinned host memory
overlapped with cg_decode_chunks on a second stream, checked against the
oracle; a failed transfer is injected on the host (no GPU fault)."""
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


@needs_gpu
def test_streamed_full_width_contexts_match_oracle():
    """Two contexts of the streamed workload at full shape (48 layers x 1024
    channels, its generator and seeds, 1536-token chunks, 512-token streams),
    cut to 1-2 chunks, streamed 4 chunks per stage: bit-exact with the oracle."""
    L, Cc, chunk, tps = synth.STREAM_L, synth.STREAM_C, synth.STREAM_CHUNK, 512
    ctx, expect = [], []
    for j, T in enumerate([2000, 1400]):
        x = synth.stream_context(j, T)
        pc = C.Config(L, T, Cc, 10, chunk, tps, C.layer_steps(L))
        oc = O.Config(L, T, Cc, 10, chunk, tps, O.layer_steps(L))
        enc = C.encode(pc, x.cuda())
        ctx.append(PL.HostObject.from_device(pc, enc))
        oenc = O.encode(oc, x.numpy().view(np.uint16), nthreads=P.nthreads())
        P.assert_same_object(P.gpu_to_np(enc), P.oracle_to_np(oenc), f"context {j}")
        expect.append(O.decode(oc, oenc, nthreads=P.nthreads()))
    outs = [torch.empty((L, 2, h.cfg.T, Cc), dtype=torch.float16, device="cuda") for h in ctx]
    PL.StreamedDecoder(ctx, "cuda", slots=3, chunks_per_stage=4, outputs=outs).run()
    for j, (o, e) in enumerate(zip(outs, expect)):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), e), f"context {j}"
