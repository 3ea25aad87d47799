"""cg_decode_chunks_noalloc: the chunked decode for callers that cannot
allocate device memory (a serving engine that owns every device byte, a
plugin that may not call cudaMalloc, or a hot path that must not pay for an
allocation).  It takes no workspace; its job descriptors live in a fixed
array inside libcg.

This file is collected last on purpose, and it also passes when run alone in
a fresh process.  It checks, through the C ABI, that two calls in a row give
exactly the output of cg_decode_chunks (the workspace version) and of the CPU
oracle's decode, and that refs needing more descriptor space than the fixed
array are refused."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from kv_cache_compression_decode_gb300 import codec as C
from kv_cache_compression_decode_gb300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu
needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _levels(L, T, Cc, chunk, tps, seed):
    """Per quality level: (config, GPU object, oracle decode); every GPU object
    is first checked byte for byte against the oracle's."""
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=seed)
    objs = []
    for m in synth.LEVEL_MULTIPLIERS:
        pc, oc = P.configs(L, T, Cc, 10, chunk, tps, m)
        enc = C.encode(pc, x.cuda())
        oenc = O.encode(oc, x.numpy().view(np.uint16))
        P.assert_same_object(P.gpu_to_np(enc), P.oracle_to_np(oenc), f"level x{m}")
        objs.append((pc, enc, O.decode(oc, oenc)))
    return objs


def _with_workspace(refs):
    ws = torch.empty(C.cg_decode_chunks_ws_bytes(refs), dtype=torch.uint8, device="cuda")
    st = C.new_status()
    C.cg_decode_chunks(refs, ws, st)
    torch.cuda.synchronize()
    assert C.read_status(st) == C.CG_OK
    return refs[0].dst.clone()


@needs_gpu
def test_noalloc_matches_workspace_decode_twice_in_a_row():
    L, T, Cc, chunk, tps = 3, 1100, 64, 256, 100
    objs = _levels(L, T, Cc, chunk, tps, seed=71)
    n_chunks = (T + chunk - 1) // chunk
    picks = [synth.mixed_levels(n_chunks, seed=0), synth.mixed_levels(n_chunks, seed=5)]
    stream = torch.cuda.current_stream()
    for call, levels in enumerate(picks):
        ref_dst = torch.full((L, 2, T, Cc), float("nan"), dtype=torch.float16, device="cuda")
        refs = [C.ChunkRef(objs[lv][0], objs[lv][1], ch, ref_dst, ch * chunk) for ch, lv in enumerate(levels)]
        expect = _with_workspace(refs)
        oracle = np.concatenate([objs[lv][2][:, :, ch * chunk:(ch + 1) * chunk] for ch, lv in enumerate(levels)],
                                axis=2)
        out = torch.full((L, 2, T, Cc), float("nan"), dtype=torch.float16, device="cuda")
        refs_na = [C.ChunkRef(r.cfg, r.enc, r.chunk, out, r.dst_token0) for r in refs]
        st = C.new_status()
        C.cg_decode_chunks_noalloc(refs_na, st, stream)
        torch.cuda.synchronize()
        assert C.read_status(st) == C.CG_OK, f"call {call}"
        got = out.cpu().numpy().view(np.uint16)
        assert np.array_equal(got, expect.cpu().numpy().view(np.uint16)), f"call {call}"
        assert np.array_equal(got, oracle), f"call {call} vs the oracle"


@needs_gpu
def test_noalloc_refuses_plans_larger_than_its_array():
    # many distinct objects: every object brings L * 2 * C / 32 jobs
    L, T, Cc = 1, 20, 32 * 256
    refs = []
    dst = torch.empty((L, 2, T, Cc), dtype=torch.float16, device="cuda")
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=3).cuda()
    pc, _ = P.configs(L, T, Cc, 10, 0, 20)
    enc = C.encode(pc, x)
    copies = []
    while sum(1 for _ in copies) * (2 * Cc // 32) * 20 < C.CG_NOALLOC_DESC_BYTES + 4096:
        copies.append(C.Encoded(*[getattr(enc, f).clone() for f in enc.fields()], sizes=enc.sizes))
    refs = [C.ChunkRef(pc, e, 0, dst, 0) for e in copies]
    assert C.cg_decode_chunks_ws_bytes(refs) > C.CG_NOALLOC_DESC_BYTES
    with pytest.raises(C.CodecError) as err:
        C.cg_decode_chunks_noalloc(refs, C.new_status())
    assert err.value.code == C.CG_ERR_RANGE
