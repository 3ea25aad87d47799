"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: every section of the encoded object byte-equal, the decoded fp16 cache
bit-equal (0 ulp).  Small cases cover several stream tiles, ragged chunks,
spans and groups, and the degenerate cases; the full-size workloads compare
whole layer ranges (the oracle encodes/decodes those layers on its own),
in the same launch configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from kv_cache_compression_decode_gb300 import codec as C
from kv_cache_compression_decode_gb300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu

needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _roundtrip_check(L, T, Cc, G, chunk, tps, x_cpu, mult=1.0, step=None):
    pc, oc = P.configs(L, T, Cc, G, chunk, tps, mult)
    if step is not None:
        pc = C.Config(L, T, Cc, G, chunk or T, tps, np.asarray(step, np.float32))
        oc = O.Config(L, T, Cc, G, chunk or T, tps, np.asarray(step, np.float32))
    x16 = x_cpu.numpy().view(np.uint16)
    oenc = O.encode(oc, x16, nthreads=P.nthreads())
    odec = O.decode(oc, oenc, nthreads=P.nthreads())
    kv = x_cpu.cuda()
    enc = C.encode(pc, kv)
    P.assert_same_object(P.gpu_to_np(enc), P.oracle_to_np(oenc), "encode")
    assert enc.sizes["total_bytes"] == oenc.total_bytes
    dec = C.decode(pc, enc)
    assert np.array_equal(dec.cpu().numpy().view(np.uint16), odec), "decode of GPU object"
    # decode of the oracle's object, uploaded: independent of the GPU encoder
    dec2 = C.decode(pc, P.upload(oenc))
    assert np.array_equal(dec2.cpu().numpy().view(np.uint16), odec), "decode of oracle object"
    return pc, enc, oenc


@needs_gpu
def test_tiny_workload_bit_exact():
    w = synth.TINY
    _roundtrip_check(w.L, w.T, w.C, 10, 0, 1536, w.generate())


SMALL = [
    # L, T, C, G, chunk, tps, seed, rho, outliers
    (2, 300, 64, 10, 128, 64, 1, 0.95, 1),      # ragged chunks and spans
    (3, 1000, 128, 7, 333, 100, 2, 0.9, 2),     # odd group size
    (2, 4100, 64, 10, 0, 1536, 3, 0.95, 1),     # ragged span tail in one chunk
    (1, 1, 32, 10, 1, 1, 4, 0.9, 0),            # one token
    (2, 57, 96, 1, 57, 20, 5, 0.9, 1),          # every token an anchor
    (2, 31, 32, 10, 10, 10, 6, 0.5, 1),         # chunk == group
    (1, 2000, 256, 10, 1536, 1536, 7, 0.95, 2), # full chunk + ragged chunk
    (4, 513, 160, 3, 100, 37, 8, 0.8, 2),
    (2, 900, 64, 23, 300, 250, 9, 0.95, 1),    # groups longer than a ring run
    (1, 700, 32, 15, 700, 700, 10, 0.9, 1),
    (2, 3000, 1024, 10, 1000, 400, 11, 0.9, 2),  # group/row fast path, ragged spans
]


@needs_gpu
@pytest.mark.parametrize("L,T,Cc,G,chunk,tps,seed,rho,nout", SMALL)
def test_small_shapes_bit_exact(L, T, Cc, G, chunk, tps, seed, rho, nout):
    x = synth.ar1_kv(L, T, Cc, rho, nout, seed=seed)
    _roundtrip_check(L, T, Cc, G, chunk, tps, x)


@needs_gpu
def test_escapes_and_extreme_values():
    L, T, Cc = 2, 400, 64
    x = synth.ar1_kv(L, T, Cc, 0.9, 2, seed=11)
    x[0, 0, 5, 3] = 60000.0
    x[0, 0, 6, 3] = -60000.0
    x[1, 1, 7, 40] = 65504.0
    x[1, 1, 8, 41] = -65504.0
    x[0, 1, 100:110, 10] = 0.0
    x[1, 0, :, 63] = 2.0 ** -24  # subnormal constant channel
    _, enc, _ = _roundtrip_check(L, T, Cc, 10, 0, 128, x)
    assert enc.sizes["n_escapes"] > 0
    # small steps force many escapes
    _, enc2, _ = _roundtrip_check(L, T, Cc, 10, 0, 128, synth.ar1_kv(L, T, Cc, 0.9, 2, seed=12),
                                  step=[2.0 ** -9, 0.01])
    assert enc2.sizes["n_escapes"] > 1000


@needs_gpu
def test_equal_spans_escapes_and_unaligned_output():
    """Five spans of equal length (a multiple of the group size) and a short
    one, escapes inside them, and an output that is only 2-byte aligned."""
    L, T, Cc = 2, 530, 96
    x = synth.ar1_kv(L, T, Cc, 0.9, 2, seed=31)
    x[0, 0, 5, 3] = 60000.0
    x[0, 1, 333, 70] = -60000.0
    x[1, 0, 201:204, 17] = 3000.0
    pc, enc, oenc = _roundtrip_check(L, T, Cc, 10, 0, 100, x)  # spans 100 x5 + 30
    assert enc.sizes["n_escapes"] > 0
    _roundtrip_check(L, T, Cc, 10, 0, 100, synth.ar1_kv(L, T, Cc, 0.9, 2, seed=32), step=[2.0 ** -9, 0.01])
    odec = O.decode(P.configs(L, T, Cc, 10, 0, 100)[1], oenc)
    flat = torch.empty(L * 2 * T * Cc + 1, dtype=torch.float16, device="cuda")
    out = flat[1:].view(L, 2, T, Cc)
    assert out.data_ptr() % 4 == 2
    status = C.new_status()
    C.cg_decode(pc, enc, out, status)
    torch.cuda.synchronize()
    assert C.read_status(status) == C.CG_OK
    assert np.array_equal(out.cpu().numpy().view(np.uint16), odec)


@needs_gpu
def test_huge_step_and_constant_cache():
    L, T, Cc = 2, 200, 64
    _roundtrip_check(L, T, Cc, 10, 0, 64, synth.ar1_kv(L, T, Cc, 0.9, 1, seed=13), step=[1e6, 1e6])
    x = torch.full((L, 2, T, Cc), 1.25, dtype=torch.float16)
    _roundtrip_check(L, T, Cc, 10, 0, 64, x)
    _roundtrip_check(L, T, Cc, 10, 0, 64, torch.zeros((L, 2, T, Cc), dtype=torch.float16))


@needs_gpu
def test_mixed_level_chunk_decode_small():
    """Chunks of one cache taken from three encodings (step x1, x2, x4)."""
    L, T, Cc, chunk, tps = 3, 1100, 64, 256, 100
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=21)
    x16 = x.numpy().view(np.uint16)
    n_chunks = (T + chunk - 1) // chunk
    levels = synth.mixed_levels(n_chunks, seed=0)
    objs, odecs = [], []
    for m in synth.LEVEL_MULTIPLIERS:
        pc, oc = P.configs(L, T, Cc, 10, chunk, tps, m)
        oenc = O.encode(oc, x16)
        odecs.append(O.decode(oc, oenc))
        enc = C.encode(pc, x.cuda())
        P.assert_same_object(P.gpu_to_np(enc), P.oracle_to_np(oenc), f"level x{m}")
        objs.append((pc, enc))
    dst = torch.empty((L, 2, T, Cc), dtype=torch.float16, device="cuda")
    refs = [C.ChunkRef(objs[lv][0], objs[lv][1], ch, dst, ch * chunk) for ch, lv in enumerate(levels)]
    ws = torch.empty(C.cg_decode_chunks_ws_bytes(refs), dtype=torch.uint8, device="cuda")
    status = C.new_status()
    C.cg_decode_chunks(refs, ws, status)
    torch.cuda.synchronize()
    assert C.read_status(status) == C.CG_OK
    got = dst.cpu().numpy().view(np.uint16)
    for ch, lv in enumerate(levels):
        sl = slice(ch * chunk, min(T, (ch + 1) * chunk))
        assert np.array_equal(got[:, :, sl], odecs[lv][:, :, sl]), f"chunk {ch} level {lv}"
    # one chunk alone into its own buffer (token offset 0)
    one = torch.empty((L, 2, chunk, Cc), dtype=torch.float16, device="cuda")
    ref = [C.ChunkRef(objs[2][0], objs[2][1], 1, one, 0)]
    ws1 = torch.empty(C.cg_decode_chunks_ws_bytes(ref), dtype=torch.uint8, device="cuda")
    C.cg_decode_chunks(ref, ws1, status)
    torch.cuda.synchronize()
    assert np.array_equal(one.cpu().numpy().view(np.uint16), odecs[2][:, :, chunk:2 * chunk])


@needs_gpu
def test_corruption_is_flagged_not_faulted():
    L, T, Cc = 2, 700, 64
    pc, oc = P.configs(L, T, Cc, 10, 0, 256)
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=31)
    enc = C.encode(pc, x.cuda())
    out = torch.empty((L, 2, T, Cc), dtype=torch.float16, device="cuda")
    cases = []
    e1 = C.Encoded(*[getattr(enc, f).clone() for f in enc.fields()], sizes=enc.sizes)
    e1.payload[200] ^= 0x5A                                   # flipped payload byte
    cases.append(e1)
    e2 = C.Encoded(*[getattr(enc, f).clone() for f in enc.fields()], sizes=enc.sizes)
    e2.stream_off[3] += 16                                    # shifted stream boundary
    cases.append(e2)
    e3 = C.Encoded(*[getattr(enc, f).clone() for f in enc.fields()], sizes=enc.sizes)
    e3.tables[3] ^= 0x01                                      # table no longer sums to 65536
    cases.append(e3)
    e4 = C.Encoded(*[getattr(enc, f).clone() for f in enc.fields()], sizes=enc.sizes)
    e4.payload = e4.payload[: e4.payload.numel() // 2]        # truncated payload section
    cases.append(e4)
    e5 = C.Encoded(*[getattr(enc, f).clone() for f in enc.fields()], sizes=enc.sizes)
    e5.table_off[5] += 1                                      # odd table offset: its 16-bit entries unaligned
    cases.append(e5)
    for i, e in enumerate(cases):
        status = C.new_status()
        C.cg_decode(pc, e, out, status)
        torch.cuda.synchronize()
        assert C.read_status(status) == C.CG_ERR_CORRUPT, f"case {i}"
    # the context is still usable
    assert torch.equal(C.decode(pc, enc), C.decode(pc, enc))


@needs_gpu
def test_encode_reads_pinned_host_cache():
    """A cache in pinned host memory is read by the kernels over the host
    link, and the object is the oracle's.  Pageable host memory is refused on
    the host (INVALID_ARG, nothing enqueued) unless the system maps it."""
    import ctypes as ct
    L, T, Cc = 2, 700, 96
    pc, oc = P.configs(L, T, Cc, 10, 256, 100)
    x = synth.ar1_kv(L, T, Cc, 0.9, 2, seed=51)
    oenc = O.encode(oc, x.numpy().view(np.uint16), nthreads=P.nthreads())
    xp = x.pin_memory()
    code, mem_type, view = C.cache_source(xp)
    assert code == C.CG_OK and mem_type == 1 and view, (code, mem_type, view)
    assert C.cache_source(x.cuda())[:2] == (C.CG_OK, 2)
    enc = C.encode(pc, xp)
    P.assert_same_object(P.gpu_to_np(enc), P.oracle_to_np(oenc), "encode from pinned host memory")
    e2 = C.Encoder(pc, "cuda")
    code = C.lib().cg_encode(ct.byref(pc.c()), x.data_ptr(), e2.ws.data_ptr(), e2.ws.numel(), ct.byref(e2.out.c()),
                             ct.byref(e2.sizes), e2.status.data_ptr(), None)
    if code == C.CG_OK:  # host memory the device reads through the system's page tables
        torch.cuda.synchronize()
        assert C.read_status(e2.status) == C.CG_OK
        P.assert_same_object(P.gpu_to_np(e2.result()), P.oracle_to_np(oenc), "encode from pageable memory")
    else:
        assert code == C.CG_ERR_INVALID_ARG


@needs_gpu
def test_nonfinite_input_and_small_capacity_flagged():
    L, T, Cc = 1, 100, 64
    pc, _ = P.configs(L, T, Cc, 10, 0, 64)
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=41).cuda()
    x[0, 1, 17, 5] = float("nan")
    with pytest.raises(C.CodecError) as e:
        C.encode(pc, x)
    assert e.value.code == C.CG_ERR_NONFINITE
    x[0, 1, 17, 5] = float("inf")
    with pytest.raises(C.CodecError) as e:
        C.encode(pc, x)
    assert e.value.code == C.CG_ERR_NONFINITE
    # escapes capacity too small -> RANGE flagged on the device
    y = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=42)
    y[0, 0, 1:9, :] = 1000.0
    pc2 = C.Config(L, T, Cc, 10, T, 64, np.array([0.5], np.float32))
    encd = C.Encoder(pc2, "cuda", escapes_cap=4)
    encd.launch(y.cuda())
    torch.cuda.synchronize()
    assert C.read_status(encd.status) == C.CG_ERR_RANGE


@needs_gpu
def test_serialized_object_decodes_on_gpu():
    L, T, Cc = 2, 500, 64
    pc, oc = P.configs(L, T, Cc, 10, 200, 100)
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=51)
    enc = C.encode(pc, x.cuda())
    buf = C.cg_serialize(pc, enc.to("cpu"))
    cfg2, host = C.cg_deserialize(buf)
    out = C.decode(cfg2, host.to("cuda"))
    odec = O.decode(oc, O.encode(oc, x.numpy().view(np.uint16)))
    assert np.array_equal(out.cpu().numpy().view(np.uint16), odec)


# --------------------------------------------------------------------------
# full-size workloads, compared on whole layer ranges
# --------------------------------------------------------------------------

def _full_size_check(w: synth.Workload, layer_ranges, mult=1.0):
    pc, _ = P.configs(w.L, w.T, w.C, 10, w.chunk_tokens, w.tokens_per_stream, mult)
    kv = w.generate(device="cuda")
    enc = C.encode(pc, kv)
    dec = C.decode(pc, enc)
    got = P.gpu_to_np(enc)
    geo = P.Geo(w.L, w.T, w.C, 10, w.chunk_tokens, w.tokens_per_stream)
    for l0, l1 in layer_ranges:
        oc = O.Config(l1 - l0, w.T, w.C, 10, w.chunk_tokens or w.T, w.tokens_per_stream,
                      O.layer_steps(w.L, mult=mult)[l0:l1])
        x16 = kv[l0:l1].cpu().numpy().view(np.uint16)
        oenc = O.encode(oc, x16, nthreads=P.nthreads())
        P.assert_same_object(P.cut_layers(got, geo, l0, l1), P.oracle_to_np(oenc), f"{w.name} layers {l0}:{l1}")
        odec = O.decode(oc, oenc, nthreads=P.nthreads())
        assert np.array_equal(dec[l0:l1].cpu().numpy().view(np.uint16), odec), f"{w.name} decode {l0}:{l1}"
    return pc, enc, kv


@needs_gpu
def test_full_size_llama70b_layer_ranges():
    w = synth.LLAMA70B
    _full_size_check(w, [(0, 1), (26, 28), (79, 80)])


@needs_gpu
def test_full_size_llama7b_layer_ranges():
    w = synth.LLAMA7B
    _full_size_check(w, [(0, 1), (15, 16), (31, 32)])


@needs_gpu
def test_full_size_mistral7b_mixed_levels():
    w = synth.MISTRAL7B
    kv = w.generate(device="cuda")
    n_chunks = (w.T + w.chunk_tokens - 1) // w.chunk_tokens
    levels = synth.mixed_levels(n_chunks, seed=0)
    geo = P.Geo(w.L, w.T, w.C, 10, w.chunk_tokens, w.tokens_per_stream)
    objs = []
    for m in synth.LEVEL_MULTIPLIERS:
        pc, _ = P.configs(w.L, w.T, w.C, 10, w.chunk_tokens, w.tokens_per_stream, m)
        enc = C.encode(pc, kv)
        objs.append((pc, enc, P.gpu_to_np(enc)))
    dst = torch.empty_like(kv)
    refs = [C.ChunkRef(objs[lv][0], objs[lv][1], ch, dst, ch * w.chunk_tokens) for ch, lv in enumerate(levels)]
    ws = torch.empty(C.cg_decode_chunks_ws_bytes(refs), dtype=torch.uint8, device="cuda")
    status = C.new_status()
    C.cg_decode_chunks(refs, ws, status)
    torch.cuda.synchronize()
    assert C.read_status(status) == C.CG_OK
    for l0, l1 in [(0, 1), (31, 32)]:
        x16 = kv[l0:l1].cpu().numpy().view(np.uint16)
        for li, m in enumerate(synth.LEVEL_MULTIPLIERS):
            oc = O.Config(l1 - l0, w.T, w.C, 10, w.chunk_tokens, w.tokens_per_stream,
                          O.layer_steps(w.L, mult=m)[l0:l1])
            oenc = O.encode(oc, x16, nthreads=P.nthreads())
            P.assert_same_object(P.cut_layers(objs[li][2], geo, l0, l1), P.oracle_to_np(oenc), f"x{m} {l0}:{l1}")
            odec = O.decode(oc, oenc, nthreads=P.nthreads())
            got = dst[l0:l1].cpu().numpy().view(np.uint16)
            for ch, lv in enumerate(levels):
                if lv != li:
                    continue
                sl = slice(ch * w.chunk_tokens, min(w.T, (ch + 1) * w.chunk_tokens))
                assert np.array_equal(got[:, :, sl], odec[:, :, sl]), f"chunk {ch} x{m} layers {l0}:{l1}"


def _paged(layout, L, npool, bt, Cc):
    """Pool shape and (layer, K/V, block, token) strides of three paged layouts."""
    if layout == "layer_major":  # [L][n_pool][2][bt][C]
        return (L, npool, 2, bt, Cc), dict(layer_stride=npool * 2 * bt * Cc, block_stride=2 * bt * Cc,
                                           kv_stride=bt * Cc, token_stride=Cc)
    if layout == "padded":  # [L][n_pool][2][bt][C + 64]: token rows longer than C
        W = Cc + 64
        return (L, npool, 2, bt, W), dict(layer_stride=npool * 2 * bt * W, block_stride=2 * bt * W,
                                          kv_stride=bt * W, token_stride=W)
    return (npool, L, 2, bt, Cc), dict(layer_stride=2 * bt * Cc, block_stride=L * 2 * bt * Cc,  # [n_pool][L][2][bt][C]
                                       kv_stride=bt * Cc, token_stride=Cc)


@needs_gpu
@pytest.mark.parametrize("layout,bt", [("layer_major", 16), ("block_major", 32), ("layer_major", 1024),
                                       ("padded", 16)])
def test_paged_decode_matches_oracle(layout, bt):
    """Decode straight into a paged block pool through a shuffled block table:
    gathering the blocks back gives the oracle's cache bit for bit, and the
    pool's unused blocks and the rows past the last token stay untouched."""
    L, T, Cc = 3, 1000, 64
    x = synth.ar1_kv(L, T, Cc, 0.9, 2, seed=51)
    x[1, 0, 37, 5] = 30000.0  # an escape
    pc, oc = P.configs(L, T, Cc, 10, 0, 128)
    odec = O.decode(oc, O.encode(oc, x.numpy().view(np.uint16)))
    enc = C.encode(pc, x.cuda())
    nb = (T + bt - 1) // bt
    npool = nb + 5
    perm = np.random.default_rng(bt).permutation(npool)[:nb]
    table = torch.tensor(perm, dtype=torch.int32, device="cuda")
    shape, st = _paged(layout, L, npool, bt, Cc)
    pool = torch.full(shape, -1, dtype=torch.int16, device="cuda")  # 0xFFFF: never a decoded value
    status = C.new_status()
    C.cg_decode_paged(pc, enc, pool.view(torch.float16).view(-1), table, bt, status=status, n_pool_blocks=npool, **st)
    torch.cuda.synchronize()
    assert C.read_status(status) == C.CG_OK
    P16 = pool.cpu().numpy().view(np.uint16)
    blk = (lambda pb: P16[:, pb]) if layout != "block_major" else (lambda pb: P16[pb])
    got = np.concatenate([blk(pb) for pb in perm], axis=2)  # [L][2][nb * bt][row length]
    assert np.array_equal(got[:, :, :T, :Cc], odec)
    assert (got[:, :, T:] == 0xFFFF).all()
    assert (got[..., Cc:] == 0xFFFF).all()  # a padded row's tail
    for pb in sorted(set(range(npool)) - set(perm.tolist())):
        assert (blk(pb) == 0xFFFF).all()


@needs_gpu
def test_paged_decode_block_outside_pool_is_flagged_not_written():
    L, T, Cc, bt = 2, 300, 32, 16
    pc, _ = P.configs(L, T, Cc, 10, 0, 128)
    enc = C.encode(pc, synth.ar1_kv(L, T, Cc, 0.9, 1, seed=52).cuda())
    nb = (T + bt - 1) // bt
    npool = nb
    table = torch.arange(nb, dtype=torch.int32, device="cuda")
    table[7] = npool  # points at the guard block past the pool
    shape, st = _paged("block_major", L, npool + 1, bt, Cc)
    pool = torch.full(shape, -1, dtype=torch.int16, device="cuda")
    status = C.new_status()
    C.cg_decode_paged(pc, enc, pool.view(torch.float16).view(-1), table, bt, status=status, n_pool_blocks=npool, **st)
    torch.cuda.synchronize()
    assert C.read_status(status) == C.CG_ERR_RANGE
    assert (pool[npool].cpu().numpy().view(np.uint16) == 0xFFFF).all()


@needs_gpu
@pytest.mark.parametrize("L,T,Cc,chunk,tps,share", [(3, 1100, 64, 256, 100, True), (3, 1100, 64, 256, 100, False),
                                                    (2, 16384, 1024, 1536, 1536, True)])
def test_multi_level_encode_matches_oracle_per_level(L, T, Cc, chunk, tps, share):
    """One cg_encode_levels call (one statistics pass for the x1/x2/x4 levels)
    gives, level by level, the oracle's object and reconstruction."""
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=61)
    x[0, 1, 50, 7] = 20000.0  # escapes at every level
    x16 = x.numpy().view(np.uint16)
    pc, _ = P.configs(L, T, Cc, 10, chunk, tps)
    res = C.encode_levels(pc, x.cuda(), synth.LEVEL_MULTIPLIERS, share_anchors=share)
    assert len(res) == len(synth.LEVEL_MULTIPLIERS)
    for (lc, enc), m in zip(res, synth.LEVEL_MULTIPLIERS):
        _, oc = P.configs(L, T, Cc, 10, chunk, tps, m)
        assert np.array_equal(lc.step, np.asarray(oc.step, np.float32))
        oenc = O.encode(oc, x16, nthreads=P.nthreads())
        P.assert_same_object(P.gpu_to_np(enc), P.oracle_to_np(oenc), f"level x{m}")
        assert np.array_equal(C.decode(lc, enc).cpu().numpy().view(np.uint16),
                              O.decode(oc, oenc, nthreads=P.nthreads())), f"level x{m}"


@needs_gpu
def test_level_encoder_relaunches_give_the_oracle_objects():
    """codec.LevelEncoder (the benchmark's repeated cg_encode_levels launch
    into preallocated buffers) gives the oracle's object at every level, on
    the first launch and again on a second launch into the same buffers."""
    L, T, Cc, chunk, tps = 2, 900, 64, 300, 100
    x = synth.ar1_kv(L, T, Cc, 0.95, 1, seed=63)
    x[1, 0, 40, 3] = -21000.0  # escapes at every level
    x16 = x.numpy().view(np.uint16)
    pc, _ = P.configs(L, T, Cc, 10, chunk, tps)
    le = C.LevelEncoder(pc, synth.LEVEL_MULTIPLIERS, "cuda")
    xd = x.cuda()
    for launch in range(2):
        le.launch(xd)
        torch.cuda.synchronize()
        assert C.read_status(le.status) == C.CG_OK
        for (lc, enc), m in zip(le.results(), synth.LEVEL_MULTIPLIERS):
            _, oc = P.configs(L, T, Cc, 10, chunk, tps, m)
            assert np.array_equal(lc.step, np.asarray(oc.step, np.float32))
            oenc = O.encode(oc, x16)
            P.assert_same_object(P.gpu_to_np(enc), P.oracle_to_np(oenc), f"launch {launch} level x{m}")


def _bits(counts: np.ndarray) -> float:
    """Sum over rows of sum_s n_s log2(N / n_s), in float64."""
    c = counts.astype(np.float64)
    N = c.sum(axis=-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(c > 0, c * (np.log2(N) - np.log2(np.where(c > 0, c, 1))), 0.0)
    return float(t.sum())


@needs_gpu
@pytest.mark.parametrize("L,T,Cc,chunk", [(3, 700, 96, 256), (2, 4096, 1024, 0)])
def test_grouping_ablation_matches_oracle_counts(L, T, Cc, chunk):
    """cg_ablation's ideal bits equal the entropies of the oracle's own symbol
    and anchor counts under the three groupings."""
    x = synth.ar1_kv(L, T, Cc, 0.9, 2, seed=71)
    x[1, 0, 33, 5] = 25000.0
    pc, oc = P.configs(L, T, Cc, 10, chunk, 128)
    got = C.ablation(pc, x.cuda())
    xn = x.numpy()
    sc = O.anchor_scales(oc, xn)
    anchors, q = O.quantize(oc, xn, sc)
    h = O.histograms(oc, q).astype(np.int64)  # [L*2*C][256]
    ah = np.stack([np.bincount(anchors[l, kv, :, c].astype(np.int64) + 127, minlength=256)
                   for l in range(L) for kv in range(2) for c in range(Cc)])
    want = {
        "values": float(L * 2 * T * Cc),
        "delta_bits_channel": _bits(h),
        "delta_bits_slice": _bits(h.reshape(L * 2, Cc, 256).sum(axis=1)),
        "delta_bits_global": _bits(h.sum(axis=0)),
        "escape_bits": 32.0 * float(h[:, 255].sum()),
        "anchor_bits_raw": 8.0 * anchors.size,
        "anchor_bits_channel": _bits(ah),
    }
    for k, v in want.items():
        assert got[k] == pytest.approx(v, rel=1e-12, abs=1e-6), k
    assert want["escape_bits"] > 0
    b = got["bits_per_value"]
    assert b["channel_tables"] < b["layer_tables"] < b["one_table"]
