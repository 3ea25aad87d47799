"""Benchmark of the KV-cache codec hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over a seeded synthetic
Llama-70B-shaped KV cache (80 layers x {K,V} x 16384 tokens x 8x128 fp16,
5.4 GB): cg_encode (anchor scale/quantize, layer-binned delta quantization,
histograms, 16-bit tables, interleaved range-ANS encode, prefix-sum pack)
then cg_decode of the result.  `value` is fp16 KV GB/s over the whole step;
the decode and encode phases are also reported on their own (CUDA events on
the launching stream).  Inputs (5.4 GB) are larger than L2, so no flush is
needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --workload streamed [--steps K] [--warmup W]

--impl reference times the CPU oracle (the plain C implementation the
parity tests use) on a bounded sample of the same workload.

--workload llama7b runs the same step on the Llama-7B-shaped cache (32
layers x {K,V} x 4096 tokens x 32x128, 2 GiB; 4096 channels per token row).
--workload mistral-mixed encodes the Mistral-7B-shaped cache (32 layers x
{K,V} x 16384 tokens x 8x128, 1536-token chunks) at three quality levels
(step x1, x2, x4) in one cg_encode_levels call, then decodes a seeded
mixed-level chunk sequence in one cg_decode_chunks launch.

--workload streamed measures the streamed batched decode instead: 64
contexts of a Llama-34B-shaped cache (48 layers x {K,V} x 8x128, lengths
uniform in 1.4K-16K tokens, about 112 GB of fp16), each encoded on the GPU
and held compressed in pinned host memory as 1536-token chunks; one step
streams every context through the device (H2D copies of each stage's
chunk ranges on a copy stream, cg_decode_chunks on a compute stream).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "cg_decode / cg_encode GB/s of fp16 KV (1xGB300, % HBM roofline); bits/value"
UNIT = "GB/s"
KERNELS_PER_STEP = 11  # k_stats, 3 x (k_scan_sums + k_scan), k_encode, k_pack, k_sizes, k_decode_all
# end-to-end leg: the cache crosses the host link in this many layer batches
E2E_LAYER_BATCHES = 8
# DRAM bytes (read + write) of one k_decode_all launch on the full Llama-70B
# workload: ncu capture of the first 8 layers (600.4 MB, grows with layers)
# scaled by 80/8.  Must be reset to None whenever k_decode_all changes.
DECODE_TRAFFIC_BYTES = 600.0e6 * 10


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class Clocks:
    """Samples nvidia-smi every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1])]
        mx = [num(r[2]) for r in self.rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in self.rows)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, rank, ws, local
    return None, 0, 1, local


def max_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device):
    if dist is not None:
        dist.barrier(device_ids=[device.index]) if device.type == "cuda" else dist.barrier()


def cpu_baseline(workload, seconds_hint=20.0):
    """The oracle as it stands, on a bounded sample: encode + decode of the
    first layers of the workload, enough (layer, K/V) slices that every host
    core has one (the oracle threads over slices), on all host cores."""
    from oracle import oracle as O
    from kv_cache_compression_decode_gb300 import synth

    cores = os.cpu_count() or 1
    L1 = max(1, min(workload.L, (cores + 1) // 2))
    x = synth.ar1_kv(L1, workload.T, workload.C, workload.rho, workload.n_outlier, workload.seed).numpy()
    oc = O.Config(L1, workload.T, workload.C, 10, workload.chunk, workload.tokens_per_stream,
                  O.layer_steps(workload.L)[:L1])
    x16 = x.view(np.uint16)
    t0 = time.perf_counter()
    reps, t_enc, t_dec = 0, 0.0, 0.0
    while True:
        ta = time.perf_counter()
        enc = O.encode(oc, x16, nthreads=cores)
        tb = time.perf_counter()
        O.decode(oc, enc, nthreads=cores)
        t_enc, t_dec = t_enc + (tb - ta), t_dec + (time.perf_counter() - tb)
        reps += 1
        if time.perf_counter() - t0 > min(seconds_hint, 30.0) or reps >= 5:
            break
    gbs = x16.nbytes / ((t_enc + t_dec) / reps) / 1e9
    # one thread on the first layer (two slices), for the per-core figure
    oc1 = O.Config(1, workload.T, workload.C, 10, workload.chunk, workload.tokens_per_stream,
                   O.layer_steps(workload.L)[:1])
    x1 = np.ascontiguousarray(x16[:1])
    ta = time.perf_counter()
    enc1 = O.encode(oc1, x1, nthreads=1)
    tb = time.perf_counter()
    O.decode(oc1, enc1, nthreads=1)
    tc = time.perf_counter()
    gbs1 = x1.nbytes / (tc - ta) / 1e9
    return {"value": gbs, "unit": UNIT, "cores": min(cores, 2 * L1), "host_cores": cores, "kind": "oracle",
            "encode_value": x16.nbytes / (t_enc / reps) / 1e9, "decode_value": x16.nbytes / (t_dec / reps) / 1e9,
            "single_thread_value": gbs1, "single_thread_encode_value": x1.nbytes / (tb - ta) / 1e9,
            "single_thread_decode_value": x1.nbytes / (tc - tb) / 1e9,
            "sample": f"encode+decode of layers 0..{L1 - 1} ({2 * L1} slices of {workload.T} tokens x "
                      f"{workload.C} channels, {x16.nbytes / 1e6:.0f} MB fp16) of {workload.name}, {reps} reps, "
                      f"one thread per (layer, K/V) slice; single_thread_value: layer 0 on one thread"}


def run_reference(args):
    """--impl reference: the CPU oracle on a bounded sample, same metric."""
    from kv_cache_compression_decode_gb300 import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = synth.LLAMA70B
    base = cpu_baseline(w, seconds_hint=max(5.0, 60.0 / max(1, args.steps + args.warmup)))
    line = {"impl": "reference", "metric": METRIC, "value": base["value"], "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "data": "synthetic",
            "dtype": "f32", "config": {"workload": w.name, "sample": base["sample"]},
            "cpu_baseline": base,
            "e2e": {"value": base["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_streamed(args):
    """--workload streamed: decode pipelined against chunked H2D copies (one
    GPU; under torchrun only rank 0 runs and reports)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from kv_cache_compression_decode_gb300 import codec as C
    from kv_cache_compression_decode_gb300 import pipeline as PL
    from kv_cache_compression_decode_gb300 import synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    lens = synth.stream_context_lengths()
    L, Cc, chunk = synth.STREAM_L, synth.STREAM_C, synth.STREAM_CHUNK
    tps = args.stream_tps
    ctx, comp = [], 0
    for j, T in enumerate(lens):
        x = synth.stream_context(j, T, device=dev)
        cfg = C.Config(L, T, Cc, 10, chunk, tps, C.layer_steps(L))
        enc = C.encode(cfg, x)
        comp += enc.sizes["total_bytes"]
        ctx.append(PL.HostObject.from_device(cfg, enc))
        del x, enc
    torch.cuda.synchronize(dev)
    sd = PL.StreamedDecoder(ctx, dev, slots=args.stream_slots, chunks_per_stage=args.stream_cps)
    for _ in range(max(3, args.warmup)):
        sd.run(timing=False)
    # the pipeline's last context against a direct decode of the same object
    last = ctx[-1]
    direct = C.decode(last.cfg, last.enc.to(dev))
    check = bool(torch.equal(direct, sd.out_view(len(ctx) - 1)))
    del direct
    runs = []
    with Clocks(dev.index) as clk:
        for _ in range(args.steps):
            runs.append(sd.run(timing=True))
    fp16 = runs[0]["fp16_bytes"]
    ms = statistics.median(r["total_ms"] for r in runs)
    pick = lambda k: round(statistics.median(r[k] for r in runs), 4)
    line = {
        "metric": "streamed decode: fp16 KV GB/s with compressed chunks streamed from pinned host memory",
        "value": round(fp16 / (ms * 1e-3) / 1e9, 2), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32+u32", "data": "synthetic",
        "config": {"workload": f"llama34b-48L-8x128-{len(lens)}ctx-streamed", "contexts": len(lens),
                   "tokens": int(sum(lens)), "fp16_bytes": fp16, "compressed_bytes": comp,
                   "bits_per_value": round(8 * comp / (fp16 / 2), 4), "chunk_tokens": chunk,
                   "tokens_per_stream": tps, "chunks_per_stage": args.stream_cps, "slots": args.stream_slots,
                   "step": "every context: H2D of its chunks (copy stream) overlapped with cg_decode_chunks "
                           "(compute stream)"},
        "h2d_gbs": pick("h2d_gbs"), "h2d_bytes_per_step": runs[0]["h2d_bytes"], "h2d_ms": pick("h2d_ms"),
        "decode_ms": pick("decode_ms"), "overlap_efficiency": pick("overlap_efficiency"),
        "decode_gbs_fp16": round(fp16 / (pick("decode_ms") * 1e-3) / 1e9, 2),
        "roofline": {"bound": "hbm", "kernel": "k_decode_jobs (sum of the stages' decode times)",
                     "achieved": round((fp16 + runs[0]["h2d_bytes"]) / (pick("decode_ms") * 1e-3) / 1e9, 1),
                     "peak": peaks()[0], "peak_kind": f"{peaks()[1]} hbm_gbs (burst copy)", "unit": "GB/s",
                     "frac": round((fp16 + runs[0]["h2d_bytes"]) / (pick("decode_ms") * 1e-3) / 1e9 / peaks()[0], 4),
                     "traffic": None, "algorithmic_bytes": fp16 + runs[0]["h2d_bytes"]},
        "last_context_equals_direct_decode": check, "gpu_launches": len(sd.stages) * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if not check:
        raise SystemExit("streamed decode differs from the direct decode")


def run_mixed(args):
    """--workload mistral-mixed: three quality levels encoded in one call,
    then one launch decoding a seeded mixed-level chunk sequence (one GPU;
    under torchrun only rank 0 runs and reports)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from kv_cache_compression_decode_gb300 import codec as C
    from kv_cache_compression_decode_gb300 import synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = synth.MISTRAL7B
    cfg = C.Config(w.L, w.T, w.C, w.group_size, w.chunk, w.tokens_per_stream, C.layer_steps(w.L))
    kv = w.generate(device=dev)
    stream = torch.cuda.current_stream(dev)
    n_chunks = (w.T + w.chunk - 1) // w.chunk
    levels = synth.mixed_levels(n_chunks, seed=0)
    le = C.LevelEncoder(cfg, synth.LEVEL_MULTIPLIERS, dev)
    le.launch(kv, stream)
    torch.cuda.synchronize(dev)
    if C.read_status(le.status) == C.CG_ERR_RANGE:
        le = C.LevelEncoder(cfg, synth.LEVEL_MULTIPLIERS, dev,
                            escapes_cap=max(int(s.n_escapes) for s in le.sizes))
        le.launch(kv, stream)
        torch.cuda.synchronize(dev)
    if C.read_status(le.status) != C.CG_OK:
        raise C.CodecError(C.read_status(le.status), "cg_encode_levels")
    objs = le.results()
    out = torch.empty_like(kv)
    refs = [C.ChunkRef(objs[q][0], objs[q][1], ch, out, ch * w.chunk) for ch, q in enumerate(levels)]
    ws = torch.empty(C.cg_decode_chunks_ws_bytes(refs), dtype=torch.uint8, device=dev)
    dstatus = C.new_status(dev)

    # bytes the decode must read: each chunk's payload, escapes, anchors and
    # stream offsets at its level, plus the tables and scales of every level used
    comp = 0
    for ch, q in enumerate(levels):
        lc, o = objs[q]
        r = C.cg_chunk_ranges(lc, ch, o.stream_off.cpu().numpy().view(np.uint64),
                              o.esc_off.cpu().numpy().view(np.uint32))
        comp += (r["payload_end"] - r["payload_begin"]) + 4 * (r["escape_end"] - r["escape_begin"]) \
            + (r["anchor_end"] - r["anchor_begin"]) + 12 * (r["stream_end"] - r["stream_begin"])
    for q in sorted(set(levels)):
        o = objs[q][1]
        comp += o.tables.numel() + 4 * o.table_off.numel() + 4 * o.scales.numel()
    enc_out = sum(o.sizes["total_bytes"] for _, o in objs)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        le.launch(kv, stream)
        if ev:
            ev[1].record(stream)
        C.cg_decode_chunks(refs, ws, dstatus, stream)
        if ev:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(dev.index) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize(dev)
    st = C.read_status(le.status) or C.read_status(dstatus)
    if st != C.CG_OK:
        raise C.CodecError(st, "timed steps")
    total_ms = t0.elapsed_time(t1) / args.steps
    enc_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    dec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    fp16 = w.fp16_bytes
    peak, peak_kind = peaks()
    dec_ach = (fp16 + comp) / (dec_ms * 1e-3) / 1e9
    enc_ach = (fp16 + enc_out) / (enc_ms * 1e-3) / 1e9
    base = None if args.no_cpu_baseline else cpu_baseline(w)
    line = {
        "metric": METRIC, "value": round(fp16 / (total_ms * 1e-3) / 1e9, 2), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(total_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32+u32", "data": "synthetic",
        "config": {"workload": f"{w.name}-3levels-mixed", "L": w.L, "T": w.T, "C": w.C,
                   "group_size": w.group_size, "chunk_tokens": w.chunk, "tokens_per_stream": w.tokens_per_stream,
                   "level_multipliers": list(synth.LEVEL_MULTIPLIERS), "chunk_levels": levels,
                   "fp16_bytes": fp16, "step": "cg_encode_levels (x1, x2, x4 in one call) + cg_decode_chunks of "
                                               "the mixed-level chunk sequence (one launch)",
                   "l2": f"inputs ({fp16 / 1e9:.1f} GB) larger than L2; no flush"},
        "decode": {"gbs_fp16": round(fp16 / (dec_ms * 1e-3) / 1e9, 2), "ms": round(dec_ms, 4),
                   "hbm_frac": round(dec_ach / peak, 4), "compressed_bytes_read": comp},
        "encode_levels": {"gbs_fp16": round(fp16 / (enc_ms * 1e-3) / 1e9, 2), "ms": round(enc_ms, 4),
                          "hbm_frac": round(enc_ach / peak, 4), "compressed_bytes_written": enc_out},
        "bits_per_value_per_level": [round(8 * o.sizes["total_bytes"] / w.values, 4) for _, o in objs],
        "bits_per_value": round(8 * comp / w.values, 4),
        "roofline": {"bound": "hbm", "kernel": "k_decode_jobs", "achieved": round(dec_ach, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (burst copy)", "unit": "GB/s",
                     "frac": round(dec_ach / peak, 4), "traffic": None, "algorithmic_bytes": fp16 + comp},
        "cpu_baseline": base,
        # one statistics pass, nine kernels per level (3 scans of 2, coder, pack, sizes), one decode
        "gpu_launches": (KERNELS_PER_STEP + 9 * (len(objs) - 1)) * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default="llama70b", choices=["llama70b", "llama7b", "mistral-mixed", "streamed"])
    ap.add_argument("--stream-tps", type=int, default=512, help="streamed: tokens per stream")
    ap.add_argument("--stream-cps", type=int, default=4, help="streamed: chunks per pipeline stage")
    ap.add_argument("--stream-slots", type=int, default=3, help="streamed: staging slots")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: use the first N layers of the workload (not a bench line)")
    ap.add_argument("--cache", default="synthetic", choices=["synthetic", "zeros", "last-layers"],
                    help="profiling only, with --layers: the workload's first layers, an all-zero cache of "
                         "that size, or the workload's last layers")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload == "streamed":
        run_streamed(args)
        return
    if args.workload == "mistral-mixed":
        run_mixed(args)
        return

    from kv_cache_compression_decode_gb300 import codec as C
    from kv_cache_compression_decode_gb300 import synth

    dist, rank, world, local = dist_init()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    base_w = synth.LLAMA70B if args.workload == "llama70b" else synth.LLAMA7B
    w = base_w
    steps = C.layer_steps(base_w.L)
    if args.layers:
        import dataclasses
        where = {"synthetic": "first", "zeros": "zero", "last-layers": "last"}[args.cache]
        w = dataclasses.replace(w, name=f"{w.name}-{where}{args.layers}layers", L=args.layers)
    if args.layers and args.cache == "last-layers":  # the whole cache drawn, its last layers kept
        kv = base_w.generate(device=dev)[base_w.L - w.L:].contiguous()
        steps = steps[base_w.L - w.L:]
    elif args.layers and args.cache == "zeros":
        kv = torch.zeros((w.L, 2, w.T, w.C), dtype=torch.float16, device=dev)
    else:
        kv = w.generate(device=dev)
    cfg = C.Config(w.L, w.T, w.C, w.group_size, w.chunk, w.tokens_per_stream, steps[: w.L])
    torch.cuda.empty_cache()
    enc = C.Encoder(cfg, dev)
    out = torch.empty_like(kv)
    dstatus = C.new_status(dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        enc.launch(kv, stream)
        if ev:
            ev[1].record(stream)
        C.cg_decode(cfg, enc.out, out, dstatus, stream)
        if ev:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    st = C.read_status(enc.status) or C.read_status(dstatus)
    if st != C.CG_OK:
        raise C.CodecError(st, "warm-up step")
    sizes = enc.result().sizes
    comp_bytes = sizes["total_bytes"]

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with Clocks(dev.index) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    total_ms = max_over_ranks(dist, t_start.elapsed_time(t_end), dev)
    enc_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    dec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    st = C.read_status(enc.status) or C.read_status(dstatus)
    if st != C.CG_OK:
        raise C.CodecError(st, "timed steps")

    fp16 = w.fp16_bytes
    ms_per_step = total_ms / args.steps
    value = world * fp16 / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = peaks()
    dec_alg = fp16 + comp_bytes  # compressed in + fp16 out per decode launch
    dec_achieved = dec_alg / (dec_ms * 1e-3) / 1e9
    enc_alg = fp16 + comp_bytes
    enc_achieved = enc_alg / (enc_ms * 1e-3) / 1e9

    # end to end through the C ABI with host buffers: pinned fp16 cache in,
    # encode + decode, the sizes (bits/value) read back, every step.  The
    # cache goes over in layer batches: the H2D copy of batch b + 1 (second
    # stream) runs under the encode + decode of batch b.  Every layer's
    # tables and streams are independent of the others, so a batch's object
    # holds exactly the streams of those layers in the whole-cache object.
    e2e = None
    if not args.no_e2e:
        host_kv = torch.empty(kv.shape, dtype=kv.dtype, pin_memory=True)
        host_kv.copy_(kv)
        nb = E2E_LAYER_BATCHES if w.L % E2E_LAYER_BATCHES == 0 else 1
        lb = w.L // nb
        steps_all = C.layer_steps(base_w.L)[: w.L]
        bcfg = [C.Config(lb, w.T, w.C, w.group_size, w.chunk, w.tokens_per_stream, steps_all[b * lb:(b + 1) * lb])
                for b in range(nb)]
        bencs = [C.Encoder(c, dev) for c in bcfg]
        copy_s = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(nb)]
        consumed = [torch.cuda.Event() for _ in range(nb)]
        for ev in consumed:
            ev.record(stream)

        def e2e_step():
            for b in range(nb):
                sl = slice(b * lb, (b + 1) * lb)
                copy_s.wait_event(consumed[b])  # the last encode of this batch has read kv[sl]
                with torch.cuda.stream(copy_s):
                    kv[sl].copy_(host_kv[sl], non_blocking=True)
                copied[b].record(copy_s)
                stream.wait_event(copied[b])
                bencs[b].launch(kv[sl], stream)
                consumed[b].record(stream)
                C.cg_decode(bcfg[b], bencs[b].out, out[sl], dstatus, stream)  # cg_encode reads its sizes back

        for i in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(dist, dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_s.wait_event(e0)
        n_e2e = max(2, min(args.steps, 5))
        for i in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        for be in bencs:
            st = C.read_status(be.status)
            if st != C.CG_OK:
                raise C.CodecError(st, "end-to-end steps")
        e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev) / n_e2e
        e2e = {"value": world * fp16 / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": fp16,
               "d2h_bytes_per_step": 32 * nb, "ms_per_step": e2e_ms,
               "pipeline": f"{nb} layer batches of {lb}: the H2D copy of a batch from pinned host memory "
                           "(second stream) overlaps the encode + decode of the previous one"}
        del host_kv, bencs

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:  # the oracle baseline belongs to the 1-GPU line
        base = cpu_baseline(w)
    # grouping ablation of the same cache (outside the timed region): ideal
    # bits/value with per-(layer, K/V, channel), per-(layer, K/V) and
    # whole-cache tables, and with entropy-coded anchors
    abl = C.ablation(cfg, kv)["bits_per_value"] if rank == 0 else None

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32+u32", "data": "synthetic",
            "config": {"workload": w.name, "L": w.L, "T": w.T, "C": w.C, "group_size": w.group_size,
                       "tokens_per_stream": w.tokens_per_stream, "steps_per_layer_third": [0.5, 1.0, 1.5],
                       "fp16_bytes": fp16, "step": "cg_encode + cg_decode of the whole cache",
                       "l2": f"inputs ({fp16 / 1e9:.1f} GB) larger than L2; no flush",
                       "parallelism": f"replicas x{world}"},
            "decode": {"gbs_fp16": round(fp16 / (dec_ms * 1e-3) / 1e9, 2), "ms": round(dec_ms, 4),
                       "hbm_frac": round(dec_achieved / peak, 4)},
            "encode": {"gbs_fp16": round(fp16 / (enc_ms * 1e-3) / 1e9, 2), "ms": round(enc_ms, 4),
                       "hbm_frac": round(enc_achieved / peak, 4)},
            "bits_per_value": round(8 * comp_bytes / w.values, 4),
            "payload_bits_per_value": round(8 * sizes["payload_bytes"] / w.values, 4),
            "compressed_bytes": comp_bytes,
            "roofline": {"bound": "hbm", "kernel": "k_decode_all", "achieved": round(dec_achieved, 1),
                         "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs (burst copy)", "unit": "GB/s",
                         "frac": round(dec_achieved / peak, 4),
                         "traffic": (DECODE_TRAFFIC_BYTES if w is synth.LLAMA70B and DECODE_TRAFFIC_BYTES
                                     else None),
                         "traffic_source": "ncu dram__bytes_read+write of an 8-layer launch x 10",
                         "algorithmic_bytes": dec_alg},
            "encode_roofline": {"bound": "hbm", "achieved": round(enc_achieved, 1), "peak": peak, "unit": "GB/s",
                                "frac": round(enc_achieved / peak, 4)},
            "cpu_baseline": base,
            "ablation_ideal_bits_per_value": {k: round(v, 4) for k, v in abl.items()},
            "e2e": e2e,
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
