// cg_decode.cu -- GPU decoder of the KV-cache codec (sm_103a).
//
// One thread block per (object, layer, K/V, 32-channel group).  Warp 0 turns
// the block's 32 compact frequency tables into shared-memory lookup tables,
// both laid out [entry][lane] so that lane i always hits bank i:
//   tab    [256][32] u32   c_s | (f_s - 1) << 16
//   coarse [256][32] u8    symbol holding slot 256*b (bucket b of the slot)
// Then every warp decodes whole streams (lane = channel): per step the lane
// looks up its symbol (coarse bucket + a forward walk over the few symbols
// that share the bucket), updates its 32-bit range-ANS state, and the warp
// renormalizes with one ballot (lanes take the next words in lane order).
// Dequantization and the anchor add happen in fp32 and the fp16 result is
// stored straight into the [L][2][T][C] layout.  This is the GPU decoder of
// the CacheGen pages (gptget.net page, method details; "CacheGen vs 传统量化
// KV缓存压缩技术深度对比与性能测试", §2.1, parallel CUDA decoding).
//
// Every loop bound comes from the configuration, never from the data, so a
// corrupt object cannot make a kernel spin; integrity failures set
// CG_ERR_CORRUPT in the status word.
#include <cuda_fp16.h>

#include <vector>

#include "cg_internal.cuh"

namespace cg {

struct DecObj {
    Geom g;
    const int8_t *anchors;
    const float *scales;
    const uint8_t *tables;
    const uint32_t *table_off;
    const uint8_t *payload;
    const uint64_t *stream_off;
    const int32_t *escapes;
    const uint32_t *esc_off;
    uint64_t tables_cap, payload_cap, escapes_cap;
    const float *step;  // device, L entries (chunk mode); unused in whole-object mode
};

struct StepTable {
    float v[CG_MAX_LAYERS];
};

// Chunk-mode descriptors (device copies in the workspace).
struct DecJob {
    uint32_t obj, slice, grp, span_begin, span_count;
};
struct SpanRef {
    uint32_t span;  // span index within the object (chunk * spans_full + span in chunk)
    uint32_t ref;   // index into RefDst
};
struct RefDst {
    uint16_t *dst;        // [L][2][dst_tokens][C]
    uint64_t dst_tokens;
    int64_t shift;        // destination token = object token + shift
};

constexpr int kMaxDecWarps = 16;

struct DecSmem {
    uint32_t tab[256 * kLanes];
    uint32_t coarse[64 * kLanes];  // bytes: [(b >> 2)][lane][b & 3]
    uint32_t hi[kLanes];
    float scale[kLanes];
    int bad;
};

__device__ __forceinline__ uint32_t coarse_get(const DecSmem &sm, uint32_t b, uint32_t lane) {
    return reinterpret_cast<const uint8_t *>(sm.coarse)[(((b >> 2) * kLanes + lane) << 2) | (b & 3u)];
}

// Warp 0: build the 32 lookup tables of (slice, grp).
__device__ void build_tables(const DecObj &o, uint32_t slice, uint32_t grp, DecSmem &sm, uint32_t *status) {
    const Geom &g = o.g;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t c = grp * kLanes + lane;
    const uint64_t table = (uint64_t)slice * g.C + c;
    uint8_t *coarse = reinterpret_cast<uint8_t *>(sm.coarse);
    const uint64_t b = o.table_off[table], e = o.table_off[table + 1];
    bool ok = e >= b + 2u && e <= o.tables_cap;
    uint32_t lo = 1, hi = 0;
    if (ok) {
        lo = o.tables[b];
        hi = o.tables[b + 1];
    }
    if (ok && lo <= hi) {
        ok = (e - b) == 2u + 2u * (hi - lo + 1u);
        uint32_t cum = 0, nb = 0;
        for (uint32_t s = lo; ok && s <= hi; s++) {
            const uint64_t at = b + 2u + 2u * (s - lo);
            const uint32_t fm1 = (uint32_t)o.tables[at] | ((uint32_t)o.tables[at + 1] << 8);
            const uint32_t end = cum + fm1 + 1u;
            if (end > kM) {
                ok = false;
                break;
            }
            sm.tab[s * kLanes + lane] = cum | (fm1 << 16);
            for (; nb < 256u && nb * 256u < end; nb++) coarse[(((nb >> 2) * kLanes + lane) << 2) | (nb & 3u)] = (uint8_t)s;
            cum = end;
        }
        ok = ok && cum == kM;
    } else if (ok) {
        // empty table (no delta token in this call): never looked up by a valid stream
        for (uint32_t nb = 0; nb < 256u; nb++) coarse[(((nb >> 2) * kLanes + lane) << 2) | (nb & 3u)] = 0;
        sm.tab[lane] = 0;
        hi = 0;
    }
    if (!ok) {
        hi = 0;
        for (uint32_t nb = 0; nb < 256u; nb++) coarse[(((nb >> 2) * kLanes + lane) << 2) | (nb & 3u)] = 0;
        sm.tab[lane] = 0xFFFF0000u;  // f = 65536 at symbol 0: any slot resolves
    }
    sm.hi[lane] = hi;
    sm.scale[lane] = o.scales[table];
    const bool all_ok = __all_sync(kFull, ok);
    if (lane == 0) {
        sm.bad = !all_ok;
        if (!all_ok) flag(status, CG_ERR_CORRUPT);
    }
}

// Decode stream (slice, grp, span sp) of object o into dst (slice base).
__device__ void decode_span(const DecObj &o, uint32_t slice, uint32_t grp, uint32_t sp, float step,
                            const DecSmem &sm, uint16_t *dst_slice, int64_t shift, uint32_t *status) {
    const Geom &g = o.g;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t c = grp * kLanes + lane;
    const uint32_t lt = lanemask_lt();
    const uint32_t ch = sp / g.spans_full, span = sp - ch * g.spans_full;
    const uint32_t c0 = ch * g.chunk, len = g.chunk_len(ch);
    const uint32_t p0 = span * g.tps, p1 = min(p0 + g.tps, len);
    const uint64_t k = g.stream_index(ch, slice, span, grp);
    const uint64_t sb = o.stream_off[k], se = o.stream_off[k + 1];
    const uint32_t eb = o.esc_off[k], ee = o.esc_off[k + 1];
    const uint32_t nsteps = g.steps_in(p0, p1);
    const uint64_t nw = (se - sb) >> 1;
    bool bad = se < sb || (sb & 15u) || (se & 15u) || se > o.payload_cap || ee < eb || ee > o.escapes_cap ||
               (nsteps == 0 && nw != 0) || (nsteps != 0 && nw < 2u * kLanes);
    if (bad) {
        if (lane == 0) flag(status, CG_ERR_CORRUPT);
        return;
    }
    const uint16_t *w = reinterpret_cast<const uint16_t *>(o.payload + sb);
    const float sa = sm.scale[lane];
    const uint32_t hi = sm.hi[lane];
    uint32_t x = nsteps ? (((uint32_t)w[2 * lane] << 16) | w[2 * lane + 1]) : 0u;
    uint64_t pw = 2u * kLanes;
    uint32_t ep = eb;

    uint32_t gp = p0 % g.G;
    const uint64_t arow0 = g.anchor_index(slice, c0 + p0);  // row of p0's group
    int64_t aidx = (int64_t)arow0 + c - (gp == 0 ? (int64_t)g.C : 0);
    float xa = gp ? __fmul_rn((float)o.anchors[aidx], sa) : 0.f;
    uint16_t *out = dst_slice + ((int64_t)(c0 + p0) + shift) * (int64_t)g.C + c;

    for (uint32_t p = p0; p < p1; p++, out += g.C) {
        if (gp == 0) {
            aidx += g.C;
            xa = __fmul_rn((float)o.anchors[aidx], sa);
            *out = __half_as_ushort(__float2half_rn(xa));
        } else {
            const uint32_t slot = x & 0xFFFFu;
            uint32_t s = coarse_get(sm, slot >> 8, lane);
            uint32_t e = sm.tab[s * kLanes + lane];
            uint32_t r = slot - (e & 0xFFFFu), f = (e >> 16) + 1u;
            while (r >= f && s < hi) {
                s++;
                e = sm.tab[s * kLanes + lane];
                r = slot - (e & 0xFFFFu);
                f = (e >> 16) + 1u;
            }
            x = f * (x >> 16) + r;
            const bool need = x < kStateLow;
            const uint32_t bal = __ballot_sync(kFull, need);
            if (need) {
                const uint64_t idx = pw + __popc(bal & lt);
                x = (x << 16) | (idx < nw ? (uint32_t)w[idx] : 0u);
            }
            pw += __popc(bal);
            int q = (int)s - 127;
            const uint32_t esb = __ballot_sync(kFull, s == kEsc);
            if (esb) {
                if (s == kEsc) {
                    const uint32_t idx = ep + __popc(esb & lt);
                    q = idx < ee ? o.escapes[idx] : 0;
                }
                ep += __popc(esb);
            }
            *out = __half_as_ushort(__float2half_rn(__fadd_rn(xa, __fmul_rn(__int2float_rn(q), step))));
        }
        if (++gp == g.G) gp = 0;
    }
    bool ok = ep == ee;
    if (nsteps) {
        ok = ok && __all_sync(kFull, x == kStateLow) && pw <= nw && nw - pw < 8u;
        bool zero = true;
        for (uint64_t i = pw + lane; i < nw; i += 32) zero = zero && w[i] == 0;
        ok = ok && __all_sync(kFull, zero);
    }
    if (!ok && lane == 0) flag(status, CG_ERR_CORRUPT);
}

__global__ void __launch_bounds__(kMaxDecWarps * 32) k_decode_all(DecObj o, StepTable st, uint16_t *out,
                                                                   uint32_t *status) {
    __shared__ DecSmem sm;
    const uint32_t grp = blockIdx.x, slice = blockIdx.y, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (warp == 0) build_tables(o, slice, grp, sm, status);
    __syncthreads();
    if (sm.bad) return;
    const float step = st.v[slice >> 1];
    uint16_t *dst = out + (uint64_t)slice * o.g.T * o.g.C;
    for (uint64_t sp = warp; sp < o.g.spans_total; sp += nw)
        decode_span(o, slice, grp, (uint32_t)sp, step, sm, dst, 0, status);
}

__global__ void __launch_bounds__(kMaxDecWarps * 32) k_decode_jobs(const DecObj *objs, const DecJob *jobs,
                                                                    const SpanRef *spans, const RefDst *refs,
                                                                    uint32_t *status) {
    __shared__ DecSmem sm;
    const DecJob job = jobs[blockIdx.x];
    const DecObj &o = objs[job.obj];
    const uint32_t warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (warp == 0) build_tables(o, job.slice, job.grp, sm, status);
    __syncthreads();
    if (sm.bad) return;
    const float step = o.step[job.slice >> 1];
    for (uint32_t i = warp; i < job.span_count; i += nw) {
        const SpanRef sr = spans[job.span_begin + i];
        const RefDst rd = refs[sr.ref];
        decode_span(o, job.slice, job.grp, sr.span, step, sm, rd.dst + (uint64_t)job.slice * rd.dst_tokens * o.g.C,
                    rd.shift, status);
    }
}

static bool fill_obj(const cg_config *cfg, const cg_encoded *enc, DecObj *o) {
    if (!make_geom(cfg, &o->g) || !enc) return false;
    if (!enc->anchors || !enc->scales || !enc->tables || !enc->table_off || !enc->stream_off || !enc->esc_off)
        return false;
    if ((!enc->payload && enc->payload_cap) || (!enc->escapes && enc->escapes_cap)) return false;
    if (reinterpret_cast<uintptr_t>(enc->payload) % 16u) return false;
    o->anchors = enc->anchors;
    o->scales = enc->scales;
    o->tables = enc->tables;
    o->table_off = enc->table_off;
    o->payload = enc->payload;
    o->stream_off = enc->stream_off;
    o->escapes = enc->escapes;
    o->esc_off = enc->esc_off;
    o->tables_cap = enc->tables_cap;
    o->payload_cap = enc->payload_cap;
    o->escapes_cap = enc->escapes_cap;
    o->step = nullptr;
    return true;
}

static uint32_t warps_for(uint64_t spans) { return (uint32_t)(spans < (uint64_t)kMaxDecWarps ? spans : kMaxDecWarps); }

// Host-side plan of a chunk batch: descriptors laid out in one buffer.
struct ChunkPlan {
    std::vector<DecObj> objs;
    std::vector<const cg_encoded *> keys;
    std::vector<std::vector<float>> steps;
    std::vector<RefDst> refs;
    std::vector<SpanRef> spans;
    std::vector<DecJob> jobs;
    uint64_t off_objs, off_refs, off_spans, off_jobs, off_steps, bytes;
    uint32_t max_spans;
};

static cg_status plan_chunks(const cg_chunk_ref *refs, uint32_t n, ChunkPlan &P) {
    if (!refs || n == 0) return CG_ERR_INVALID_ARG;
    std::vector<uint32_t> obj_of(n);
    for (uint32_t i = 0; i < n; i++) {
        const cg_chunk_ref &r = refs[i];
        DecObj o;
        if (!fill_obj(r.cfg, r.enc, &o) || !r.dst) return CG_ERR_INVALID_ARG;
        if (r.chunk >= o.g.n_chunks) return CG_ERR_INVALID_ARG;
        if ((uint64_t)r.dst_token0 + o.g.chunk_len(r.chunk) > r.dst_tokens) return CG_ERR_INVALID_ARG;
        uint32_t k = 0;
        while (k < P.keys.size() && P.keys[k] != r.enc) k++;
        if (k == P.keys.size()) {
            P.keys.push_back(r.enc);
            P.objs.push_back(o);
            P.steps.emplace_back(r.cfg->step, r.cfg->step + r.cfg->L);
        } else {
            const Geom &a = P.objs[k].g, &b = o.g;
            if (a.L != b.L || a.T != b.T || a.C != b.C || a.G != b.G || a.chunk != b.chunk || a.tps != b.tps)
                return CG_ERR_INVALID_ARG;
        }
        obj_of[i] = k;
        RefDst d;
        d.dst = r.dst;
        d.dst_tokens = r.dst_tokens;
        d.shift = (int64_t)r.dst_token0 - (int64_t)r.chunk * o.g.chunk;
        P.refs.push_back(d);
    }
    P.max_spans = 1;
    for (uint32_t k = 0; k < P.objs.size(); k++) {
        const Geom &g = P.objs[k].g;
        const uint32_t sb = (uint32_t)P.spans.size();
        for (uint32_t i = 0; i < n; i++) {
            if (obj_of[i] != k) continue;
            const uint32_t ch = refs[i].chunk;
            for (uint32_t s = 0; s < g.spc(ch); s++) P.spans.push_back(SpanRef{ch * g.spans_full + s, i});
        }
        const uint32_t cnt = (uint32_t)P.spans.size() - sb;
        if (cnt > P.max_spans) P.max_spans = cnt;
        for (uint32_t slice = 0; slice < g.n_slices; slice++)
            for (uint32_t grp = 0; grp < g.NG; grp++) P.jobs.push_back(DecJob{k, slice, grp, sb, cnt});
    }
    uint64_t o = 0;
    auto take = [&](uint64_t bytes) {
        uint64_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    P.off_objs = take(P.objs.size() * sizeof(DecObj));
    P.off_refs = take(P.refs.size() * sizeof(RefDst));
    P.off_spans = take(P.spans.size() * sizeof(SpanRef));
    P.off_jobs = take(P.jobs.size() * sizeof(DecJob));
    P.off_steps = o;
    for (auto &s : P.steps) take(s.size() * sizeof(float));
    P.bytes = o;
    return CG_OK;
}

}  // namespace cg

using namespace cg;

extern "C" cg_status cg_decode(const cg_config *cfg, const cg_encoded *enc, uint16_t *kv_out, uint32_t *dev_status,
                               void *stream) {
    DecObj o;
    if (!fill_obj(cfg, enc, &o) || !kv_out) return CG_ERR_INVALID_ARG;
    StepTable st;
    for (uint32_t l = 0; l < o.g.L; l++) st.v[l] = cfg->step[l];
    const dim3 grid(o.g.NG, o.g.n_slices);
    k_decode_all<<<grid, warps_for(o.g.spans_total) * 32, 0, static_cast<cudaStream_t>(stream)>>>(o, st, kv_out,
                                                                                                  dev_status);
    CG_CUDA_TRY(cudaGetLastError());
    return CG_OK;
}

extern "C" cg_status cg_decode_chunks_ws_bytes(const cg_chunk_ref *refs, uint32_t n, size_t *ws_bytes) {
    if (!ws_bytes) return CG_ERR_INVALID_ARG;
    ChunkPlan P;
    cg_status st = plan_chunks(refs, n, P);
    if (st != CG_OK) return st;
    *ws_bytes = P.bytes;
    return CG_OK;
}

extern "C" cg_status cg_decode_chunks(const cg_chunk_ref *refs, uint32_t n, void *ws, size_t ws_bytes,
                                      uint32_t *dev_status, void *stream) {
    ChunkPlan P;
    cg_status st = plan_chunks(refs, n, P);
    if (st != CG_OK) return st;
    if (!ws || reinterpret_cast<uintptr_t>(ws) % 256u) return CG_ERR_INVALID_ARG;
    if (ws_bytes < P.bytes) return CG_ERR_RANGE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    std::vector<uint8_t> host(P.bytes, 0);
    uint64_t so = P.off_steps;
    for (size_t k = 0; k < P.objs.size(); k++) {
        P.objs[k].step = reinterpret_cast<const float *>(w + so);
        memcpy(host.data() + so, P.steps[k].data(), P.steps[k].size() * sizeof(float));
        so = round_up(so + P.steps[k].size() * sizeof(float), 256);
    }
    memcpy(host.data() + P.off_objs, P.objs.data(), P.objs.size() * sizeof(DecObj));
    memcpy(host.data() + P.off_refs, P.refs.data(), P.refs.size() * sizeof(RefDst));
    memcpy(host.data() + P.off_spans, P.spans.data(), P.spans.size() * sizeof(SpanRef));
    memcpy(host.data() + P.off_jobs, P.jobs.data(), P.jobs.size() * sizeof(DecJob));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Pageable source: the copy is staged before cudaMemcpyAsync returns, so
    // `host` may be released when this function returns.
    CG_CUDA_TRY(cudaMemcpyAsync(w, host.data(), P.bytes, cudaMemcpyHostToDevice, s));
    k_decode_jobs<<<(unsigned)P.jobs.size(), warps_for(P.max_spans) * 32, 0, s>>>(
        reinterpret_cast<const DecObj *>(w + P.off_objs), reinterpret_cast<const DecJob *>(w + P.off_jobs),
        reinterpret_cast<const SpanRef *>(w + P.off_spans), reinterpret_cast<const RefDst *>(w + P.off_refs),
        dev_status);
    CG_CUDA_TRY(cudaGetLastError());
    return CG_OK;
}
