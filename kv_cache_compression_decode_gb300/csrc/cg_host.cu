// cg_host.cu -- host-only entry points of libcg: status text, chunk ranges
// and the serialized object format.  No CUDA call is made here.
//
// A serialized object is what the CacheGen pages store per context (and per
// quality level) before streaming it ("CacheGen vs 传统量化KV缓存压缩技术深度
// 对比与性能测试", §2.2): header + sections, each section starting on a
// 16-byte boundary so the payload can be used in place.
#include <math.h>
#include <string.h>

#include "cg_internal.cuh"

using namespace cg;

namespace {

constexpr uint32_t kVersion = 1;

struct SectionSizes {
    uint64_t scales, anchors, table_off, tables, stream_off, esc_off, escapes, payload;
};

SectionSizes section_sizes(const Geom &g, const cg_sizes &s) {
    SectionSizes z;
    z.scales = g.n_tables * 4u;
    z.anchors = (uint64_t)g.n_slices * g.A * g.C;
    z.table_off = (g.n_tables + 1u) * 4u;
    z.tables = s.tables_bytes;
    z.stream_off = (g.n_streams + 1u) * 8u;
    z.esc_off = (g.n_streams + 1u) * 4u;
    z.escapes = s.n_escapes * 4u;
    z.payload = s.payload_bytes;
    return z;
}

uint64_t header_bytes(uint32_t L) { return round_up(4 + 4 + 6 * 4 + 4ull * L + 4 * 8, 16); }

void put32(uint8_t *&p, uint32_t v) {
    memcpy(p, &v, 4);
    p += 4;
}
void put64(uint8_t *&p, uint64_t v) {
    memcpy(p, &v, 8);
    p += 8;
}
uint32_t get32(const uint8_t *&p) {
    uint32_t v;
    memcpy(&v, p, 4);
    p += 4;
    return v;
}
uint64_t get64(const uint8_t *&p) {
    uint64_t v;
    memcpy(&v, p, 8);
    p += 8;
    return v;
}

}  // namespace

extern "C" const char *cg_status_string(cg_status s) {
    switch (s) {
        case CG_OK: return "ok";
        case CG_ERR_INVALID_ARG: return "invalid argument";
        case CG_ERR_NONFINITE: return "input holds NaN or Inf";
        case CG_ERR_RANGE: return "buffer too small or size out of range";
        case CG_ERR_CORRUPT: return "encoded object is corrupt";
        case CG_ERR_TIMEOUT: return "bounded device wait timed out";
        case CG_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

extern "C" cg_status cg_status_from_flags(uint32_t flags) {
    for (uint32_t c = 1; c < 16; c++)  // bits 16+ are diagnostics
        if (flags & (1u << c)) return (cg_status)c;
    return CG_OK;
}

extern "C" cg_status cg_chunk_ranges(const cg_config *cfg, uint32_t chunk, const uint64_t *stream_off,
                                     const uint32_t *esc_off, cg_chunk_range *r) {
    Geom g;
    if (!make_geom(cfg, &g) || !r || !stream_off || !esc_off || chunk >= g.n_chunks) return CG_ERR_INVALID_ARG;
    r->stream_begin = g.chunk_stream0(chunk);
    r->stream_end = r->stream_begin + (uint64_t)g.n_slices * g.spc(chunk) * g.NG;
    r->payload_begin = stream_off[r->stream_begin];
    r->payload_end = stream_off[r->stream_end];
    r->escape_begin = esc_off[r->stream_begin];
    r->escape_end = esc_off[r->stream_end];
    r->anchor_begin = g.chunk_anchor_row0(chunk) * g.C;
    r->anchor_end = r->anchor_begin + (uint64_t)g.n_slices * g.apc(chunk) * g.C;
    return CG_OK;
}

extern "C" cg_status cg_serialize(const cg_config *cfg, const cg_encoded *obj, const cg_sizes *sizes, void *buf,
                                  size_t *len) {
    Geom g;
    if (!make_geom(cfg, &g) || !sizes || !len) return CG_ERR_INVALID_ARG;
    const SectionSizes z = section_sizes(g, *sizes);
    const uint64_t parts[8] = {z.scales, z.anchors, z.table_off, z.tables, z.stream_off, z.esc_off, z.escapes, z.payload};
    uint64_t total = header_bytes(g.L);
    for (uint64_t p : parts) total += round_up(p, 16);
    if (!buf) {
        *len = total;
        return CG_OK;
    }
    if (*len < total || !obj) return CG_ERR_RANGE;
    uint8_t *p = static_cast<uint8_t *>(buf);
    memset(p, 0, total);
    memcpy(p, "CGKV", 4);
    p += 4;
    put32(p, kVersion);
    put32(p, cfg->L);
    put32(p, cfg->T);
    put32(p, cfg->C);
    put32(p, cfg->group_size);
    put32(p, cfg->chunk_tokens);
    put32(p, cfg->tokens_per_stream);
    for (uint32_t l = 0; l < cfg->L; l++) {
        memcpy(p, &cfg->step[l], 4);
        p += 4;
    }
    put64(p, sizes->payload_bytes);
    put64(p, sizes->tables_bytes);
    put64(p, sizes->n_escapes);
    put64(p, sizes->total_bytes);
    p = static_cast<uint8_t *>(buf) + header_bytes(g.L);
    const void *src[8] = {obj->scales, obj->anchors, obj->table_off, obj->tables, obj->stream_off, obj->esc_off,
                          obj->escapes, obj->payload};
    for (int i = 0; i < 8; i++) {
        if (parts[i] && !src[i]) return CG_ERR_INVALID_ARG;
        if (parts[i]) memcpy(p, src[i], parts[i]);
        p += round_up(parts[i], 16);
    }
    *len = total;
    return CG_OK;
}

extern "C" cg_status cg_deserialize_header(const void *buf, size_t len, cg_config *cfg, float *step,
                                           cg_sizes *sizes) {
    if (!buf || !cfg || !step || !sizes || len < 32) return CG_ERR_INVALID_ARG;
    const uint8_t *p = static_cast<const uint8_t *>(buf);
    if (memcmp(p, "CGKV", 4) != 0) return CG_ERR_CORRUPT;
    p += 4;
    if (get32(p) != kVersion) return CG_ERR_CORRUPT;
    cfg->L = get32(p);
    cfg->T = get32(p);
    cfg->C = get32(p);
    cfg->group_size = get32(p);
    cfg->chunk_tokens = get32(p);
    cfg->tokens_per_stream = get32(p);
    if (cfg->L == 0 || cfg->L > CG_MAX_LAYERS || len < header_bytes(cfg->L)) return CG_ERR_CORRUPT;
    memcpy(step, p, 4ull * cfg->L);
    p += 4ull * cfg->L;
    cfg->step = step;
    sizes->payload_bytes = get64(p);
    sizes->tables_bytes = get64(p);
    sizes->n_escapes = get64(p);
    sizes->total_bytes = get64(p);
    Geom g;
    if (!make_geom(cfg, &g)) return CG_ERR_CORRUPT;
    size_t need = 0;
    cg_encoded none;
    memset(&none, 0, sizeof(none));
    if (cg_serialize(cfg, &none, sizes, nullptr, &need) != CG_OK || len < need) return CG_ERR_CORRUPT;
    return CG_OK;
}

extern "C" cg_status cg_deserialize(const void *buf, size_t len, const cg_encoded *obj) {
    cg_config cfg;
    static thread_local float step[CG_MAX_LAYERS];
    cg_sizes sizes;
    cg_status st = cg_deserialize_header(buf, len, &cfg, step, &sizes);
    if (st != CG_OK) return st;
    if (!obj) return CG_ERR_INVALID_ARG;
    Geom g;
    if (!make_geom(&cfg, &g)) return CG_ERR_CORRUPT;
    const SectionSizes z = section_sizes(g, sizes);
    if (obj->tables_cap < z.tables || obj->payload_cap < z.payload || obj->escapes_cap < sizes.n_escapes)
        return CG_ERR_RANGE;
    const uint64_t parts[8] = {z.scales, z.anchors, z.table_off, z.tables, z.stream_off, z.esc_off, z.escapes, z.payload};
    void *dst[8] = {obj->scales, obj->anchors, obj->table_off, obj->tables, obj->stream_off, obj->esc_off,
                    obj->escapes, obj->payload};
    const uint8_t *p = static_cast<const uint8_t *>(buf) + header_bytes(cfg.L);
    for (int i = 0; i < 8; i++) {
        if (parts[i] && !dst[i]) return CG_ERR_INVALID_ARG;
        if (parts[i]) memcpy(dst[i], p, parts[i]);
        p += round_up(parts[i], 16);
    }
    return CG_OK;
}

// ---------------------------------------------------------------------------
// Level planner ("CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §2.2).
// ---------------------------------------------------------------------------
namespace {

// End of a transfer of `bytes` that starts at t0 under the piecewise-constant
// trace (slot k covers [k slot_s, (k + 1) slot_s); the last slot holds on).
double transfer_end(const cg_level_plan &p, double t0, double bytes) {
    double t = t0, rem = bytes;
    double kf = floor(t / p.slot_s);
    uint32_t k = kf >= (double)(p.n_slots - 1) ? p.n_slots - 1 : (uint32_t)kf;
    for (; k + 1 < p.n_slots; k++) {
        const double end = (double)(k + 1) * p.slot_s;
        if (end <= t) continue;
        const double cap = (end - t) * p.bw[k];
        if (cap >= rem) return t + rem / p.bw[k];
        rem -= cap;
        t = end;
    }
    return t + rem / p.bw[p.n_slots - 1];
}

// Completion of the context if chunk i takes level q and every later chunk
// the lowest quality, at constant bandwidth b, from link/GPU free times.
double predict_finish(const cg_level_plan &p, uint32_t i, uint32_t q, double t_link, double t_gpu, double b) {
    const uint32_t Q = p.n_levels, low = Q - 1;
    double tl = t_link + (double)p.bytes[(uint64_t)i * Q + q] / b;
    double tg = fmax(tl, t_gpu) + p.decode_s[(uint64_t)i * Q + q];
    for (uint32_t j = i + 1; j < p.n_chunks; j++) {
        tl += (double)p.bytes[(uint64_t)j * Q + low] / b;
        tg = fmax(tl, tg) + p.decode_s[(uint64_t)j * Q + low];
    }
    return tg;
}

bool finite_nonneg(double v) { return isfinite(v) && v >= 0.0; }

}  // namespace

extern "C" cg_status cg_plan_levels(const cg_level_plan *p, uint32_t *level, cg_chunk_time *time, double *finish_s) {
    if (!p || !level || !time || !finish_s || !p->bytes || !p->decode_s || !p->bw) return CG_ERR_INVALID_ARG;
    if (p->n_chunks == 0 || p->n_levels == 0 || p->n_slots == 0) return CG_ERR_INVALID_ARG;
    if (!(isfinite(p->slot_s) && p->slot_s > 0.0) || !finite_nonneg(p->slo_s)) return CG_ERR_INVALID_ARG;
    for (uint32_t k = 0; k < p->n_slots; k++)
        if (!(isfinite(p->bw[k]) && p->bw[k] > 0.0)) return CG_ERR_INVALID_ARG;
    for (uint64_t k = 0; k < (uint64_t)p->n_chunks * p->n_levels; k++)
        if (!finite_nonneg(p->decode_s[k])) return CG_ERR_INVALID_ARG;
    double t_link = 0.0, t_gpu = 0.0, b = p->bw[0];
    for (uint32_t i = 0; i < p->n_chunks; i++) {
        uint32_t q = p->n_levels - 1;
        for (uint32_t c = 0; c + 1 < p->n_levels; c++)
            if (predict_finish(*p, i, c, t_link, t_gpu, b) <= p->slo_s) {
                q = c;
                break;
            }
        const double bytes = (double)p->bytes[(uint64_t)i * p->n_levels + q];
        const double arrive = transfer_end(*p, t_link, bytes);
        if (arrive > t_link) b = bytes / (arrive - t_link);  // throughput seen by this chunk
        t_gpu = fmax(arrive, t_gpu) + p->decode_s[(uint64_t)i * p->n_levels + q];
        t_link = arrive;
        level[i] = q;
        time[i].arrive_s = arrive;
        time[i].done_s = t_gpu;
    }
    *finish_s = t_gpu;
    return CG_OK;
}
