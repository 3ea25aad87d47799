/*
 * cgo.c -- plain CPU oracle of the CacheGen KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm load this library.  The product
 * path (the CUDA library and its Python binding) never calls it, and this
 * file shares no code, header, table or constant with the product.
 *
 * What is computed (sources are the five web pages on CacheGen, cited by
 * page title and section):
 *
 *  - Tokens are cut into groups of G (10) tokens; the first token of a group
 *    is the anchor, kept at 8 bits, and every other token of the group is
 *    coded as a delta against that anchor, not against the previous token
 *    ("CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §2.1, stage 1 of
 *    the compression pipeline; "CacheGen: KV Cache Compression and Streaming
 *    for Fast Large Language Model Serving", method details, delta coding).
 *  - Deltas are quantized uniformly with a per-layer step; the pages give
 *    0.5 / 1.0 / 1.5 for shallow / middle / deep layers (same page, §1 and
 *    §2.1 stage 2).  The step array is an input here.
 *  - The quantized symbols are arithmetic-coded with symbol statistics kept
 *    separately per (layer, channel) (same page, §1 "grouped arithmetic
 *    coding"; sciencestack page, TL;DR and Figure 5).
 *  - Long contexts are cut into independently decodable chunks of ~1.5K
 *    tokens (same page, §2.2).
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes of the repository):
 *  R1 anchor: symmetric int8, one fp32 scale per (layer, K/V, channel) over
 *     all anchor rows of the call, s = absmax / 127 (1.0 when absmax is 0),
 *     q_a = clamp(rint(x * (1 / s)), -127, 127); stored raw, not entropy
 *     coded.
 *  R2 deltas are taken against the reconstructed anchor q_a * s (fp32).
 *  R3 q = rint((x - xa) * (1 / step)) in fp32, round half to even, with the
 *     reciprocal 1 / step rounded once per layer (a uniform quantizer
 *     multiplies by the inverse step); symbol q + 127 when |q| <= 127, else
 *     the escape symbol 255 with q sent in an int32 side array.
 *  R4 reconstruction: fp16_rn(xa + float(q) * step); anchors fp16_rn(q_a*s).
 *     Every fp32 operation is separately rounded (no fused multiply-add).
 *  R5 tables: counts per (layer, K/V, channel) over the call, normalized to
 *     a 16-bit total (M = 65536) by the rule in cgo_normalize().
 *  R6 coder: 32-bit-state range ANS, lower bound 2^16, 16-bit words, 32
 *     interleaved lanes (one per channel of a 32-channel group) per stream;
 *     a stream is (layer, K/V, chunk, span of <= tokens_per_stream tokens,
 *     channel group).  Word order is fixed in cgo_rans_encode().
 *  R7 groups restart at every chunk start, so chunks decode alone.
 *
 * Precision: the codec's decisions are made in fp32 on both sides (the
 * kernel's precision), so this file is compiled without fast-math and with
 * -ffp-contract=off.  The fp16 conversions below are written from the IEEE
 * 754 binary16 definition.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
    CGO_OK = 0,
    CGO_ERR_INVALID_ARG = 1,
    CGO_ERR_NONFINITE = 2,
    CGO_ERR_RANGE = 3,
    CGO_ERR_CORRUPT = 4,
    CGO_ERR_NOMEM = 7
};

#define CGO_M 65536u         /* total of a normalized frequency table */
#define CGO_LANES 32u        /* channels per stream */
#define CGO_ESC 255u         /* escape symbol */
#define CGO_STATE0 65536u    /* initial (and final) coder state */

typedef struct {
    uint32_t L, T, C, G, chunk_tokens, tokens_per_stream;
    const float *step; /* L entries */
} cgo_config;

typedef struct {
    int8_t *anchors;      /* [chunk][L][2][anchor rows of the chunk][C] */
    float *scales;        /* [L][2][C] */
    uint8_t *tables;      /* compact tables, see cgo_encode() */
    uint32_t *table_off;  /* [L*2*C + 1] byte offsets into tables */
    uint8_t *payload;     /* stream words */
    uint64_t *stream_off; /* [n_streams + 1] byte offsets into payload */
    int32_t *escapes;     /* escaped q values */
    uint32_t *esc_off;    /* [n_streams + 1] indices into escapes */
    uint64_t tables_cap, payload_cap, escapes_cap; /* capacities (bytes, bytes, count) */
} cgo_encoded;

typedef struct {
    uint64_t payload_bytes, tables_bytes, n_escapes, total_bytes;
} cgo_sizes;

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary32                                            */
/* ------------------------------------------------------------------------ */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

float cgo_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
    if (e == 0) {
        /* zero or subnormal: m * 2^-24, exact in binary32 */
        float v = (float)m * bits_to_f32(0x33800000u); /* 2^-24 */
        return sign ? -v : v;
    }
    if (e == 31) return bits_to_f32(sign | 0x7F800000u | (m << 13));
    return bits_to_f32(sign | ((e - 15u + 127u) << 23) | (m << 13));
}

/* Round to nearest, ties to even. */
uint16_t cgo_f32_to_f16(float f)
{
    uint32_t u = f32_to_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a >= 0x7F800000u) return (uint16_t)(sign | (a > 0x7F800000u ? 0x7E00u : 0x7C00u));
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520 -> inf */
    if (a >= 0x38800000u) {                                   /* >= 2^-14: normal */
        uint32_t h = (((a >> 23) - 127u + 15u) << 10) | ((a & 0x7FFFFFu) >> 13);
        uint32_t rem = a & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h++;
        return (uint16_t)(sign | h);
    }
    /* subnormal half: round |f| * 2^24 to an integer, ties to even */
    uint32_t e = a >> 23;
    if (e == 0) return sign; /* binary32 zero or subnormal: far below 2^-25 */
    uint32_t mant = (a & 0x7FFFFFu) | 0x800000u; /* value = mant * 2^(e-150) */
    uint32_t shift = 126u - e;                   /* |f|*2^24 = mant * 2^(e-126) */
    if (shift >= 32u) return sign;
    uint32_t q = mant >> shift, rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (q & 1u))) q++;
    return (uint16_t)(sign | q);
}

void cgo_f32_to_f16_array(const float *in, uint16_t *out, uint64_t n)
{
    for (uint64_t i = 0; i < n; i++) out[i] = cgo_f32_to_f16(in[i]);
}

void cgo_f16_to_f32_array(const uint16_t *in, float *out, uint64_t n)
{
    for (uint64_t i = 0; i < n; i++) out[i] = cgo_f16_to_f32(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Geometry: chunks, groups, spans, streams                                  */
/* ------------------------------------------------------------------------ */

static uint32_t ceil_div(uint32_t a, uint32_t b) { return (a + b - 1u) / b; }

typedef struct {
    uint32_t n_chunks;
    uint32_t anchors_per_full_chunk;
    uint32_t spans_full;     /* spans in a full chunk */
    uint32_t A;              /* anchor rows in total */
    uint32_t spans_total;    /* spans over all chunks */
    uint32_t NG;             /* channel groups */
    uint32_t n_slices;       /* L * 2 */
    uint64_t n_streams;
    uint64_t n_tables;
} geom;

static int check_config(const cgo_config *cfg)
{
    if (!cfg || !cfg->step) return CGO_ERR_INVALID_ARG;
    if (cfg->L == 0 || cfg->T == 0 || cfg->C == 0 || cfg->C % CGO_LANES) return CGO_ERR_INVALID_ARG;
    if (cfg->G == 0 || cfg->chunk_tokens == 0 || cfg->tokens_per_stream == 0) return CGO_ERR_INVALID_ARG;
    for (uint32_t l = 0; l < cfg->L; l++) {
        float s = cfg->step[l];
        if (!(s > 0x1p-10f) || !isfinite(s)) return CGO_ERR_INVALID_ARG;
    }
    return CGO_OK;
}

static uint32_t chunk_len(const cgo_config *cfg, uint32_t ch)
{
    uint32_t c0 = ch * cfg->chunk_tokens;
    uint32_t rest = cfg->T - c0;
    return rest < cfg->chunk_tokens ? rest : cfg->chunk_tokens;
}

static void make_geom(const cgo_config *cfg, geom *g)
{
    g->n_chunks = ceil_div(cfg->T, cfg->chunk_tokens);
    g->anchors_per_full_chunk = ceil_div(cfg->chunk_tokens, cfg->G);
    g->spans_full = ceil_div(cfg->chunk_tokens, cfg->tokens_per_stream);
    g->n_slices = cfg->L * 2u;
    g->A = 0;
    g->spans_total = 0;
    for (uint32_t ch = 0; ch < g->n_chunks; ch++) {
        uint32_t len = chunk_len(cfg, ch);
        g->A += ceil_div(len, cfg->G);
        g->spans_total += ceil_div(len, cfg->tokens_per_stream);
    }
    g->NG = cfg->C / CGO_LANES;
    g->n_streams = (uint64_t)cfg->L * 2u * g->spans_total * g->NG;
    g->n_tables = (uint64_t)cfg->L * 2u * cfg->C;
}

/* Position of token t inside its chunk, and whether it is an anchor. */
static uint32_t pos_in_chunk(const cgo_config *cfg, uint32_t t) { return t % cfg->chunk_tokens; }
static int is_anchor(const cgo_config *cfg, uint32_t t) { return pos_in_chunk(cfg, t) % cfg->G == 0; }

/* Row, among one slice's anchor rows in token order, of the anchor of token
 * t's group (R7: groups restart at every chunk). */
static uint32_t anchor_row(const cgo_config *cfg, const geom *g, uint32_t t)
{
    uint32_t ch = t / cfg->chunk_tokens;
    return ch * g->anchors_per_full_chunk + pos_in_chunk(cfg, t) / cfg->G;
}

/* The object keeps everything chunk-major so that one chunk is one
 * contiguous range of every per-chunk section.  Anchor plane:
 * [chunk][L*2 slices][anchor rows of the chunk][C]; this is the index of
 * (slice, anchor of token t, channel 0). */
static uint64_t anchor_index(const cgo_config *cfg, const geom *g, uint32_t slice, uint32_t t)
{
    uint32_t ch = t / cfg->chunk_tokens;
    uint32_t apc = ceil_div(chunk_len(cfg, ch), cfg->G);
    uint64_t row = (uint64_t)ch * g->anchors_per_full_chunk * g->n_slices + (uint64_t)slice * apc +
                   pos_in_chunk(cfg, t) / cfg->G;
    return row * cfg->C;
}

/* Streams are ordered (chunk, slice, span in chunk, channel group). */
static uint64_t stream_index(const cgo_config *cfg, const geom *g, uint32_t ch, uint32_t slice, uint32_t span,
                             uint32_t gi)
{
    uint32_t spc = ceil_div(chunk_len(cfg, ch), cfg->tokens_per_stream);
    return (((uint64_t)ch * g->spans_full * g->n_slices + (uint64_t)slice * spc + span) * g->NG) + gi;
}

/* Worst-case sizes: out[0]=A, [1]=spans_total, [2]=n_streams, [3]=n_tables,
 * [4]=tables_max_bytes, [5]=payload_max_bytes, [6]=escapes_max_count. */
int cgo_geometry(const cgo_config *cfg, uint64_t out[7])
{
    int st = check_config(cfg);
    if (st) return st;
    geom g;
    make_geom(cfg, &g);
    out[0] = g.A;
    out[1] = g.spans_total;
    out[2] = g.n_streams;
    out[3] = g.n_tables;
    out[4] = g.n_tables * (2u + 2u * 256u);
    /* every step emits at most one word per lane, plus the 2-word flush per
     * lane, rounded up to 8 words (16 bytes) */
    uint64_t steps_all = 0; /* non-anchor tokens summed over spans */
    for (uint32_t ch = 0; ch < g.n_chunks; ch++) {
        uint32_t len = chunk_len(cfg, ch), c0 = ch * cfg->chunk_tokens;
        for (uint32_t s0 = 0; s0 < len; s0 += cfg->tokens_per_stream) {
            uint32_t s1 = s0 + cfg->tokens_per_stream < len ? s0 + cfg->tokens_per_stream : len;
            uint64_t n = 0;
            for (uint32_t t = s0; t < s1; t++) n += !is_anchor(cfg, c0 + t);
            if (n) steps_all += ((n + 2u) * CGO_LANES + 7u) / 8u * 8u;
        }
    }
    out[5] = steps_all * 2u * cfg->L * 2u * g.NG;
    out[6] = (uint64_t)cfg->L * 2u * ((uint64_t)cfg->T - g.A) * cfg->C;
    return CGO_OK;
}

/* ------------------------------------------------------------------------ */
/* Stage E1: anchor scale per (layer, K/V, channel)  (R1)                    */
/* ------------------------------------------------------------------------ */

/* x: one (layer, K/V) slice [T][C] of fp16 bits.  scales: [C]. */
static int slice_anchor_scales(const cgo_config *cfg, const uint16_t *x, float *scales)
{
    for (uint32_t c = 0; c < cfg->C; c++) {
        float amax = 0.0f;
        for (uint32_t t = 0; t < cfg->T; t++) {
            float v = cgo_f16_to_f32(x[(uint64_t)t * cfg->C + c]);
            if (!isfinite(v)) return CGO_ERR_NONFINITE;
            if (is_anchor(cfg, t) && fabsf(v) > amax) amax = fabsf(v);
        }
        scales[c] = amax > 0.0f ? amax / 127.0f : 1.0f;
    }
    return CGO_OK;
}

/* ------------------------------------------------------------------------ */
/* Stages E2 + E3: anchor quantization, delta quantization  (R1-R3)          */
/* ------------------------------------------------------------------------ */

static int8_t quantize_anchor(float v, float inv_s)
{
    float r = rintf(v * inv_s);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    return (int8_t)r;
}

/* Fills anchors [A][C] and q [T][C] (q at anchor positions is 0). */
static void slice_quantize(const cgo_config *cfg, const geom *g, uint32_t l, const uint16_t *x,
                           const float *scales, int8_t *anchors, int32_t *q)
{
    const float inv_step = 1.0f / cfg->step[l];
    for (uint32_t t = 0; t < cfg->T; t++) {
        uint32_t row = anchor_row(cfg, g, t);
        for (uint32_t c = 0; c < cfg->C; c++) {
            uint64_t i = (uint64_t)t * cfg->C + c;
            float v = cgo_f16_to_f32(x[i]);
            if (is_anchor(cfg, t)) {
                anchors[(uint64_t)row * cfg->C + c] = quantize_anchor(v, 1.0f / scales[c]);
                q[i] = 0;
            } else {
                float xa = (float)anchors[(uint64_t)row * cfg->C + c] * scales[c];
                float d = v - xa;
                q[i] = (int32_t)rintf(d * inv_step);
            }
        }
    }
}

static uint32_t symbol_of(int32_t q) { return (q >= -127 && q <= 127) ? (uint32_t)(q + 127) : CGO_ESC; }

/* ------------------------------------------------------------------------ */
/* Stage E5: normalize counts to a 16-bit frequency table  (R5)              */
/* ------------------------------------------------------------------------ */

/*
 * N = sum n.  Empty table when N == 0 (lo = 1, hi = 0).  Otherwise [lo, hi]
 * is the smallest range holding every symbol seen; each symbol in it gets
 * f = max(1, floor(n * 65536 / N)).  A positive remainder 65536 - sum f goes
 * to the most frequent symbol (smallest symbol on a tie); while the sum is
 * over 65536, the largest f (smallest symbol on a tie) gives back as much as
 * it can while staying >= 1.
 */
int cgo_normalize(const uint32_t n[256], uint32_t f[256], int32_t *lo_out, int32_t *hi_out)
{
    uint64_t N = 0;
    int lo = 256, hi = -1;
    for (int s = 0; s < 256; s++) {
        f[s] = 0;
        N += n[s];
        if (n[s]) {
            if (lo == 256) lo = s;
            hi = s;
        }
    }
    if (N == 0) {
        *lo_out = 1;
        *hi_out = 0;
        return CGO_OK;
    }
    int64_t sum = 0;
    for (int s = lo; s <= hi; s++) {
        uint64_t v = ((uint64_t)n[s] * CGO_M) / N;
        f[s] = v < 1u ? 1u : (uint32_t)v;
        sum += f[s];
    }
    int64_t R = (int64_t)CGO_M - sum;
    if (R > 0) {
        int best = lo;
        for (int s = lo; s <= hi; s++)
            if (n[s] > n[best]) best = s;
        f[best] += (uint32_t)R;
    }
    while (R < 0) {
        int best = lo;
        for (int s = lo; s <= hi; s++)
            if (f[s] > f[best]) best = s;
        int64_t dec = (int64_t)f[best] - 1;
        if (dec > -R) dec = -R;
        if (dec <= 0) return CGO_ERR_CORRUPT; /* cannot happen for W <= 256 */
        f[best] -= (uint32_t)dec;
        R += dec;
    }
    *lo_out = lo;
    *hi_out = hi;
    return CGO_OK;
}

static void cumulative(const uint32_t f[256], uint32_t c[256])
{
    uint32_t acc = 0;
    for (int s = 0; s < 256; s++) {
        c[s] = acc;
        acc += f[s];
    }
}

/* ------------------------------------------------------------------------ */
/* Stage E6 / D2: interleaved rANS  (R6)                                     */
/* ------------------------------------------------------------------------ */

/*
 * Encode one stream of `lanes` interleaved lanes over `steps` steps.
 * sym[j * lanes + i] is lane i's symbol at step j; lane i's table is
 * f[i*256 .. i*256+255].  Every lane starts at state 2^16.  Steps are taken
 * in reverse and, inside a step, lanes from the last to the first.  Before
 * a symbol with frequency f is coded, a state >= f * 2^16 (computed in 64
 * bits) first pushes its low 16 bits and shifts right by 16; then
 * x = floor(x / f) * 2^16 + (x mod f) + c.  At the end every lane, from the
 * last to the first, pushes its low then high half, and the pushed word list
 * is reversed.  A stream with no step holds no word.
 */
int cgo_rans_encode(uint32_t lanes, uint32_t steps, const uint8_t *sym, const uint32_t *f,
                    uint16_t *out, uint64_t cap, uint64_t *nout)
{
    if (lanes == 0 || lanes > CGO_LANES) return CGO_ERR_INVALID_ARG;
    *nout = 0;
    if (steps == 0) return CGO_OK;
    uint32_t cum[CGO_LANES][256];
    for (uint32_t i = 0; i < lanes; i++) cumulative(f + (uint64_t)i * 256u, cum[i]);
    uint32_t x[CGO_LANES];
    for (uint32_t i = 0; i < lanes; i++) x[i] = CGO_STATE0;
    uint64_t n = 0;
    for (uint32_t j = steps; j-- > 0;) {
        for (uint32_t i = lanes; i-- > 0;) {
            uint32_t s = sym[(uint64_t)j * lanes + i];
            uint32_t fs = f[(uint64_t)i * 256u + s], cs = cum[i][s];
            if (fs == 0) return CGO_ERR_INVALID_ARG; /* symbol outside the table */
            if ((uint64_t)x[i] >= ((uint64_t)fs << 16)) {
                if (n >= cap) return CGO_ERR_RANGE;
                out[n++] = (uint16_t)(x[i] & 0xFFFFu);
                x[i] >>= 16;
            }
            x[i] = ((x[i] / fs) << 16) + (x[i] % fs) + cs;
        }
    }
    for (uint32_t i = lanes; i-- > 0;) {
        if (n + 2 > cap) return CGO_ERR_RANGE;
        out[n++] = (uint16_t)(x[i] & 0xFFFFu);
        out[n++] = (uint16_t)(x[i] >> 16);
    }
    for (uint64_t a = 0, b = n - 1; a < b; a++, b--) {
        uint16_t t = out[a];
        out[a] = out[b];
        out[b] = t;
    }
    *nout = n;
    return CGO_OK;
}

/*
 * Decode one stream.  Lane i starts from (w[2i] << 16) | w[2i+1].  At every
 * step each lane finds the unique symbol s in [lo_i, hi_i] with
 * c_s <= (x & 0xFFFF) < c_s + f_s and sets x = f_s * (x >> 16) + slot - c_s;
 * then lanes in order, each whose state fell below 2^16, shift in the next
 * word.  A valid stream ends with every state back at 2^16 and every word
 * consumed (*consumed reports the count).
 */
int cgo_rans_decode(uint32_t lanes, uint32_t steps, const uint16_t *w, uint64_t nw, const uint32_t *f,
                    const int32_t *lo, const int32_t *hi, uint8_t *sym, uint64_t *consumed)
{
    if (lanes == 0 || lanes > CGO_LANES) return CGO_ERR_INVALID_ARG;
    *consumed = 0;
    if (steps == 0) return nw == 0 ? CGO_OK : CGO_ERR_CORRUPT;
    if (nw < 2u * lanes) return CGO_ERR_CORRUPT;
    uint32_t cum[CGO_LANES][256];
    for (uint32_t i = 0; i < lanes; i++) cumulative(f + (uint64_t)i * 256u, cum[i]);
    uint32_t x[CGO_LANES];
    for (uint32_t i = 0; i < lanes; i++) x[i] = ((uint32_t)w[2 * i] << 16) | w[2 * i + 1];
    uint64_t p = 2u * lanes;
    for (uint32_t j = 0; j < steps; j++) {
        for (uint32_t i = 0; i < lanes; i++) {
            const uint32_t *fi = f + (uint64_t)i * 256u;
            uint32_t slot = x[i] & 0xFFFFu;
            int found = -1;
            for (int s = lo[i]; s <= hi[i]; s++) {
                if (fi[s] && cum[i][s] <= slot && slot < cum[i][s] + fi[s]) {
                    found = s;
                    break;
                }
            }
            if (found < 0) return CGO_ERR_CORRUPT;
            x[i] = fi[found] * (x[i] >> 16) + slot - cum[i][found];
            sym[(uint64_t)j * lanes + i] = (uint8_t)found;
        }
        for (uint32_t i = 0; i < lanes; i++) {
            if (x[i] < CGO_STATE0) {
                if (p >= nw) return CGO_ERR_CORRUPT;
                x[i] = (x[i] << 16) | w[p++];
            }
        }
    }
    for (uint32_t i = 0; i < lanes; i++)
        if (x[i] != CGO_STATE0) return CGO_ERR_CORRUPT;
    *consumed = p;
    return CGO_OK;
}

/* ------------------------------------------------------------------------ */
/* Whole-slice encode / decode                                               */
/* ------------------------------------------------------------------------ */

/* Per (layer, K/V) slice result before global offsets are known. */
typedef struct {
    int status;
    float *scales;          /* [C] */
    int8_t *anchors;        /* [A][C] */
    uint8_t *tables;        /* compact, slice-local */
    uint32_t *table_size;   /* [C] */
    uint64_t tables_bytes;
    uint16_t *words;        /* all streams, padded, slice-local */
    uint64_t *stream_words; /* [spans_total * NG], padded word counts */
    uint64_t n_words;
    int32_t *esc;           /* slice escapes */
    uint32_t *stream_esc;   /* [spans_total * NG] */
    uint64_t n_esc;
} slice_enc;

static void slice_free(slice_enc *s)
{
    free(s->scales);
    free(s->anchors);
    free(s->tables);
    free(s->table_size);
    free(s->words);
    free(s->stream_words);
    free(s->esc);
    free(s->stream_esc);
    memset(s, 0, sizeof(*s));
}

/* Non-anchor tokens of span [t0, t1) (absolute token indices), ascending. */
static uint32_t span_steps(const cgo_config *cfg, uint32_t t0, uint32_t t1, uint32_t *tok)
{
    uint32_t n = 0;
    for (uint32_t t = t0; t < t1; t++)
        if (!is_anchor(cfg, t)) tok[n++] = t;
    return n;
}

static int slice_encode(const cgo_config *cfg, const geom *g, uint32_t l, const uint16_t *x, slice_enc *out)
{
    const uint32_t T = cfg->T, C = cfg->C;
    memset(out, 0, sizeof(*out));
    out->scales = malloc(sizeof(float) * C);
    out->anchors = malloc((size_t)g->A * C);
    out->table_size = malloc(sizeof(uint32_t) * C);
    out->tables = malloc((size_t)C * (2u + 2u * 256u));
    int32_t *q = malloc(sizeof(int32_t) * (size_t)T * C);
    uint32_t *hist = calloc((size_t)C * 256u, sizeof(uint32_t));
    uint32_t *freq = malloc(sizeof(uint32_t) * (size_t)C * 256u);
    int32_t *lo = malloc(sizeof(int32_t) * C), *hi = malloc(sizeof(int32_t) * C);
    uint32_t *tok = malloc(sizeof(uint32_t) * cfg->tokens_per_stream);
    uint64_t n_str = (uint64_t)g->spans_total * g->NG;
    out->stream_words = malloc(sizeof(uint64_t) * n_str);
    out->stream_esc = malloc(sizeof(uint32_t) * n_str);
    uint64_t words_cap = 0;
    for (uint32_t ch = 0; ch < g->n_chunks; ch++) {
        uint32_t len = chunk_len(cfg, ch);
        for (uint32_t s0 = 0; s0 < len; s0 += cfg->tokens_per_stream) {
            uint32_t sl = len - s0 < cfg->tokens_per_stream ? len - s0 : cfg->tokens_per_stream;
            words_cap += (((uint64_t)sl + 2u) * CGO_LANES + 7u) / 8u * 8u * g->NG;
        }
    }
    out->words = malloc(sizeof(uint16_t) * (words_cap ? words_cap : 1));
    uint64_t esc_cap = 1024;
    out->esc = malloc(sizeof(int32_t) * esc_cap);
    uint8_t *sym = malloc((size_t)cfg->tokens_per_stream * CGO_LANES);
    int st = CGO_OK;
    if (!out->scales || !out->anchors || !out->table_size || !out->tables || !q || !hist || !freq || !lo ||
        !hi || !tok || !out->stream_words || !out->stream_esc || !out->words || !out->esc || !sym) {
        st = CGO_ERR_NOMEM;
        goto done;
    }

    /* E1 */
    st = slice_anchor_scales(cfg, x, out->scales);
    if (st) goto done;
    /* E2, E3 */
    slice_quantize(cfg, g, l, x, out->scales, out->anchors, q);
    /* E4: histogram of delta symbols per channel */
    for (uint32_t t = 0; t < T; t++) {
        if (is_anchor(cfg, t)) continue;
        for (uint32_t c = 0; c < C; c++) hist[(size_t)c * 256u + symbol_of(q[(size_t)t * C + c])]++;
    }
    /* E5: normalize, write compact tables: u8 lo, u8 hi, u16 (f-1)[hi-lo+1] */
    out->tables_bytes = 0;
    for (uint32_t c = 0; c < C; c++) {
        st = cgo_normalize(hist + (size_t)c * 256u, freq + (size_t)c * 256u, &lo[c], &hi[c]);
        if (st) goto done;
        uint8_t *p = out->tables + out->tables_bytes;
        p[0] = (uint8_t)lo[c];
        p[1] = (uint8_t)hi[c];
        uint32_t sz = 2;
        for (int32_t s = lo[c]; s <= hi[c]; s++) {
            uint32_t fm1 = freq[(size_t)c * 256u + (uint32_t)s] - 1u;
            p[sz] = (uint8_t)(fm1 & 0xFFu);
            p[sz + 1] = (uint8_t)(fm1 >> 8);
            sz += 2;
        }
        out->table_size[c] = sz;
        out->tables_bytes += sz;
    }
    /* E6: one stream per (chunk, span, channel group), in that order */
    uint64_t k = 0;
    for (uint32_t ch = 0; ch < g->n_chunks; ch++) {
        uint32_t c0 = ch * cfg->chunk_tokens, len = chunk_len(cfg, ch);
        for (uint32_t s0 = 0; s0 < len; s0 += cfg->tokens_per_stream) {
            uint32_t s1 = s0 + cfg->tokens_per_stream < len ? s0 + cfg->tokens_per_stream : len;
            uint32_t nst = span_steps(cfg, c0 + s0, c0 + s1, tok);
            for (uint32_t gi = 0; gi < g->NG; gi++, k++) {
                uint32_t nesc = 0;
                for (uint32_t j = 0; j < nst; j++) {
                    for (uint32_t i = 0; i < CGO_LANES; i++) {
                        int32_t v = q[(size_t)tok[j] * C + gi * CGO_LANES + i];
                        uint32_t s = symbol_of(v);
                        sym[(size_t)j * CGO_LANES + i] = (uint8_t)s;
                        if (s == CGO_ESC) {
                            if (out->n_esc + 1 > esc_cap) {
                                esc_cap *= 2;
                                int32_t *ne = realloc(out->esc, sizeof(int32_t) * esc_cap);
                                if (!ne) {
                                    st = CGO_ERR_NOMEM;
                                    goto done;
                                }
                                out->esc = ne;
                            }
                            out->esc[out->n_esc++] = v;
                            nesc++;
                        }
                    }
                }
                uint64_t nw = 0;
                st = cgo_rans_encode(CGO_LANES, nst, sym, freq + (size_t)gi * CGO_LANES * 256u,
                                     out->words + out->n_words, words_cap - out->n_words, &nw);
                if (st) goto done;
                uint64_t padded = (nw + 7u) / 8u * 8u;
                for (uint64_t z = nw; z < padded; z++) out->words[out->n_words + z] = 0;
                out->n_words += padded;
                out->stream_words[k] = padded;
                out->stream_esc[k] = nesc;
            }
        }
    }
done:
    free(q);
    free(hist);
    free(freq);
    free(lo);
    free(hi);
    free(tok);
    free(sym);
    out->status = st;
    return st;
}

/* Decode one (layer, K/V) slice.  tables/off: the slice's C tables and their
 * byte offsets relative to `tables`; streams k0.. of the object. */
static int slice_decode(const cgo_config *cfg, const geom *g, uint32_t l, const cgo_encoded *in, uint64_t slice,
                        uint16_t *y)
{
    const uint32_t T = cfg->T, C = cfg->C;
    const float step = cfg->step[l];
    const float *scales = in->scales + slice * C;
    const int8_t *anch = in->anchors;
    uint32_t *freq = calloc((size_t)C * 256u, sizeof(uint32_t));
    int32_t *lo = malloc(sizeof(int32_t) * C), *hi = malloc(sizeof(int32_t) * C);
    uint32_t *tok = malloc(sizeof(uint32_t) * cfg->tokens_per_stream);
    uint8_t *sym = malloc((size_t)cfg->tokens_per_stream * CGO_LANES);
    int st = CGO_OK;
    if (!freq || !lo || !hi || !tok || !sym) {
        st = CGO_ERR_NOMEM;
        goto done;
    }
    /* tables */
    for (uint32_t c = 0; c < C; c++) {
        uint64_t ti = slice * C + c;
        uint32_t b = in->table_off[ti], e = in->table_off[ti + 1];
        if (e < b + 2u || e > in->tables_cap) {
            st = CGO_ERR_CORRUPT;
            goto done;
        }
        const uint8_t *p = in->tables + b;
        lo[c] = p[0];
        hi[c] = p[1];
        if (lo[c] > hi[c]) { /* empty table */
            if (e != b + 2u) {
                st = CGO_ERR_CORRUPT;
                goto done;
            }
            continue;
        }
        if (e - b != 2u + 2u * (uint32_t)(hi[c] - lo[c] + 1)) {
            st = CGO_ERR_CORRUPT;
            goto done;
        }
        uint64_t sum = 0;
        for (int32_t s = lo[c]; s <= hi[c]; s++) {
            uint32_t o = 2u + 2u * (uint32_t)(s - lo[c]);
            uint32_t fs = (uint32_t)p[o] | ((uint32_t)p[o + 1] << 8);
            freq[(size_t)c * 256u + (uint32_t)s] = fs + 1u;
            sum += fs + 1u;
        }
        if (sum != CGO_M) {
            st = CGO_ERR_CORRUPT;
            goto done;
        }
    }
    /* anchors */
    for (uint32_t t = 0; t < T; t++) {
        if (!is_anchor(cfg, t)) continue;
        uint64_t ai = anchor_index(cfg, g, (uint32_t)slice, t);
        for (uint32_t c = 0; c < C; c++)
            y[(size_t)t * C + c] = cgo_f32_to_f16((float)anch[ai + c] * scales[c]);
    }
    /* streams */
    for (uint32_t ch = 0; ch < g->n_chunks; ch++) {
        uint32_t c0 = ch * cfg->chunk_tokens, len = chunk_len(cfg, ch);
        for (uint32_t s0 = 0; s0 < len; s0 += cfg->tokens_per_stream) {
            uint32_t s1 = s0 + cfg->tokens_per_stream < len ? s0 + cfg->tokens_per_stream : len;
            uint32_t nst = span_steps(cfg, c0 + s0, c0 + s1, tok);
            for (uint32_t gi = 0; gi < g->NG; gi++) {
                uint64_t k = stream_index(cfg, g, ch, (uint32_t)slice, s0 / cfg->tokens_per_stream, gi);
                uint64_t b = in->stream_off[k], e = in->stream_off[k + 1];
                if (e < b || (b & 15u) || (e & 15u) || e > in->payload_cap) {
                    st = CGO_ERR_CORRUPT;
                    goto done;
                }
                const uint16_t *w = (const uint16_t *)(in->payload + b);
                uint64_t padded = (e - b) / 2u, used = 0;
                int32_t flo[CGO_LANES], fhi[CGO_LANES];
                for (uint32_t i = 0; i < CGO_LANES; i++) {
                    flo[i] = lo[gi * CGO_LANES + i];
                    fhi[i] = hi[gi * CGO_LANES + i];
                }
                st = cgo_rans_decode(CGO_LANES, nst, w, padded, freq + (size_t)gi * CGO_LANES * 256u, flo, fhi,
                                     sym, &used);
                if (st) goto done;
                if ((used + 7u) / 8u * 8u != padded) {
                    st = CGO_ERR_CORRUPT;
                    goto done;
                }
                for (uint64_t z = used; z < padded; z++)
                    if (w[z]) {
                        st = CGO_ERR_CORRUPT;
                        goto done;
                    }
                uint32_t eb = in->esc_off[k], ee = in->esc_off[k + 1], ep = eb;
                if (ee < eb || ee > in->escapes_cap) {
                    st = CGO_ERR_CORRUPT;
                    goto done;
                }
                for (uint32_t j = 0; j < nst; j++) {
                    uint32_t t = tok[j];
                    uint64_t ai = anchor_index(cfg, g, (uint32_t)slice, t);
                    for (uint32_t i = 0; i < CGO_LANES; i++) {
                        uint32_t c = gi * CGO_LANES + i, s = sym[(size_t)j * CGO_LANES + i];
                        int32_t qv;
                        if (s == CGO_ESC) {
                            if (ep >= ee) {
                                st = CGO_ERR_CORRUPT;
                                goto done;
                            }
                            qv = in->escapes[ep++];
                        } else {
                            qv = (int32_t)s - 127;
                        }
                        float xa = (float)anch[ai + c] * scales[c];
                        float dq = (float)qv * step;
                        y[(size_t)t * C + c] = cgo_f32_to_f16(xa + dq);
                    }
                }
                if (ep != ee) {
                    st = CGO_ERR_CORRUPT;
                    goto done;
                }
            }
        }
    }
done:
    free(freq);
    free(lo);
    free(hi);
    free(tok);
    free(sym);
    return st;
}

/* ------------------------------------------------------------------------ */
/* Public encode / decode over all slices, optionally threaded               */
/* ------------------------------------------------------------------------ */

typedef struct {
    const cgo_config *cfg;
    const geom *g;
    const uint16_t *kv;
    uint16_t *out;
    const cgo_encoded *in;
    slice_enc *slices;
    uint32_t n_slices, next_stride, first;
    int status;
} work;

static void *enc_worker(void *arg)
{
    work *w = arg;
    const uint64_t sl_vals = (uint64_t)w->cfg->T * w->cfg->C;
    for (uint32_t s = w->first; s < w->n_slices; s += w->next_stride) {
        int st = slice_encode(w->cfg, w->g, s / 2u, w->kv + s * sl_vals, &w->slices[s]);
        if (st && !w->status) w->status = st;
    }
    return NULL;
}

static void *dec_worker(void *arg)
{
    work *w = arg;
    const uint64_t sl_vals = (uint64_t)w->cfg->T * w->cfg->C;
    for (uint32_t s = w->first; s < w->n_slices; s += w->next_stride) {
        int st = slice_decode(w->cfg, w->g, s / 2u, w->in, s, w->out + s * sl_vals);
        if (st && !w->status) w->status = st;
    }
    return NULL;
}

static int run_threads(work *proto, void *(*fn)(void *), int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if ((uint32_t)nthreads > proto->n_slices) nthreads = (int)proto->n_slices;
    work *ws = calloc((size_t)nthreads, sizeof(work));
    pthread_t *th = calloc((size_t)nthreads, sizeof(pthread_t));
    if (!ws || !th) {
        free(ws);
        free(th);
        return CGO_ERR_NOMEM;
    }
    for (int i = 0; i < nthreads; i++) {
        ws[i] = *proto;
        ws[i].first = (uint32_t)i;
        ws[i].next_stride = (uint32_t)nthreads;
        ws[i].status = 0;
    }
    char *started = calloc((size_t)nthreads, 1);
    if (!started) {
        free(ws);
        free(th);
        return CGO_ERR_NOMEM;
    }
    for (int i = 1; i < nthreads; i++) started[i] = pthread_create(&th[i], NULL, fn, &ws[i]) == 0;
    fn(&ws[0]);
    /* a share whose thread could not be started runs here */
    for (int i = 1; i < nthreads; i++)
        if (!started[i]) fn(&ws[i]);
    for (int i = 1; i < nthreads; i++)
        if (started[i]) pthread_join(th[i], NULL);
    free(started);
    int st = CGO_OK;
    for (int i = 0; i < nthreads; i++)
        if (ws[i].status && !st) st = ws[i].status;
    free(ws);
    free(th);
    return st;
}

/*
 * Encode a whole cache kv [L][2][T][C] (fp16 bits).  Layout of the object
 * (per-chunk sections are chunk-major, so one chunk is one contiguous range
 * of each of them):
 *   anchors    int8  [chunk][L][2][anchor rows of the chunk][C]
 *   scales     fp32  [L][2][C]
 *   tables     per (l, kv, c) in that order: u8 lo, u8 hi, then the 16-bit
 *              little-endian values f_s - 1 for s = lo..hi; an empty table is
 *              lo = 1, hi = 0 (2 bytes)
 *   table_off  u32   [L*2*C + 1] byte offsets of the tables
 *   payload    streams ordered by (chunk, l, kv, span, group); a stream is
 *              its 16-bit words followed by zero words up to a multiple of 8
 *   stream_off u64   [n_streams + 1] byte offsets (multiples of 16)
 *   escapes    int32 escaped q values, per stream in (step, lane) order
 *   esc_off    u32   [n_streams + 1]
 */
int cgo_encode(const cgo_config *cfg, const uint16_t *kv, cgo_encoded *out, cgo_sizes *sizes, int nthreads)
{
    int st = check_config(cfg);
    if (st) return st;
    if (!kv || !out || !sizes) return CGO_ERR_INVALID_ARG;
    geom g;
    make_geom(cfg, &g);
    const uint32_t n_slices = cfg->L * 2u;
    slice_enc *sl = calloc(n_slices, sizeof(slice_enc));
    if (!sl) return CGO_ERR_NOMEM;
    work w = {cfg, &g, kv, NULL, NULL, sl, n_slices, 1, 0, 0};
    st = run_threads(&w, enc_worker, nthreads);
    if (st) goto done;
    /* global offsets and copies: tables and scales slice by slice, then the
     * per-chunk sections chunk-major */
    uint64_t toff = 0, poff = 0, eoff = 0, k = 0;
    const uint64_t n_sl_str = (uint64_t)g.spans_total * g.NG;
    uint64_t *wpre = malloc(sizeof(uint64_t) * (n_sl_str + 1) * n_slices);
    uint64_t *epre = malloc(sizeof(uint64_t) * (n_sl_str + 1) * n_slices);
    if (!wpre || !epre) {
        free(wpre);
        free(epre);
        st = CGO_ERR_NOMEM;
        goto done;
    }
    for (uint32_t s = 0; s < n_slices; s++) {
        slice_enc *e = &sl[s];
        memcpy(out->scales + (uint64_t)s * cfg->C, e->scales, sizeof(float) * cfg->C);
        if (toff + e->tables_bytes > out->tables_cap) {
            st = CGO_ERR_RANGE;
            break;
        }
        memcpy(out->tables + toff, e->tables, e->tables_bytes);
        for (uint32_t c = 0; c < cfg->C; c++) {
            out->table_off[(uint64_t)s * cfg->C + c] = (uint32_t)toff;
            toff += e->table_size[c];
        }
        uint64_t *wp = wpre + (uint64_t)s * (n_sl_str + 1), *ep = epre + (uint64_t)s * (n_sl_str + 1);
        wp[0] = ep[0] = 0;
        for (uint64_t j = 0; j < n_sl_str; j++) {
            wp[j + 1] = wp[j] + e->stream_words[j];
            ep[j + 1] = ep[j] + e->stream_esc[j];
        }
    }
    uint64_t arow = 0;
    for (uint32_t ch = 0; ch < g.n_chunks && !st; ch++) {
        uint32_t len = chunk_len(cfg, ch);
        uint32_t apc = ceil_div(len, cfg->G), spc = ceil_div(len, cfg->tokens_per_stream);
        for (uint32_t s = 0; s < n_slices && !st; s++) {
            slice_enc *e = &sl[s];
            memcpy(out->anchors + arow * cfg->C, e->anchors + (uint64_t)ch * g.anchors_per_full_chunk * cfg->C,
                   (size_t)apc * cfg->C);
            arow += apc;
            const uint64_t *wp = wpre + (uint64_t)s * (n_sl_str + 1), *ep = epre + (uint64_t)s * (n_sl_str + 1);
            uint64_t j0 = (uint64_t)ch * g.spans_full * g.NG, j1 = j0 + (uint64_t)spc * g.NG;
            for (uint64_t j = j0; j < j1; j++, k++) {
                uint64_t nb = 2u * e->stream_words[j], ne = e->stream_esc[j];
                if (poff + nb > out->payload_cap || eoff + ne > out->escapes_cap) {
                    st = CGO_ERR_RANGE;
                    break;
                }
                out->stream_off[k] = poff;
                out->esc_off[k] = (uint32_t)eoff;
                memcpy(out->payload + poff, e->words + wp[j], nb);
                memcpy(out->escapes + eoff, e->esc + ep[j], sizeof(int32_t) * ne);
                poff += nb;
                eoff += ne;
            }
        }
    }
    free(wpre);
    free(epre);
    if (st) goto done;
    out->table_off[g.n_tables] = (uint32_t)toff;
    out->stream_off[g.n_streams] = poff;
    out->esc_off[g.n_streams] = (uint32_t)eoff;
    sizes->payload_bytes = poff;
    sizes->tables_bytes = toff;
    sizes->n_escapes = eoff;
    sizes->total_bytes = poff + toff + 4u * eoff + (uint64_t)n_slices * g.A * cfg->C + 4u * (uint64_t)n_slices * cfg->C +
                         4u * (g.n_tables + 1u) + 8u * (g.n_streams + 1u) + 4u * (g.n_streams + 1u);
done:
    for (uint32_t s = 0; s < n_slices; s++) slice_free(&sl[s]);
    free(sl);
    return st;
}

int cgo_decode(const cgo_config *cfg, const cgo_encoded *in, uint16_t *kv_out, int nthreads)
{
    int st = check_config(cfg);
    if (st) return st;
    if (!in || !kv_out) return CGO_ERR_INVALID_ARG;
    geom g;
    make_geom(cfg, &g);
    work w = {cfg, &g, NULL, kv_out, in, NULL, cfg->L * 2u, 1, 0, 0};
    return run_threads(&w, dec_worker, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Stage-level entry points used by the oracle's own tests                   */
/* ------------------------------------------------------------------------ */

/* E1 for a whole cache: scales [L][2][C]. */
int cgo_anchor_scales(const cgo_config *cfg, const uint16_t *kv, float *scales)
{
    int st = check_config(cfg);
    if (st) return st;
    for (uint32_t s = 0; s < cfg->L * 2u; s++) {
        st = slice_anchor_scales(cfg, kv + (uint64_t)s * cfg->T * cfg->C, scales + (uint64_t)s * cfg->C);
        if (st) return st;
    }
    return CGO_OK;
}

/* E2 + E3 for a whole cache: anchors [L][2][A][C] (each slice's anchor rows
 * in token order, not the object's chunk-major plane), q [L][2][T][C]. */
int cgo_quantize(const cgo_config *cfg, const uint16_t *kv, const float *scales, int8_t *anchors, int32_t *q)
{
    int st = check_config(cfg);
    if (st) return st;
    geom g;
    make_geom(cfg, &g);
    for (uint32_t s = 0; s < cfg->L * 2u; s++) {
        uint64_t sv = (uint64_t)s * cfg->T * cfg->C;
        slice_quantize(cfg, &g, s / 2u, kv + sv, scales + (uint64_t)s * cfg->C, anchors + (uint64_t)s * g.A * cfg->C,
                       q + sv);
    }
    return CGO_OK;
}

/* E4 for a whole cache: hist [L*2*C][256] over delta symbols. */
int cgo_histograms(const cgo_config *cfg, const int32_t *q, uint32_t *hist)
{
    int st = check_config(cfg);
    if (st) return st;
    const uint32_t T = cfg->T, C = cfg->C;
    memset(hist, 0, sizeof(uint32_t) * (size_t)cfg->L * 2u * C * 256u);
    for (uint32_t s = 0; s < cfg->L * 2u; s++)
        for (uint32_t t = 0; t < T; t++) {
            if (is_anchor(cfg, t)) continue;
            for (uint32_t c = 0; c < C; c++)
                hist[((size_t)s * C + c) * 256u + symbol_of(q[((size_t)s * T + t) * C + c])]++;
        }
    return CGO_OK;
}

/* 1 if token t is an anchor under cfg (chunked groups), else 0. */
int cgo_is_anchor(const cgo_config *cfg, uint32_t t) { return is_anchor(cfg, t); }

/* Per-layer steps by layer thirds: bin(l) = floor(3 l / L) picks base[bin]. */
void cgo_layer_steps(uint32_t L, const float base[3], float mult, float *step)
{
    for (uint32_t l = 0; l < L; l++) step[l] = base[(3u * l) / L] * mult;
}
