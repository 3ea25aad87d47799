// cg_encode.cu -- GPU encoder of the KV-cache codec (sm_103a).
//
// Pipeline (the CacheGen compression pipeline: anchor/delta, layer-binned
// quantization, arithmetic coding with per-(layer, channel) statistics;
// "CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §1 and §2.1):
//   k_stats   one block per (32-channel group, layer, K/V): anchor absmax ->
//             scale; then every warp walks its own run of row tiles, staged
//             by cp.async in a shared-memory ring: int8 anchors, delta
//             quantization (multiplication by the once-rounded inverse of
//             the scale / step), shared-memory histograms (lane = channel,
//             bank = lane: conflict-free atomics), the u8 symbol of every
//             delta (kept in the workspace for the coder), escape counts per
//             stream; normalization of the 32 histograms to 16-bit frequency
//             tables (warp-cooperative).
//   k_scan    exclusive scans of table sizes, escape counts and stream sizes
//             (block sums, then each block scans its tile).
//   k_encode  one warp per stream (lane = channel): interleaved range ANS
//             over the stored symbols of the span's delta tokens in reverse
//             (a group with an escape is quantized again from its fp16
//             values, for the escape values), words written backwards into
//             a per-stream scratch region, escapes placed from the end of
//             the stream's escape range.
//   k_pack    one warp per stream: copies the stream words into the
//             payload at its prefix-sum offset, zero-padded to 16 bytes.
#include <cuda_fp16.h>
#include <string.h>

#include "cg_internal.cuh"

namespace cg {

struct StepTable {
    float v[CG_MAX_LAYERS];
};

struct EncArgs {
    Geom g;
    const uint16_t *kv;
    int8_t *anchors;
    float *scales;
    uint8_t *tables;
    uint32_t *table_off;
    uint8_t *payload;
    uint64_t *stream_off;
    int32_t *escapes;
    uint32_t *esc_off;
    uint64_t tables_cap, payload_cap, escapes_cap;
    // workspace
    uint16_t *ftab;        // [n_tables][256] f - 1
    uint32_t *tlohi;       // [n_tables] lo | hi << 8
    uint32_t *twidth;      // [n_tables] compact table bytes
    uint32_t *esc_count;   // [n_streams]
    uint32_t *words_count; // [n_streams]
    uint16_t *scratch;     // [n_streams][region_words]
    const uint8_t *sym;    // [slice][T][C] delta symbols of this level (written by the statistics pass)
    uint64_t region_words;
    cg_sizes *dsizes;
    uint32_t *status;
};

// Quality levels one multi-level encode can produce (the pages store each
// chunk at three: "CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §2.2).
constexpr uint32_t kMaxLevels = 4;

// Per-level outputs of the statistics pass: a multi-level encode counts the
// symbols of every level in one read of the cache.  Level l quantizes with
// the layer's step times mult[l].
struct StatsLevels {
    uint16_t *ftab[kMaxLevels];
    uint32_t *tlohi[kMaxLevels], *twidth[kMaxLevels], *esc_count[kMaxLevels];
    float mult[kMaxLevels];
    // optional raw counts [n_tables][256] of level 0's delta symbols and of
    // the anchors (q_a + 127), for the grouping ablation; null otherwise
    uint32_t *raw_delta, *raw_anchor;
    // every delta's symbol, [level][slice][T][C] (level l at sym + l * sym_stride;
    // anchor rows are not written), so that the coder does not quantize again
    uint8_t *sym;
    uint64_t sym_stride;
};

// Prefix scans: kScanThreads threads per block, kScanRows rows each.
constexpr uint32_t kScanThreads = 256, kScanRows = 16, kScanTile = kScanThreads * kScanRows;

// Workspace carving (256-byte aligned pieces): per-level tables and counts,
// one scratch region shared by the levels (they are coded one after another).
struct WsLayout {
    uint64_t ftab[kMaxLevels], tlohi[kMaxLevels], twidth[kMaxLevels], esc_count[kMaxLevels],
        words_count[kMaxLevels], dsizes[kMaxLevels];
    uint64_t scan_part, scratch, sym, sym_stride, total, region_words;
};

static WsLayout ws_layout(const Geom &g, uint32_t levels = 1) {
    WsLayout w;
    uint64_t o = 0;
    auto take = [&](uint64_t bytes) {
        uint64_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    w.region_words = round_up((uint64_t)kLanes * (g.tps + 2u), 8);
    for (uint32_t l = 0; l < levels; l++) {
        w.ftab[l] = take(g.n_tables * 256u * 2u);
        w.tlohi[l] = take(g.n_tables * 4u);
        w.twidth[l] = take(g.n_tables * 4u);
        w.esc_count[l] = take(g.n_streams * 4u);
        w.words_count[l] = take(g.n_streams * 4u);
        w.dsizes[l] = take(sizeof(cg_sizes));
    }
    const uint64_t most = g.n_tables > g.n_streams ? g.n_tables : g.n_streams;
    w.scan_part = take(((most + kScanTile - 1) / kScanTile + 1) * 8u);
    w.scratch = take(g.n_streams * w.region_words * 2u);
    w.sym_stride = round_up((uint64_t)g.n_slices * g.T * g.C, 256);
    w.sym = take(w.sym_stride * levels);
    w.total = o;
    return w;
}

__device__ __forceinline__ float ld_half(const uint16_t *p) { return __half2float(__ushort_as_half(*p)); }

__device__ __forceinline__ uint32_t symbol_of(int q) {
    return (uint32_t)(q + 127) <= 254u ? (uint32_t)(q + 127) : kEsc;
}

// Warp reductions in one instruction each (integer add / min / max).
__device__ __forceinline__ uint32_t warp_sum(uint32_t v) { return __reduce_add_sync(kFull, v); }

// (value, symbol) argmax, smallest symbol on a tie.
__device__ __forceinline__ void warp_argmax(uint32_t &v, uint32_t &s) {
    const uint32_t m = __reduce_max_sync(kFull, v);
    s = __reduce_min_sync(kFull, v == m ? s : 0xFFFFFFFFu);
    v = m;
}

constexpr int kStatsWarps = 16;
// Staging of the statistics pass.  A slice's tokens are cut into tiles that
// never cross a chunk: R rows each, R a whole number of groups when a group
// fits a slot (such tiles start on an anchor row), else one slot of rows.
// Every warp takes a contiguous run of tiles and copies them (the block's 32
// channels: 64 bytes a row) with cp.async into a ring of kStStages
// shared-memory slots, kStStages - 1 tiles ahead of the one it counts.
constexpr uint32_t kStSlotRows = 30;
constexpr uint32_t kStStages = 2;
constexpr uint32_t kStRowBytes = kLanes * 2u;
constexpr uint32_t kStSlotBytes = kStSlotRows * kStRowBytes;              // 1920 B
constexpr uint32_t kStRingBytes = kStatsWarps * kStStages * kStSlotBytes;  // 60 KB
constexpr uint32_t kE1Batch = 8;  // 16-byte anchor-row loads in flight per lane

template <uint32_t NL>
constexpr uint32_t stats_smem_bytes() {
    return NL * 256u * kLanes * 4u + kStRingBytes;
}

// Token of anchor row r (over all chunks of one slice).
__device__ __forceinline__ uint32_t anchor_token(const Geom &g, uint32_t r) {
    const uint32_t ch = r / g.apc_full;
    return ch * g.chunk + (r - ch * g.apc_full) * g.G;
}

__device__ __forceinline__ __half2 u2h2(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}
__device__ __forceinline__ uint32_t h22u(__half2 h) {
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}
__device__ __forceinline__ float h2f(uint16_t u) { return __half2float(__ushort_as_half(u)); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(__cvta_generic_to_global(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most kStStages - 1 of this thread's copy groups are pending.
__device__ __forceinline__ void cp_async_wait_ring() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kStStages - 1u) : "memory");
}

// Copy rows [t0, t0 + n) (n <= kStSlotRows) of the block's 32 channels into
// the slot at shared address slot (row k at slot + 64 k) in 16-byte pieces:
// the lane's pieces are rows lane / 4 + 8 k, quarter lane % 4, so it starts
// from xl = (row lane / 4, channel 8 (lane % 4)) of the group and C8 = 8 C.
__device__ __forceinline__ void stage_tile(uint32_t slot, const uint16_t *xl, uint32_t C, uint64_t C8, uint32_t t0,
                                           uint32_t n, uint32_t lane) {
    const uint16_t *src = xl + (uint64_t)t0 * C;
    const uint32_t dst = slot + lane * 16u, r = lane >> 2;
#pragma unroll
    for (uint32_t k = 0; k < (kStSlotRows + 7u) / 8u; k++)
        if (r + 8u * k < n) cp_async16(dst + k * 512u, src + k * C8);
}

// Walk over the tiles of one slice: tile (ch, j) holds the chunk-relative
// rows [j R, min((j + 1) R, clen)) of chunk ch.
struct TileCursor {
    uint32_t ch, j, clen;
    __device__ __forceinline__ void init(const Geom &g, uint32_t tpc, uint32_t u) {
        ch = u / tpc;
        j = u - ch * tpc;
        clen = g.chunk_len(ch);
    }
    __device__ __forceinline__ void next(const Geom &g, uint32_t R) {
        j++;
        if (j * R >= clen) {
            ch++;
            j = 0;
            clen = g.chunk_len(ch);
        }
    }
    __device__ __forceinline__ uint32_t first(uint32_t R) const { return j * R; }
    __device__ __forceinline__ uint32_t rows(uint32_t R) const { return min(R, clen - j * R); }
};

// floor(n * 65536 / N) for n <= N, exactly: a float estimate (within one of
// the quotient, which is at most 65536, for rN = 1/N rounded) corrected by
// the integer remainder.
__device__ __forceinline__ uint32_t scaled_count(uint32_t n, uint32_t N, float rN) {
    uint32_t q = __float2uint_rz(__fmul_rn(__fmul_rn(__uint2float_rn(n), rN), 65536.f));
    const int64_t r = (int64_t)((uint64_t)n << 16) - (int64_t)((uint64_t)q * N);
    if (r < 0) q--;
    else if (r >= (int64_t)N) q++;
    return q;
}

// Symbol of delta d quantized with inverse step inv: q + 127, or the escape
// symbol for |q| > 127.
__device__ __forceinline__ uint32_t delta_symbol(float d, float inv) {
    const int q = __float2int_rn(__fmul_rn(d, inv));
    return min((uint32_t)q + 127u, kEsc);
}

// Quantized anchor value of v: clamp(rint(v / s_a), -127, 127).
__device__ __forceinline__ float anchor_q(float v, float inv_sa) {
    return fminf(fmaxf(rintf(__fmul_rn(v, inv_sa)), -127.f), 127.f);
}

// Count m delta rows (row i at rows[i * 32], chunk-relative token pos + i)
// against anchor value xa at every level and store their symbols (row i of
// level l at sp + l * sym_stride + i * C); escapes, which are rare, are then
// counted per stream in a second look at the same rows.
template <uint32_t NL, uint32_t kM_, uint32_t kC>
__device__ __forceinline__ void count_rows(const Geom &g, const StatsLevels &lv, const uint16_t *rows, uint32_t m,
                                           float xa, const float (&inv_step)[NL], uint32_t *hl, uint8_t *sp,
                                           float &nan_acc, uint32_t slice, uint32_t grp, uint32_t ch, uint32_t pos) {
    const uint32_t cnt = kM_ ? kM_ : m;
    const uint32_t C = kC ? kC : g.C;
    bool esc = false;
    auto row = [&](uint32_t i) {
        const float v = h2f(rows[i * kLanes]);
        nan_acc = __fmaf_rn(v, 0.f, nan_acc);  // v * 0 is NaN exactly for a NaN or infinite v
        const float d = __fsub_rn(v, xa);
#pragma unroll
        for (uint32_t l = 0; l < NL; l++) {
            const uint32_t s = delta_symbol(d, inv_step[l]);
            atomicAdd(hl + l * 256u * kLanes + s * kLanes, 1u);
            sp[l * lv.sym_stride + (uint64_t)i * C] = (uint8_t)s;
            esc = esc || s == kEsc;
        }
    };
    if constexpr (kM_ > 0) {
#pragma unroll
        for (uint32_t i = 0; i < kM_; i++) row(i);
    } else {
#pragma unroll 3
        for (uint32_t i = 0; i < m; i++) row(i);
    }
    if (__any_sync(kFull, esc)) {
        for (uint32_t i = 0; i < cnt; i++) {
            const float d = __fsub_rn(h2f(rows[i * kLanes]), xa);
#pragma unroll
            for (uint32_t l = 0; l < NL; l++)
                if (delta_symbol(d, inv_step[l]) == kEsc)
                    atomicAdd(&lv.esc_count[l][g.stream_index(ch, slice, (pos + i) / g.tps, grp)], 1u);
        }
    }
}

// NL levels in one pass: their histograms side by side in dynamic shared
// memory (NL x 32 KB), then the warps' staging rings; anchors and scales are
// the same for every level.  kC = 1024 fixes the row stride of the symbol
// and anchor stores at compile time (0: runtime); kRaw adds the raw counts
// of the grouping ablation.
template <uint32_t NL, uint32_t kC, bool kRaw>
__global__ void __launch_bounds__(kStatsWarps * 32, NL == 1 ? 2 : 1) k_stats(EncArgs a, StepTable st, StatsLevels lv) {
    const Geom &g = a.g;
    const uint32_t grp = blockIdx.x, slice = blockIdx.y;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t c = grp * kLanes + lane;
    const uint16_t *xg = a.kv + (uint64_t)slice * g.T * g.C + grp * kLanes;  // channel 0 of the group
    const float step = st.v[slice >> 1];

    extern __shared__ __align__(16) uint32_t hist[];  // [level][symbol][lane], then the rings
    __shared__ float red[kStatsWarps][kLanes];
    __shared__ float s_scale[kLanes];
    uint8_t *ring = reinterpret_cast<uint8_t *>(hist + NL * 256u * kLanes) + warp * kStStages * kStSlotBytes;
    const uint32_t ring_s = smem_u32(ring);

    // The warp's run of tiles; its first tiles' copies are in flight during E1.
    const uint32_t G = g.G;
    const uint32_t R = G <= kStSlotRows ? G * (kStSlotRows / G) : kStSlotRows;
    const uint32_t tpc = ceil_div(g.chunk, R);
    const uint32_t U = (g.n_chunks - 1u) * tpc + ceil_div(g.last_len, R);
    const uint32_t Uw = ceil_div(U, kStatsWarps);
    const uint32_t u0 = min(warp * Uw, U), nt = min(U - u0, Uw);
    const uint16_t *xl = xg + (uint64_t)(lane >> 2) * g.C + (lane & 3u) * 8u;
    const uint64_t C8 = 8ull * g.C;
    TileCursor in, cur;  // next tile to copy, next tile to count
    in.init(g, tpc, u0);
    cur = in;
#pragma unroll
    for (uint32_t j = 0; j + 1u < kStStages; j++) {
        if (j < nt) {
            stage_tile(ring_s + j * kStSlotBytes, xl, g.C, C8, in.ch * g.chunk + in.first(R), in.rows(R), lane);
            in.next(g, R);
        }
        cp_async_commit();
    }
    // A run that starts inside a group (groups longer than a slot) needs
    // that group's anchor value.
    const uint32_t gpos0 = cur.first(R) % G;
    const uint16_t a_raw = (nt && gpos0) ? xg[(uint64_t)(cur.ch * g.chunk + cur.first(R) - gpos0) * g.C + lane]
                                         : (uint16_t)0;

    for (uint32_t i = threadIdx.x; i < NL * 256u * kLanes; i += blockDim.x) hist[i] = 0;

    // E1: absmax over this call's anchor rows -> scale = absmax / 127.  A
    // lane loads 8 channels (16 bytes) of one row, a warp 8 rows at a time;
    // |v| and max are exact in fp16.
    const uint32_t A = (uint32_t)g.A, q = lane & 3u;
    __half2 m2[4];
#pragma unroll
    for (int k = 0; k < 4; k++) m2[k] = __float2half2_rn(0.f);
    for (uint32_t r0 = warp * 8u + (lane >> 2); r0 < A; r0 += kStatsWarps * 8u * kE1Batch) {
        uint4 v[kE1Batch];
#pragma unroll
        for (uint32_t i = 0; i < kE1Batch; i++) {
            const uint32_t r = r0 + i * kStatsWarps * 8u;
            v[i] = r < A ? *reinterpret_cast<const uint4 *>(xg + (uint64_t)anchor_token(g, r) * g.C + q * 8u)
                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (uint32_t i = 0; i < kE1Batch; i++) {
            m2[0] = __hmax2(m2[0], __habs2(u2h2(v[i].x)));
            m2[1] = __hmax2(m2[1], __habs2(u2h2(v[i].y)));
            m2[2] = __hmax2(m2[2], __habs2(u2h2(v[i].z)));
            m2[3] = __hmax2(m2[3], __habs2(u2h2(v[i].w)));
        }
    }
#pragma unroll
    for (int k = 0; k < 4; k++)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) m2[k] = __hmax2(m2[k], u2h2(__shfl_xor_sync(kFull, h22u(m2[k]), o)));
    if (lane < 4u) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            red[warp][q * 8u + 2u * k] = __low2float(m2[k]);
            red[warp][q * 8u + 2u * k + 1u] = __high2float(m2[k]);
        }
    }
    __syncthreads();
    if (warp == 0) {
        float m = red[0][lane];
        for (int w = 1; w < kStatsWarps; w++) m = fmaxf(m, red[w][lane]);
        float s = m > 0.f ? __fdiv_rn(m, 127.f) : 1.f;
        s_scale[lane] = s;
        a.scales[(uint64_t)slice * g.C + c] = s;
    }
    __syncthreads();
    const float sa = s_scale[lane];

    // E2 + E3 + E4 over the warp's tiles: an anchor row quantizes and stores
    // the group's anchor; a delta row counts its symbol at every level.
    const float inv_sa = __fdiv_rn(1.f, sa);  // one rounding each
    float inv_step[NL];
#pragma unroll
    for (uint32_t l = 0; l < NL; l++) inv_step[l] = __fdiv_rn(1.f, __fmul_rn(step, lv.mult[l]));
    uint32_t *hl = hist + lane;
    uint32_t ach = 0xFFFFFFFFu;  // chunk of the cached anchor base
    uint64_t abase = 0;          // anchor row of group 0 of chunk ach
    float xa = gpos0 ? __fmul_rn(anchor_q(h2f(a_raw), inv_sa), sa) : 0.f;
    float nan_acc = 0.f;
    // tiles are consecutive in token order: each starts where the one before ends
    uint32_t t0_in = in.ch * g.chunk + in.first(R);
    uint8_t *spt = lv.sym + ((uint64_t)slice * g.T + cur.ch * g.chunk + cur.first(R)) * (kC ? kC : g.C) + c;
    for (uint32_t t = 0; t < nt; t++) {
        if (t + kStStages - 1u < nt) {
            const uint32_t rr = in.rows(R);
            stage_tile(ring_s + ((t + kStStages - 1u) % kStStages) * kStSlotBytes, xl, g.C, C8, t0_in, rr, lane);
            t0_in += rr;
            in.next(g, R);
        }
        cp_async_commit();
        cp_async_wait_ring();
        __syncwarp();
        const uint16_t *rows = reinterpret_cast<const uint16_t *>(ring + (t % kStStages) * kStSlotBytes) + lane;
        const uint32_t ch = cur.ch, p = cur.first(R), n = cur.rows(R);
        if (ch != ach) {
            ach = ch;
            abase = g.chunk_anchor_row0(ch) + (uint64_t)slice * g.apc(ch);
        }
        if (G == 10 && n == kStSlotRows) {  // the common tile: three whole 10-token groups
#pragma unroll
            for (uint32_t h = 0; h < kStSlotRows / 10u; h++) {
                const uint16_t *gr = rows + h * 10u * kLanes;
                const float v0 = h2f(gr[0]);
                nan_acc = __fmaf_rn(v0, 0.f, nan_acc);
                const float qa = anchor_q(v0, inv_sa);
                a.anchors[(abase + p / 10u + h) * (kC ? kC : g.C) + c] = (int8_t)qa;
                if (kRaw)
                    atomicAdd(&lv.raw_anchor[((uint64_t)slice * g.C + c) * 256u + (uint32_t)((int)qa + 127)], 1u);
                xa = __fmul_rn(qa, sa);
                count_rows<NL, 9, kC>(g, lv, gr + kLanes, 9, xa, inv_step, hl, spt + (h * 10u + 1u) * (kC ? kC : g.C),
                                      nan_acc, slice, grp, ch, p + h * 10u + 1u);
            }
        } else {  // any group size, a chunk's last tile, or groups cut by tiles
            uint32_t gi = p / G, gpos = p - gi * G, k = 0;
            while (k < n) {
                if (gpos == 0) {  // the group's anchor row
                    const float v = h2f(rows[k * kLanes]);
                    nan_acc = __fmaf_rn(v, 0.f, nan_acc);
                    const float qa = anchor_q(v, inv_sa);
                    a.anchors[(abase + gi) * g.C + c] = (int8_t)qa;
                    if (kRaw)
                        atomicAdd(&lv.raw_anchor[((uint64_t)slice * g.C + c) * 256u + (uint32_t)((int)qa + 127)],
                                  1u);
                    xa = __fmul_rn(qa, sa);
                    k++;
                    gpos = 1;
                } else {  // the group's delta rows inside this tile (a tile ends with its chunk)
                    const uint32_t m = min(n - k, G - gpos);
                    count_rows<NL, 0, kC>(g, lv, rows + k * kLanes, m, xa, inv_step, hl,
                                          spt + (uint64_t)k * (kC ? kC : g.C), nan_acc, slice, grp, ch, p + k);
                    k += m;
                    gpos += m;
                }
                if (gpos == G) {
                    gpos = 0;
                    gi++;
                }
            }
        }
        spt += (uint64_t)n * (kC ? kC : g.C);
        cur.next(g, R);
        __syncwarp();  // the slot is read by every lane before it is refilled
    }
    const bool nonfinite = nan_acc != nan_acc;
    if (__any_sync(kFull, nonfinite) && lane == 0) flag(a.status, CG_ERR_NONFINITE);
    __syncthreads();
    if (kRaw)  // level 0's counts, [table][symbol]
        for (uint32_t i = threadIdx.x; i < 256u * kLanes; i += blockDim.x)
            lv.raw_delta[((uint64_t)slice * g.C + grp * kLanes + (i & 31u)) * 256u + (i >> 5)] = hist[i];

    // E5: normalize each channel's counts to a 16-bit table (warp per
    // (level, channel)).  A level's [symbol][channel] counts are first
    // copied channel-major into the staging ring, which is free by now, with
    // rows of 257 words: a channel's 256 counts are then spread over all
    // banks, where in place they all sit in one.
    asm volatile("cp.async.wait_all;" ::: "memory");
    uint32_t *histT = reinterpret_cast<uint32_t *>(hist + NL * 256u * kLanes);
    static_assert(kLanes * 257u * 4u <= kStRingBytes, "transposed counts fit the ring");
    for (uint32_t lvl = 0; lvl < NL; lvl++) {
      __syncthreads();
      for (uint32_t s = warp; s < 256u; s += kStatsWarps) histT[lane * 257u + s] = hist[(lvl * 256u + s) * kLanes + lane];
      __syncthreads();
      for (uint32_t j = warp; j < kLanes; j += kStatsWarps) {
        const uint32_t *hl = histT + j * 257u;
        uint16_t *ftab = lv.ftab[lvl];
        uint32_t *tlohi = lv.tlohi[lvl], *twidth = lv.twidth[lvl];
        const uint64_t table = (uint64_t)slice * g.C + grp * kLanes + j;
        uint32_t n[8], f[8];
        uint32_t N = 0, lo = 256, hi = 0;
        bool any = false;
        #pragma unroll
        for (int i = 0; i < 8; i++) {
            uint32_t s = (uint32_t)i * 32u + lane;
            n[i] = hl[s];
            N += n[i];
            if (n[i]) {
                lo = min(lo, s);
                hi = max(hi, s);
                any = true;
            }
        }
        N = warp_sum(N);
        const float rN = __frcp_rn(__uint2float_rn(N));  // used only when N > 0
        lo = __reduce_min_sync(kFull, lo);
        hi = __reduce_max_sync(kFull, hi);
        any = __any_sync(kFull, any);
        if (!any) {
            if (lane == 0) {
                tlohi[table] = 1u;
                twidth[table] = 2u;
            }
            continue;
        }
        uint32_t sum = 0, bn = 0, bs = 256;
        #pragma unroll
        for (int i = 0; i < 8; i++) {
            uint32_t s = (uint32_t)i * 32u + lane;
            f[i] = 0;
            if (s >= lo && s <= hi) {
                const uint32_t v = scaled_count(n[i], N, rN);
                f[i] = v < 1u ? 1u : v;
            }
            sum += f[i];
            if (n[i] > bn) {
                bn = n[i];
                bs = s;
            }
        }
        sum = warp_sum(sum);
        int R = (int)kM - (int)sum;
        if (R > 0) {
            warp_argmax(bn, bs);
            if ((bs & 31u) == lane) {
#pragma unroll
                for (int i = 0; i < 8; i++)
                    if ((uint32_t)i == (bs >> 5)) f[i] += (uint32_t)R;
            }
        }
        for (int guard = 0; R < 0 && guard < 512; guard++) {
            uint32_t bf = 0, bfs = 256;
            #pragma unroll
            for (int i = 0; i < 8; i++)
                if (f[i] > bf) {
                    bf = f[i];
                    bfs = (uint32_t)i * 32u + lane;
                }
            warp_argmax(bf, bfs);
            int dec = min((int)bf - 1, -R);
            if (dec <= 0) break;
            if ((bfs & 31u) == lane) {
#pragma unroll
                for (int i = 0; i < 8; i++)
                    if ((uint32_t)i == (bfs >> 5)) f[i] -= (uint32_t)dec;
            }
            R += dec;
        }
        #pragma unroll
        for (int i = 0; i < 8; i++) {
            uint32_t s = (uint32_t)i * 32u + lane;
            if (s >= lo && s <= hi) ftab[table * 256u + s] = (uint16_t)(f[i] - 1u);
        }
        if (lane == 0) {
            tlohi[table] = lo | (hi << 8);
            twidth[table] = 2u + 2u * (hi - lo + 1u);
        }
      }
    }
}

// Exclusive scan of n u32 values (optionally padded words -> bytes) into
// out[0..n], out[n] = total; flags RANGE if the total exceeds `cap` or the
// output type.  Two passes over tiles of kScanTile values read row by row
// (coalesced): block sums, then each block scans its tile from the sum of
// the tiles before it.
template <bool kWordsToBytes>
__device__ __forceinline__ uint64_t scan_value(const uint32_t *in, uint64_t i, uint64_t n) {
    if (i >= n) return 0;
    const uint32_t v = in[i];
    return kWordsToBytes ? round_up((uint64_t)v, 8) * 2u : (uint64_t)v;
}

// Block-wide exclusive scan of one value per thread (kScanThreads threads);
// *total receives the block's sum.  sh: kScanThreads / 32 words of shared memory.
__device__ __forceinline__ uint64_t block_exclusive(uint64_t v, uint64_t *total, uint64_t *sh) {
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    constexpr uint32_t kWarps = kScanThreads / 32;
    uint64_t x = v;
    for (uint32_t o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint64_t w = lane < kWarps ? sh[lane] : 0;
        for (uint32_t o = 1; o < kWarps; o <<= 1) {
            const uint64_t y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kWarps) sh[lane] = w;
    }
    __syncthreads();
    const uint64_t before = warp ? sh[warp - 1] : 0;
    *total = sh[kWarps - 1];
    __syncthreads();  // sh is reused by the next call
    return before + x - v;
}

template <bool kWordsToBytes>
__global__ void __launch_bounds__(kScanThreads) k_scan_sums(const uint32_t *in, uint64_t n, uint64_t *part) {
    __shared__ uint64_t sh[kScanThreads / 32];
    const uint64_t base = (uint64_t)blockIdx.x * kScanTile;
    uint64_t v = 0;
    for (uint32_t r = 0; r < kScanRows; r++) v += scan_value<kWordsToBytes>(in, base + r * kScanThreads + threadIdx.x, n);
    uint64_t total;
    block_exclusive(v, &total, sh);
    if (threadIdx.x == 0) part[blockIdx.x] = total;
}

template <typename OutT, bool kWordsToBytes>
__global__ void __launch_bounds__(kScanThreads) k_scan(const uint32_t *in, uint64_t n, const uint64_t *part,
                                                       OutT *out, uint64_t cap, uint32_t *status) {
    __shared__ uint64_t sh[kScanThreads / 32];
    uint64_t pre = 0, total;
    for (uint32_t b = threadIdx.x; b < blockIdx.x; b += kScanThreads) pre += part[b];
    block_exclusive(pre, &total, sh);
    uint64_t run = total;  // sum of the tiles before this one
    const uint64_t base = (uint64_t)blockIdx.x * kScanTile;
    for (uint32_t r = 0; r < kScanRows; r++) {
        const uint64_t i = base + r * kScanThreads + threadIdx.x;
        const uint64_t v = scan_value<kWordsToBytes>(in, i, n);
        const uint64_t ex = block_exclusive(v, &total, sh);
        if (i < n) out[i] = (OutT)(run + ex);
        run += total;
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
        out[n] = (OutT)run;
        if (run > cap || run > (uint64_t)(OutT)~(OutT)0) flag(status, CG_ERR_RANGE);
    }
}

static uint32_t scan_blocks(uint64_t n) { return (uint32_t)((n + kScanTile - 1) / kScanTile) + (n == 0); }

template <typename OutT, bool kWordsToBytes>
static void launch_scan(const uint32_t *in, uint64_t n, OutT *out, uint64_t cap, uint32_t *status, uint64_t *part,
                        cudaStream_t s) {
    const uint32_t nb = scan_blocks(n);
    k_scan_sums<kWordsToBytes><<<nb, kScanThreads, 0, s>>>(in, n, part);
    k_scan<OutT, kWordsToBytes><<<nb, kScanThreads, 0, s>>>(in, n, part, out, cap, status);
}

constexpr int kMaxEncWarps = 12;
constexpr uint32_t kEtabWords = 256 * kLanes;                   // one [symbol][lane] table
constexpr uint32_t kEncSmemBytes = 2u * kEtabWords * 4u;         // coder table + reciprocals

struct EncStream {
    uint16_t *region;
    uint32_t top, xs, e_top;
    uint64_t e_base;
    bool esc_bad;
};

// Quantized delta of v against anchor value xa: rint((v - xa) * RN(1/step)),
// the statistics pass's arithmetic.
__device__ __forceinline__ int quantize(float v, float xa, float inv_step) {
    return __float2int_rn(__fmul_rn(__fsub_rn(v, xa), inv_step));
}

// One coder step of the lane's symbol, in reverse order: emit the low half
// of the state if coding the symbol would overflow it (the warp's emitters
// write in lane order), then x = floor(x / f) * 2^16 + x mod f + c.
// etab: [symbol][lane] c | (f - 1) << 16, followed by [symbol][lane] floor((2^32 - 1) / f).
// s: the lane's symbol, q: its quantized delta (read only for an escape).
// kHasEsc = false when no lane of the warp escapes in this step (the caller
// checked).
template <bool kHasEsc>
__device__ __forceinline__ void enc_step(const EncArgs &a, const uint32_t *etab, uint32_t s, int q, uint32_t lane,
                                         uint32_t lt, EncStream &S) {
    const uint32_t eb = kHasEsc ? __ballot_sync(kFull, s == kEsc) : 0u;
    if (eb) {
        const uint32_t ne = __popc(eb);
        if (ne > S.e_top) {
            S.esc_bad = true;
        } else {
            if (s == kEsc) {
                const uint64_t idx = S.e_base + S.e_top - ne + __popc(eb & lt);
                if (idx < a.escapes_cap) a.escapes[idx] = q;
            }
            S.e_top -= ne;
        }
    }
    // In PTX, so that emission, the state shift and the quotient correction
    // run under predicates instead of selects.  The emitted word is stored
    // from a copy (the ballot's register, free by then): a store from the
    // state register itself made the shift that follows wait until the store
    // had read it.  Entry e = c | (f - 1) << 16
    // and the reciprocal m = floor((2^32 - 1) / f) 32 KB further on.  The
    // state emits its low half when x >= f * 2^16, i.e. x > (e | 0xFFFF)
    // (never for f = 2^16); the emitting lanes write in lane order below the
    // warp's top (branch-free: every lane forms the address).  Then, with
    // x < f * 2^16, x * m / 2^32 lies in (x / f - 1, x / f], so q =
    // umulhi(x, m) is floor(x / f) or one less; r = x - q f is corrected once,
    // and x = q * 2^16 + r + c.
    static_assert(kEtabWords * 4u == 32768u, "reciprocal table offset");
    const uint32_t es = (uint32_t)__cvta_generic_to_shared(etab + s * kLanes + lane);
    asm volatile("{\n\t.reg .pred p, k;\n\t.reg .b32 e, m, t, mb, f, q, r;\n\t.reg .b64 ad;\n\t"
                 "ld.shared.u32 e, [%3];\n\t"
                 "ld.shared.u32 m, [%3+32768];\n\t"
                 "or.b32 t, e, 65535;\n\t"
                 "setp.gt.u32 p, %0, t;\n\t"
                 "vote.sync.ballot.b32 mb, p, 0xffffffff;\n\t"
                 "popc.b32 t, mb;\n\t"
                 "sub.u32 %1, %1, t;\n\t"
                 "and.b32 t, mb, %4;\n\t"
                 "popc.b32 t, t;\n\t"
                 "add.u32 t, %1, t;\n\t"
                 "mad.wide.u32 ad, t, 2, %2;\n\t"
                 "and.b32 mb, %0, 65535;\n\t"               // the stored word in a register of its own,
                 "@p st.global.u16 [ad], mb;\n\t"          // so the shift below need not wait for
                 "@p shr.u32 %0, %0, 16;\n\t"              // the store to read the state
                 "shr.u32 f, e, 16;\n\t"
                 "add.u32 f, f, 1;\n\t"
                 "mul.hi.u32 q, %0, m;\n\t"
                 "mul.lo.u32 t, q, f;\n\t"
                 "sub.u32 r, %0, t;\n\t"
                 "setp.ge.u32 k, r, f;\n\t"
                 "@k add.u32 q, q, 1;\n\t"
                 "@k sub.u32 r, r, f;\n\t"
                 "and.b32 t, e, 65535;\n\t"
                 "add.u32 r, r, t;\n\t"
                 "mad.lo.u32 %0, q, 65536, r;\n\t}"
                 : "+r"(S.xs), "+r"(S.top)
                 : "l"(S.region), "r"(es), "r"(lt)
                 : "memory");
}

// Encode one stream: groups from the span's last to its first, each group's
// deltas in reverse.  The symbols of whole groups (kG deltas + anchor inside
// the span), as the statistics pass stored them, are loaded one group ahead
// of the one being coded.  kC = 1024 fixes the row stride at compile time (0:
// runtime); the group's rows and its anchor are reached by pointers stepped
// back one group at a time.
template <uint32_t kG, uint32_t kC>
__device__ __forceinline__ void encode_span(const EncArgs &a, const uint32_t *etab, const uint16_t *x, uint32_t slice,
                                            uint32_t grp, uint32_t ch, uint32_t span, float sa, float inv_step) {
    const Geom &g = a.g;
    const uint32_t lane = threadIdx.x & 31u, lt = lanemask_lt();
    const uint32_t c = grp * kLanes + lane;
    const uint32_t G = kG ? kG : g.G;
    const uint32_t C = kC ? kC : g.C;
    constexpr uint32_t kV = kG > 1 ? kG - 1u : 1u;
    const uint32_t c0 = ch * g.chunk, len = g.chunk_len(ch);
    const uint32_t p0 = span * g.tps, p1 = min(p0 + g.tps, len);
    const uint64_t k = g.stream_index(ch, slice, span, grp);
    if (g.steps_in(p0, p1) == 0) {
        if (lane == 0) a.words_count[k] = 0;
        return;
    }
    EncStream S;
    S.region = a.scratch + k * a.region_words;
    S.top = (uint32_t)a.region_words;
    S.e_top = a.esc_count[k];
    S.e_base = a.esc_off[k];
    S.esc_bad = false;
    S.xs = kStateLow;

    uint32_t gs = (p1 - 1u) - (p1 - 1u) % G;  // chunk position of the last group's anchor
    // this group's anchor (row gs / G of the chunk's anchor rows of this slice) and first row
    const int8_t *ap = a.anchors + (g.chunk_anchor_row0(ch) + (uint64_t)slice * g.apc(ch) + gs / G) * C + c;
    const uint16_t *xp = x + (uint64_t)(c0 + gs) * C;
    const uint8_t *sp = a.sym + ((uint64_t)slice * g.T + c0 + gs) * C + c;
    uint32_t b0[kV], b1[kV];
    auto load_group = [&](const uint8_t *gp, uint32_t (&buf)[kV]) {
#pragma unroll
        for (uint32_t i = 0; i < kV; i++) buf[i] = gp[(uint64_t)(i + 1u) * C];
    };
    bool cur_full = kG > 1 && gs >= p0 && gs + G <= p1;
    if (cur_full) load_group(sp, b0);
    // A stream without escapes (the statistics pass counted them per stream)
    // codes every whole group straight from its symbols; otherwise one vote
    // per whole group tells whether any of its values escapes.  If none does
    // (nearly always), its steps skip the escape handling; otherwise -- and
    // for groups cut by the span -- the values are reloaded, quantized and
    // coded one by one with it.
    const bool any_esc = S.e_top != 0;
    // One group, coded from `cur` when whole, with the next group's symbols
    // loaded into `nxt`; false once the span's first group is coded.  Two
    // calls per loop trip swap the buffers' roles instead of copying.
    auto group = [&](uint32_t (&cur)[kV], uint32_t (&nxt)[kV]) -> bool {
        const bool has_next = gs > p0;
        const uint32_t gn = has_next ? gs - G : 0u;
        const bool nxt_full = kG > 1 && has_next && gn >= p0;
        if (nxt_full) load_group(sp - (uint64_t)G * C, nxt);
        bool fast = cur_full;
        if (cur_full && any_esc) {
            bool esc = false;
#pragma unroll
            for (uint32_t i = 0; i < kV; i++) esc = esc || cur[i] == kEsc;
            fast = !__any_sync(kFull, esc);
        }
        if (fast) {
#pragma unroll
            for (uint32_t i = kV; i-- > 0;) enc_step<false>(a, etab, cur[i], 0, lane, lt, S);
        } else {
            const float xa = __fmul_rn((float)*ap, sa);
            const uint32_t t_lo = max(gs + 1u, p0), t_hi = min(gs + G, p1);
            if (kG > 1) {  // the group's values loaded together: one memory latency, not one per step
                float v[kV];
#pragma unroll
                for (uint32_t i = 0; i < kV; i++) {
                    const uint32_t t = gs + 1u + i;
                    v[i] = t >= t_lo && t < t_hi ? ld_half(xp + (uint64_t)(i + 1u) * C) : 0.f;
                }
#pragma unroll
                for (uint32_t i = kV; i-- > 0;) {
                    const uint32_t t = gs + 1u + i;
                    if (t >= t_lo && t < t_hi) {
                        const int q = quantize(v[i], xa, inv_step);
                        enc_step<true>(a, etab, symbol_of(q), q, lane, lt, S);
                    }
                }
            } else {
                for (uint32_t t = t_hi; t-- > t_lo;) {
                    const int q = quantize(ld_half(xp + (uint64_t)(t - gs) * C), xa, inv_step);
                    enc_step<true>(a, etab, symbol_of(q), q, lane, lt, S);
                }
            }
        }
        if (!has_next) return false;
        gs = gn;
        xp -= (uint64_t)G * C;
        sp -= (uint64_t)G * C;
        ap -= C;
        cur_full = nxt_full;
        return true;
    };
    while (group(b0, b1) && group(b1, b0)) {
    }
    S.top -= 2u * kLanes;
    S.region[S.top + 2u * lane] = (uint16_t)(S.xs >> 16);
    S.region[S.top + 2u * lane + 1u] = (uint16_t)(S.xs & 0xFFFFu);
    if (lane == 0) {
        a.words_count[k] = (uint32_t)a.region_words - S.top;
        if (S.esc_bad || S.e_top != 0) flag(a.status, CG_ERR_CORRUPT);
    }
}

// One block per (32-channel group, slice); one warp per stream of that
// column (up to kMaxEncWarps, then warps take several).  kG / kC: the
// compile-time group size and row stride of encode_span (0: runtime).
template <uint32_t kG, uint32_t kC>
__global__ void __launch_bounds__(kMaxEncWarps * 32, 3) k_encode(EncArgs a, StepTable st) {
    const Geom &g = a.g;
    const uint32_t grp = blockIdx.x, slice = blockIdx.y;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const uint32_t c = grp * kLanes + lane;
    const uint16_t *x = a.kv + (uint64_t)slice * g.T * g.C + c;
    const float step = st.v[slice >> 1];

    extern __shared__ __align__(16) uint32_t etab[];  // see enc_step
    __shared__ float s_scale[kLanes];

    if (warp == 0) {
        const uint64_t table = (uint64_t)slice * g.C + c;
        const uint32_t lh = a.tlohi[table], lo = lh & 255u, hi = (lh >> 8) & 255u;
        const uint64_t off = a.table_off[table];
        const bool fits = off + a.twidth[table] <= a.tables_cap;
        if (fits) {
            a.tables[off] = (uint8_t)lo;
            a.tables[off + 1] = (uint8_t)hi;
        }
        // the lane's f - 1 row, 8 symbols (16 bytes) per load, the next load
        // issued before the current 8 are used; compact entries are u16 (the
        // tables section is 2-byte aligned and every table offset is even)
        const uint16_t *frow = a.ftab + table * 256u;
        uint32_t cum = 0, s0 = lo & ~7u;
        uint4 w = *reinterpret_cast<const uint4 *>(frow + s0);
        for (; s0 <= hi; s0 += 8u) {
            const uint4 wn = s0 + 8u <= hi ? *reinterpret_cast<const uint4 *>(frow + s0 + 8u) : w;
#pragma unroll
            for (uint32_t i = 0; i < 8; i++) {
                const uint32_t s = s0 + i;
                const uint32_t word = i < 2 ? w.x : i < 4 ? w.y : i < 6 ? w.z : w.w;
                const uint32_t fm1 = (i & 1u) ? word >> 16 : word & 0xFFFFu;
                if (s >= lo && s <= hi) {
                    etab[s * kLanes + lane] = cum | (fm1 << 16);
                    etab[kEtabWords + s * kLanes + lane] = 0xFFFFFFFFu / (fm1 + 1u);
                    if (fits) *reinterpret_cast<uint16_t *>(a.tables + off + 2u + 2u * (s - lo)) = (uint16_t)fm1;
                    cum += fm1 + 1u;
                }
            }
            w = wn;
        }
        s_scale[lane] = a.scales[(uint64_t)slice * g.C + c];
    }
    __syncthreads();
    const float sa = s_scale[lane];
    const float inv_step = __fdiv_rn(1.f, step);  // the quantizer multiplies by this rounded inverse

    for (uint64_t sp = warp; sp < g.spans_total; sp += nwarps) {
        const uint32_t ch = (uint32_t)(sp / g.spans_full), span = (uint32_t)(sp - (uint64_t)ch * g.spans_full);
        encode_span<kG, kC>(a, etab, x, slice, grp, ch, span, sa, inv_step);
    }
}

// Copy of one stream's words, which end at the end of its 16-byte aligned
// scratch region and so start m words (m = 2 K or 2 K + 1) past a 16-byte
// boundary: output piece j (16 bytes) takes the aligned source pieces j and
// j + 1 and shifts them down by m words -- K whole 32-bit words picked at
// compile time, then 16 bits by a funnel shift when m is odd.  Piece j + 1
// is read only while it starts inside the stream's words (else zero), so
// nothing past the region is read and the words past the stream, which the
// payload pads with zeros, come out as zeros.
template <uint32_t K>
__device__ __forceinline__ void pack_stream(const uint4 *src, uint4 *dst, uint64_t n16, uint64_t a0, uint64_t wend,
                                            uint32_t m, uint32_t lane) {
    const uint32_t sh = (m & 1u) * 16u;
    for (uint64_t j = lane; j < n16; j += 32) {
        const uint4 x = src[j];
        const uint4 y = m && a0 + 8u * j + 8u < wend ? src[j + 1] : make_uint4(0, 0, 0, 0);
        const uint32_t r[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
        dst[j] = make_uint4(__funnelshift_r(r[K], r[K + 1], sh), __funnelshift_r(r[K + 1], r[K + 2], sh),
                            __funnelshift_r(r[K + 2], r[K + 3], sh), __funnelshift_r(r[K + 3], r[K + 4], sh));
    }
}

__global__ void __launch_bounds__(256) k_pack(EncArgs a) {
    const uint64_t k = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    if (k >= a.g.n_streams) return;
    const uint32_t cnt = a.words_count[k];
    const uint64_t off = a.stream_off[k], end = a.stream_off[k + 1];
    if (end > a.payload_cap) return;  // RANGE already flagged by the scan
    // the stream's words: [w0, wend) of the scratch buffer, wend = the end of
    // its region (a multiple of 8 words); stream offsets and the payload are
    // 16-byte aligned, and the stream takes ceil(cnt / 8) pieces of it
    const uint64_t wend = (k + 1u) * a.region_words, w0 = wend - cnt;
    const uint32_t m = (uint32_t)(w0 & 7u);
    const uint64_t a0 = w0 - m;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.scratch + a0);
    uint4 *dst = reinterpret_cast<uint4 *>(a.payload + off);
    const uint64_t n16 = (end - off) >> 4;
    switch (m >> 1) {
        case 0: pack_stream<0>(src, dst, n16, a0, wend, m, lane); break;
        case 1: pack_stream<1>(src, dst, n16, a0, wend, m, lane); break;
        case 2: pack_stream<2>(src, dst, n16, a0, wend, m, lane); break;
        default: pack_stream<3>(src, dst, n16, a0, wend, m, lane); break;
    }
}

__global__ void k_sizes(EncArgs a, uint64_t fixed_bytes) {
    cg_sizes s;
    s.payload_bytes = a.stream_off[a.g.n_streams];
    s.tables_bytes = a.table_off[a.g.n_tables];
    s.n_escapes = a.esc_off[a.g.n_streams];
    s.total_bytes = s.payload_bytes + s.tables_bytes + 4u * s.n_escapes + fixed_bytes;
    *a.dsizes = s;
}

}  // namespace cg

using namespace cg;

extern "C" cg_status cg_encode_bounds(const cg_config *cfg, cg_bounds *b) {
    Geom g;
    if (!b || !make_geom(cfg, &g)) return CG_ERR_INVALID_ARG;
    b->A = g.A;
    b->n_chunks = g.n_chunks;
    b->spans_total = g.spans_total;
    b->n_streams = g.n_streams;
    b->n_tables = g.n_tables;
    b->anchors_bytes = (uint64_t)g.n_slices * g.A * g.C;
    b->scales_bytes = g.n_tables * 4u;
    b->table_off_bytes = (g.n_tables + 1u) * 4u;
    b->tables_max_bytes = g.n_tables * (2u + 2u * 256u);
    b->stream_off_bytes = (g.n_streams + 1u) * 8u;
    b->esc_off_bytes = (g.n_streams + 1u) * 4u;
    uint64_t words = 0;  // worst-case padded words of one slice-group column
    for (uint32_t ch = 0; ch < g.n_chunks; ch++) {
        uint32_t len = g.chunk_len(ch);
        for (uint32_t p0 = 0; p0 < len; p0 += g.tps) {
            uint32_t p1 = p0 + g.tps < len ? p0 + g.tps : len;
            uint32_t n = g.steps_in(p0, p1);
            if (n) words += round_up((uint64_t)kLanes * (n + 2u), 8);
        }
    }
    b->payload_max_bytes = words * 2u * g.n_slices * g.NG;
    b->escapes_max_count = (uint64_t)g.n_slices * (g.T - g.A) * g.C;
    b->workspace_bytes = ws_layout(g).total;
    if (b->tables_max_bytes > 0xFFFFFFFFull) return CG_ERR_RANGE;
    return CG_OK;
}

static bool outputs_ok(const cg_encoded *out) {
    return out && out->anchors && out->scales && out->tables && out->table_off && out->stream_off && out->esc_off &&
           (out->payload || !out->payload_cap) && (out->escapes || !out->escapes_cap) && sections_aligned(*out);
}

template <uint32_t NL>
static cudaError_t launch_stats(dim3 grid, cudaStream_t s, const EncArgs &a, const StepTable &st, const StatsLevels &lv) {
    constexpr int bytes = (int)stats_smem_bytes<NL>();
    // the raw counts (grouping ablation) only come with one level
    auto k = NL > 1                ? (a.g.C == 1024 ? k_stats<NL, 1024, false> : k_stats<NL, 0, false>)
             : lv.raw_delta        ? (a.g.C == 1024 ? k_stats<1, 1024, true> : k_stats<1, 0, true>)
             : a.g.C == 1024       ? k_stats<1, 1024, false>
             : a.g.C == 4096       ? k_stats<1, 4096, false>
                                   : k_stats<1, 0, false>;
    // per device, so set before every launch (a host-side call)
    const cudaError_t attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (attr != cudaSuccess) return attr;
    k<<<grid, kStatsWarps * 32, bytes, s>>>(a, st, lv);
    return cudaGetLastError();
}

// Where the kernels of the current device read the cache at kv: memory of
// the current device or managed memory (at kv), or page-locked host memory
// mapped into the device's address space (at its device address, the same
// as kv on a unified-addressing system: the cache is then read straight
// from host memory, over the host link).  Anything else is refused before
// any kernel could touch it.
static cg_status cache_source(const void *kv, int *mem_type, const void **view) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, kv) != cudaSuccess) {
        cudaGetLastError();
        return CG_ERR_CUDA;
    }
    *mem_type = (int)at.type;
    int dev = -1;
    CG_CUDA_TRY(cudaGetDevice(&dev));
    if ((at.type == cudaMemoryTypeDevice && at.device == dev) || at.type == cudaMemoryTypeManaged) {
        *view = kv;
        return CG_OK;
    }
    if (at.type == cudaMemoryTypeHost && at.devicePointer) {
        *view = at.devicePointer;
        return CG_OK;
    }
    return CG_ERR_INVALID_ARG;  // unregistered host memory, another device's memory
}

// Whether the kernels of the current device can use p as it is (a
// workspace or an output section): device or managed memory, or host memory
// mapped at the same address.
static cg_status usable_as_is(const void *p) {
    int mt = 0;
    const void *view = nullptr;
    const cg_status st = cache_source(p, &mt, &view);
    if (st != CG_OK) return st;
    return view == p ? CG_OK : CG_ERR_INVALID_ARG;
}

static cg_status outputs_usable(const cg_encoded &o) {
    const void *ptrs[] = {o.anchors, o.scales, o.tables, o.table_off, o.payload, o.stream_off, o.escapes, o.esc_off};
    for (const void *p : ptrs)
        if (p) {
            const cg_status st = usable_as_is(p);
            if (st != CG_OK) return st;
        }
    return CG_OK;
}

// The encode of `levels` quality levels of one cache: level l uses the
// configured steps times mult[l].  One statistics pass reads the cache for
// every level (anchors, scales and all levels' tables); then each level is
// coded and packed in turn, sharing the scratch region.  Level 0 receives
// the anchors and scales; a later level whose sections are other buffers
// gets a copy.
static cg_status encode_levels(const cg_config *cfg, uint32_t levels, const float *mult, const uint16_t *kv, void *ws,
                               size_t ws_bytes, const cg_encoded *outs, cg_sizes *sizes, uint32_t *dev_status,
                               void *stream) {
    Geom g;
    if (!make_geom(cfg, &g) || levels == 0 || levels > kMaxLevels || !mult) return CG_ERR_INVALID_ARG;
    if (!kv || !ws || !outs || !sizes || reinterpret_cast<uintptr_t>(ws) % 256u || reinterpret_cast<uintptr_t>(kv) % 16u)
        return CG_ERR_INVALID_ARG;
    for (uint32_t l = 0; l < levels; l++) {
        if (!outputs_ok(&outs[l]) || !(mult[l] > 0.f) || !isfinite(mult[l])) return CG_ERR_INVALID_ARG;
        for (uint32_t k = 0; k < g.L; k++) {  // every level's steps must be valid steps
            const float st = cfg->step[k] * mult[l];
            if (!(st > 1.0f / 1024.0f) || !(st < 3e38f)) return CG_ERR_INVALID_ARG;
        }
    }
    cg_bounds bd;
    cg_status bs = cg_encode_bounds(cfg, &bd);
    if (bs != CG_OK) return bs;
    const WsLayout L = ws_layout(g, levels);
    if (ws_bytes < L.total) return CG_ERR_RANGE;
    int mt = 0;
    const void *view = nullptr;
    const cg_status kr = cache_source(kv, &mt, &view);
    if (kr != CG_OK) return kr;
    if (reinterpret_cast<uintptr_t>(view) % 16u) return CG_ERR_INVALID_ARG;
    kv = static_cast<const uint16_t *>(view);
    cg_status us = usable_as_is(ws);  // the workspace and every output section
    for (uint32_t l = 0; l < levels && us == CG_OK; l++) us = outputs_usable(outs[l]);
    if (us != CG_OK) return us;
    uint8_t *w = static_cast<uint8_t *>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    auto args = [&](uint32_t l) {
        const cg_encoded *out = &outs[l];
        EncArgs a;
        a.g = g;
        a.kv = kv;
        a.anchors = out->anchors;
        a.scales = out->scales;
        a.tables = out->tables;
        a.table_off = out->table_off;
        a.payload = out->payload;
        a.stream_off = out->stream_off;
        a.escapes = out->escapes;
        a.esc_off = out->esc_off;
        a.tables_cap = out->tables_cap;
        a.payload_cap = out->payload_cap;
        a.escapes_cap = out->escapes_cap;
        a.ftab = reinterpret_cast<uint16_t *>(w + L.ftab[l]);
        a.tlohi = reinterpret_cast<uint32_t *>(w + L.tlohi[l]);
        a.twidth = reinterpret_cast<uint32_t *>(w + L.twidth[l]);
        a.esc_count = reinterpret_cast<uint32_t *>(w + L.esc_count[l]);
        a.words_count = reinterpret_cast<uint32_t *>(w + L.words_count[l]);
        a.scratch = reinterpret_cast<uint16_t *>(w + L.scratch);
        a.sym = w + L.sym + l * L.sym_stride;
        a.region_words = L.region_words;
        a.dsizes = reinterpret_cast<cg_sizes *>(w + L.dsizes[l]);
        a.status = dev_status;
        return a;
    };
    StatsLevels lv;
    lv.raw_delta = lv.raw_anchor = nullptr;
    lv.sym = w + L.sym;
    lv.sym_stride = L.sym_stride;
    for (uint32_t l = 0; l < kMaxLevels; l++) {
        const EncArgs a = args(l < levels ? l : 0);
        lv.ftab[l] = a.ftab;
        lv.tlohi[l] = a.tlohi;
        lv.twidth[l] = a.twidth;
        lv.esc_count[l] = a.esc_count;
        lv.mult[l] = l < levels ? mult[l] : 1.f;
        if (l < levels) CG_CUDA_TRY(cudaMemsetAsync(a.esc_count, 0, g.n_streams * 4u, s));
    }
    StepTable st;
    for (uint32_t k = 0; k < g.L; k++) st.v[k] = cfg->step[k];
    const dim3 grid(g.NG, g.n_slices);
    const EncArgs a0 = args(0);
    cudaError_t e = levels == 1 ? launch_stats<1>(grid, s, a0, st, lv)
                    : levels == 2 ? launch_stats<2>(grid, s, a0, st, lv)
                    : levels == 3 ? launch_stats<3>(grid, s, a0, st, lv)
                                  : launch_stats<4>(grid, s, a0, st, lv);
    CG_CUDA_TRY(e);
    // compile-time row strides for the two common widths: 8 and 32 heads of 128
    auto k_enc = g.G == 10 && g.C == 1024   ? k_encode<10, 1024>
                 : g.G == 10 && g.C == 4096 ? k_encode<10, 4096>
                 : g.G == 10                ? k_encode<10, 0>
                                            : k_encode<0, 0>;
    CG_CUDA_TRY(cudaFuncSetAttribute(k_enc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kEncSmemBytes));
    const uint32_t enc_warps = (uint32_t)(g.spans_total < (uint64_t)kMaxEncWarps ? g.spans_total : kMaxEncWarps);
    const uint64_t fixed = bd.anchors_bytes + bd.scales_bytes + bd.table_off_bytes + bd.stream_off_bytes +
                           bd.esc_off_bytes;
    for (uint32_t l = 0; l < levels; l++) {
        const EncArgs a = args(l);
        StepTable stl;
        for (uint32_t k = 0; k < g.L; k++) stl.v[k] = cfg->step[k] * mult[l];
        if (l > 0 && a.anchors != a0.anchors)
            CG_CUDA_TRY(cudaMemcpyAsync(a.anchors, a0.anchors, bd.anchors_bytes, cudaMemcpyDeviceToDevice, s));
        if (l > 0 && a.scales != a0.scales)
            CG_CUDA_TRY(cudaMemcpyAsync(a.scales, a0.scales, bd.scales_bytes, cudaMemcpyDeviceToDevice, s));
        uint64_t *part = reinterpret_cast<uint64_t *>(w + L.scan_part);
        launch_scan<uint32_t, false>(a.twidth, g.n_tables, a.table_off, a.tables_cap, a.status, part, s);
        launch_scan<uint32_t, false>(a.esc_count, g.n_streams, a.esc_off, a.escapes_cap, a.status, part, s);
        k_enc<<<grid, enc_warps * 32, kEncSmemBytes, s>>>(a, stl);
        launch_scan<uint64_t, true>(a.words_count, g.n_streams, a.stream_off, a.payload_cap, a.status, part, s);
        const uint64_t pack_blocks = (g.n_streams * 32u + 255u) / 256u;
        k_pack<<<(unsigned)pack_blocks, 256, 0, s>>>(a);
        k_sizes<<<1, 1, 0, s>>>(a, fixed);
        CG_CUDA_TRY(cudaGetLastError());
        CG_CUDA_TRY(cudaMemcpyAsync(&sizes[l], a.dsizes, sizeof(cg_sizes), cudaMemcpyDeviceToHost, s));
    }
    return CG_OK;
}

extern "C" cg_status cg_encode(const cg_config *cfg, const uint16_t *kv, void *ws, size_t ws_bytes,
                               const cg_encoded *out, cg_sizes *sizes, uint32_t *dev_status, void *stream) {
    const float one = 1.f;
    return encode_levels(cfg, 1, &one, kv, ws, ws_bytes, out, sizes, dev_status, stream);
}

extern "C" cg_status cg_encode_levels_ws_bytes(const cg_config *cfg, uint32_t n_levels, size_t *ws_bytes) {
    Geom g;
    if (!make_geom(cfg, &g) || !ws_bytes || n_levels == 0 || n_levels > kMaxLevels) return CG_ERR_INVALID_ARG;
    *ws_bytes = ws_layout(g, n_levels).total;
    return CG_OK;
}

extern "C" cg_status cg_encode_levels(const cg_config *cfg, uint32_t n_levels, const float *mult,
                                      const uint16_t *kv, void *ws, size_t ws_bytes, const cg_encoded *outs,
                                      cg_sizes *sizes, uint32_t *dev_status, void *stream) {
    return encode_levels(cfg, n_levels, mult, kv, ws, ws_bytes, outs, sizes, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Grouping ablation (the per-(layer, channel) statistics of the CacheGen
// pages: "CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §1, and the
// sciencestack page's Figure 5, entropy per grouping strategy).  Ideal coded
// bits, sum over symbols of n_s log2(N / n_s), of the same delta symbols
// with one table per (layer, K/V, channel), one per (layer, K/V), or one for
// the whole cache; and of the int8 anchors kept raw or entropy-coded with
// one table per (layer, K/V, channel).
// ---------------------------------------------------------------------------
namespace cg {

// n log2(N / n) summed over a warp's 8 x 32 bins (counts as doubles).
__device__ __forceinline__ double warp_bits(const double (&n)[8], double N) {
    double b = 0.0;
#pragma unroll
    for (int i = 0; i < 8; i++)
        if (n[i] > 0.0) b += n[i] * (log2(N) - log2(n[i]));
    for (int o = 16; o; o >>= 1) b += __shfl_xor_sync(kFull, b, o);
    return b;
}

__device__ __forceinline__ double warp_total(const double (&n)[8]) {
    double t = 0.0;
#pragma unroll
    for (int i = 0; i < 8; i++) t += n[i];
    for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
    return t;
}

// Warp per table: bits of each [256] histogram into *bits; 32 bits per
// count of symbol 255 into *esc when esc is given.
__global__ void k_bits_tables(const uint32_t *hist, uint64_t n_tables, double *bits, double *esc) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t t = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= n_tables) return;
    double n[8];
#pragma unroll
    for (int i = 0; i < 8; i++) n[i] = hist[t * 256u + (uint32_t)i * 32u + lane];
    const double N = warp_total(n);
    if (N == 0.0) return;
    const double b = warp_bits(n, N);
    if (lane == 0) {
        atomicAdd(bits, b);
        if (esc) atomicAdd(esc, 32.0 * (double)hist[t * 256u + 255u]);
    }
}

// Block per slice: the slice's C histograms merged into one table; the
// merged counts are also added to the whole-cache counts.
__global__ void k_bits_slices(const uint32_t *hist, uint32_t C, double *bits, unsigned long long *global) {
    __shared__ unsigned long long m[256];
    const uint64_t t0 = (uint64_t)blockIdx.x * C;
    for (uint32_t s = threadIdx.x; s < 256u; s += blockDim.x) {
        unsigned long long v = 0;
        for (uint32_t c = 0; c < C; c++) v += hist[(t0 + c) * 256u + s];
        m[s] = v;
        atomicAdd(&global[s], v);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const uint32_t lane = threadIdx.x;
        double n[8];
#pragma unroll
        for (int i = 0; i < 8; i++) n[i] = (double)m[(uint32_t)i * 32u + lane];
        const double N = warp_total(n);
        if (N > 0.0) {
            const double b = warp_bits(n, N);
            if (lane == 0) atomicAdd(bits, b);
        }
    }
}

__global__ void k_bits_global(const unsigned long long *global, cg_ablation_bits *out, double values,
                              double anchors) {
    const uint32_t lane = threadIdx.x;
    double n[8];
#pragma unroll
    for (int i = 0; i < 8; i++) n[i] = (double)global[(uint32_t)i * 32u + lane];
    const double N = warp_total(n);
    const double b = N > 0.0 ? warp_bits(n, N) : 0.0;
    if (lane == 0) {
        out->delta_bits_global = b;
        out->values = values;
        out->anchor_bits_raw = 8.0 * anchors;
    }
}

struct AblationWs {
    uint64_t enc, anchors, scales, raw_delta, raw_anchor, global, total;
};
static AblationWs ablation_ws(const Geom &g) {
    AblationWs w;
    uint64_t o = 0;
    auto take = [&](uint64_t bytes) {
        uint64_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    w.enc = take(ws_layout(g, 1).total);
    w.anchors = take((uint64_t)g.n_slices * g.A * g.C);
    w.scales = take(g.n_tables * 4u);
    w.raw_delta = take(g.n_tables * 256u * 4u);
    w.raw_anchor = take(g.n_tables * 256u * 4u);
    w.global = take(256u * 8u);
    w.total = o;
    return w;
}

}  // namespace cg

extern "C" cg_status cg_cache_source(const void *kv, int *mem_type, const void **device_view) {
    if (!kv || !mem_type || !device_view) return CG_ERR_INVALID_ARG;
    *mem_type = 0;
    *device_view = nullptr;
    return cache_source(kv, mem_type, device_view);
}

extern "C" cg_status cg_ablation_ws_bytes(const cg_config *cfg, size_t *ws_bytes) {
    Geom g;
    if (!make_geom(cfg, &g) || !ws_bytes) return CG_ERR_INVALID_ARG;
    *ws_bytes = ablation_ws(g).total;
    return CG_OK;
}

extern "C" cg_status cg_ablation(const cg_config *cfg, const uint16_t *kv, void *ws, size_t ws_bytes,
                                 cg_ablation_bits *out, uint32_t *dev_status, void *stream) {
    Geom g;
    if (!make_geom(cfg, &g) || !kv || !ws || !out || reinterpret_cast<uintptr_t>(ws) % 256u ||
        reinterpret_cast<uintptr_t>(kv) % 16u)
        return CG_ERR_INVALID_ARG;
    const AblationWs W = ablation_ws(g);
    if (ws_bytes < W.total) return CG_ERR_RANGE;
    int mt = 0;
    const void *view = nullptr;
    const cg_status kr = cache_source(kv, &mt, &view);
    if (kr != CG_OK) return kr;
    if (reinterpret_cast<uintptr_t>(view) % 16u) return CG_ERR_INVALID_ARG;
    kv = static_cast<const uint16_t *>(view);
    cg_status us = usable_as_is(ws);
    if (us == CG_OK) us = usable_as_is(out);
    if (us != CG_OK) return us;
    uint8_t *w = static_cast<uint8_t *>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const WsLayout L = ws_layout(g, 1);
    uint8_t *we = w + W.enc;
    EncArgs a;
    memset(&a, 0, sizeof(a));
    a.g = g;
    a.kv = kv;
    a.anchors = reinterpret_cast<int8_t *>(w + W.anchors);
    a.scales = reinterpret_cast<float *>(w + W.scales);
    a.ftab = reinterpret_cast<uint16_t *>(we + L.ftab[0]);
    a.tlohi = reinterpret_cast<uint32_t *>(we + L.tlohi[0]);
    a.twidth = reinterpret_cast<uint32_t *>(we + L.twidth[0]);
    a.esc_count = reinterpret_cast<uint32_t *>(we + L.esc_count[0]);
    a.status = dev_status;
    StatsLevels lv;
    for (uint32_t l = 0; l < kMaxLevels; l++) {
        lv.ftab[l] = a.ftab;
        lv.tlohi[l] = a.tlohi;
        lv.twidth[l] = a.twidth;
        lv.esc_count[l] = a.esc_count;
        lv.mult[l] = 1.f;
    }
    lv.raw_delta = reinterpret_cast<uint32_t *>(w + W.raw_delta);
    lv.raw_anchor = reinterpret_cast<uint32_t *>(w + W.raw_anchor);
    lv.sym = we + L.sym;  // written, not used
    lv.sym_stride = L.sym_stride;
    auto *glob = reinterpret_cast<unsigned long long *>(w + W.global);
    CG_CUDA_TRY(cudaMemsetAsync(a.esc_count, 0, g.n_streams * 4u, s));
    CG_CUDA_TRY(cudaMemsetAsync(lv.raw_anchor, 0, g.n_tables * 256u * 4u, s));
    CG_CUDA_TRY(cudaMemsetAsync(glob, 0, 256u * 8u, s));
    CG_CUDA_TRY(cudaMemsetAsync(out, 0, sizeof(cg_ablation_bits), s));
    StepTable st;
    for (uint32_t k = 0; k < g.L; k++) st.v[k] = cfg->step[k];
    CG_CUDA_TRY(launch_stats<1>(dim3(g.NG, g.n_slices), s, a, st, lv));
    const unsigned tb = (unsigned)((g.n_tables * 32u + 255u) / 256u);
    k_bits_tables<<<tb, 256, 0, s>>>(lv.raw_delta, g.n_tables, &out->delta_bits_channel, &out->escape_bits);
    k_bits_tables<<<tb, 256, 0, s>>>(lv.raw_anchor, g.n_tables, &out->anchor_bits_channel, nullptr);
    k_bits_slices<<<g.n_slices, 256, 0, s>>>(lv.raw_delta, g.C, &out->delta_bits_slice, glob);
    k_bits_global<<<1, 32, 0, s>>>(glob, out, (double)g.n_slices * g.T * g.C, (double)g.n_slices * g.A * g.C);
    CG_CUDA_TRY(cudaGetLastError());
    return CG_OK;
}
