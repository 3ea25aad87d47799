// cg_encode.cu -- GPU encoder of the KV-cache codec (sm_103a).
//
// Pipeline (the CacheGen compression pipeline: anchor/delta, layer-binned
// quantization, arithmetic coding with per-(layer, channel) statistics;
// "CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §1 and §2.1):
//   k_stats   one block per (32-channel group, layer, K/V): anchor absmax ->
//             scale, int8 anchors, delta quantization (multiplication by the
//             once-rounded inverse of the scale / step), shared-memory
//             histograms (lane = channel, bank = lane: conflict-free
//             atomics), escape counts per stream, normalization of the 32
//             histograms to 16-bit frequency tables (warp-cooperative).
//   k_scan    exclusive scans of table sizes, escape counts and stream sizes
//             (block sums, then each block scans its tile).
//   k_encode  one warp per stream (lane = channel): interleaved range ANS
//             over the span's delta tokens in reverse, words written
//             backwards into a per-stream scratch region, escapes placed
//             from the end of the stream's escape range.
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
};

// Prefix scans: kScanThreads threads per block, kScanRows rows each.
constexpr uint32_t kScanThreads = 256, kScanRows = 16, kScanTile = kScanThreads * kScanRows;

// Workspace carving (256-byte aligned pieces): per-level tables and counts,
// one scratch region shared by the levels (they are coded one after another).
struct WsLayout {
    uint64_t ftab[kMaxLevels], tlohi[kMaxLevels], twidth[kMaxLevels], esc_count[kMaxLevels],
        words_count[kMaxLevels], dsizes[kMaxLevels];
    uint64_t scan_part, scratch, total, region_words;
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
    w.total = o;
    return w;
}

__device__ __forceinline__ float ld_half(const uint16_t *p) { return __half2float(__ushort_as_half(*p)); }

__device__ __forceinline__ uint32_t symbol_of(int q) {
    return (uint32_t)(q + 127) <= 254u ? (uint32_t)(q + 127) : kEsc;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// (value, symbol) argmax, smallest symbol on a tie.
__device__ __forceinline__ void warp_argmax(uint32_t &v, uint32_t &s) {
    for (int o = 16; o; o >>= 1) {
        uint32_t ov = __shfl_xor_sync(kFull, v, o), os = __shfl_xor_sync(kFull, s, o);
        if (ov > v || (ov == v && os < s)) {
            v = ov;
            s = os;
        }
    }
}

constexpr int kStatsWarps = 8;

// Token of anchor row r (over all chunks of one slice).
__device__ __forceinline__ uint32_t anchor_token(const Geom &g, uint32_t r) {
    const uint32_t ch = r / g.apc_full;
    return ch * g.chunk + (r - ch * g.apc_full) * g.G;
}

// Quantize one group's anchor and deltas and count the delta symbols.
// v[0] is the anchor token's value, v[1..N-1] the deltas' (already loaded).
// Symbol of delta d at each level: count it in that level's histogram
// (hist + level * 256 * 32) and, for an escape, in the stream's count.
template <uint32_t NL>
__device__ __forceinline__ void count_delta(const EncArgs &a, const StatsLevels &lv, float d, const float (&inv_step)[NL],
                                            uint32_t *hist, uint32_t lane, uint64_t stream) {
#pragma unroll
    for (uint32_t l = 0; l < NL; l++) {
        const int q = __float2int_rn(__fmul_rn(d, inv_step[l]));
        const uint32_t s = symbol_of(q);
        atomicAdd(&hist[l * 256u * kLanes + s * kLanes + lane], 1u);
        if (s == kEsc) atomicAdd(&lv.esc_count[l][stream], 1u);
    }
}

template <uint32_t N, uint32_t NL>
__device__ __forceinline__ void stats_full_group(const EncArgs &a, const StatsLevels &lv, uint32_t slice, uint32_t grp,
                                                 uint32_t ch, uint32_t c0, uint32_t p0, const float (&v)[N], float sa,
                                                 float inv_sa, const float (&inv_step)[NL], uint32_t *hist,
                                                 bool &nonfinite) {
    const Geom &g = a.g;
    const uint32_t lane = threadIdx.x & 31u, c = grp * kLanes + lane;
    nonfinite |= !isfinite(v[0]);
    const float qa = fminf(fmaxf(rintf(__fmul_rn(v[0], inv_sa)), -127.f), 127.f);
    a.anchors[g.anchor_index(slice, c0 + p0) + c] = (int8_t)qa;
    if (lv.raw_anchor) atomicAdd(&lv.raw_anchor[((uint64_t)slice * g.C + c) * 256u + (uint32_t)((int)qa + 127)], 1u);
    const float xa = __fmul_rn(qa, sa);
#pragma unroll
    for (uint32_t i = 1; i < N; i++) {
        nonfinite |= !isfinite(v[i]);
        count_delta<NL>(a, lv, __fsub_rn(v[i], xa), inv_step, hist, lane,
                        g.stream_index(ch, slice, (p0 + i) / g.tps, grp));
    }
}

// Same for a group of any length n (loads inside the loop).
template <uint32_t NL>
__device__ __forceinline__ void stats_any_group(const EncArgs &a, const StatsLevels &lv, uint32_t slice, uint32_t grp,
                                             uint32_t ch, uint32_t c0, uint32_t p0, uint32_t n, const uint16_t *x,
                                             float sa, float inv_sa, const float (&inv_step)[NL], uint32_t *hist,
                                             bool &nonfinite) {
    const Geom &g = a.g;
    const uint32_t lane = threadIdx.x & 31u, c = grp * kLanes + lane;
    const uint16_t *xp = x + (uint64_t)(c0 + p0) * g.C;
    const float v0 = ld_half(xp);
    nonfinite |= !isfinite(v0);
    const float qa = fminf(fmaxf(rintf(__fmul_rn(v0, inv_sa)), -127.f), 127.f);
    a.anchors[g.anchor_index(slice, c0 + p0) + c] = (int8_t)qa;
    if (lv.raw_anchor) atomicAdd(&lv.raw_anchor[((uint64_t)slice * g.C + c) * 256u + (uint32_t)((int)qa + 127)], 1u);
    const float xa = __fmul_rn(qa, sa);
    for (uint32_t i = 1; i < n; i++) {
        const float vi = ld_half(xp + (uint64_t)i * g.C);
        nonfinite |= !isfinite(vi);
        count_delta<NL>(a, lv, __fsub_rn(vi, xa), inv_step, hist, lane,
                        g.stream_index(ch, slice, (p0 + i) / g.tps, grp));
    }
}

// All groups of one slice and channel group, warps strided over groups.
// kG > 0: compile-time group size; two whole groups are loaded before either
// is processed so that 2 kG row loads are in flight per lane.
template <uint32_t kG, uint32_t NL>
__device__ __forceinline__ void stats_groups(const EncArgs &a, const StatsLevels &lv, uint32_t slice, uint32_t grp,
                                             const uint16_t *x, float sa, float inv_sa, const float (&inv_step)[NL],
                                             uint32_t *hist, bool &nonfinite) {
    const Geom &g = a.g;
    const uint32_t warp = threadIdx.x >> 5, A = (uint32_t)g.A;
    for (uint32_t r0 = warp; r0 < A; r0 += 2u * kStatsWarps) {
        uint32_t ch[2], c0[2], p0[2], n[2];
        float v0[kG ? kG : 1], v1[kG ? kG : 1];
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const uint32_t r = r0 + (uint32_t)j * kStatsWarps;
            n[j] = 0;
            ch[j] = c0[j] = p0[j] = 0;
            if (r < A) {
                ch[j] = r / g.apc_full;
                c0[j] = ch[j] * g.chunk;
                p0[j] = (r - ch[j] * g.apc_full) * g.G;
                n[j] = min(g.G, g.chunk_len(ch[j]) - p0[j]);
            }
        }
        if (kG) {
            if (n[0] == kG) {
                const uint16_t *xp = x + (uint64_t)(c0[0] + p0[0]) * g.C;
#pragma unroll
                for (uint32_t i = 0; i < (kG ? kG : 1); i++) v0[i] = ld_half(xp + (uint64_t)i * g.C);
            }
            if (n[1] == kG) {
                const uint16_t *xp = x + (uint64_t)(c0[1] + p0[1]) * g.C;
#pragma unroll
                for (uint32_t i = 0; i < (kG ? kG : 1); i++) v1[i] = ld_half(xp + (uint64_t)i * g.C);
            }
        }
        if (kG && n[0] == kG)
            stats_full_group(a, lv, slice, grp, ch[0], c0[0], p0[0], v0, sa, inv_sa, inv_step, hist, nonfinite);
        else if (n[0])
            stats_any_group(a, lv, slice, grp, ch[0], c0[0], p0[0], n[0], x, sa, inv_sa, inv_step, hist, nonfinite);
        if (kG && n[1] == kG)
            stats_full_group(a, lv, slice, grp, ch[1], c0[1], p0[1], v1, sa, inv_sa, inv_step, hist, nonfinite);
        else if (n[1])
            stats_any_group(a, lv, slice, grp, ch[1], c0[1], p0[1], n[1], x, sa, inv_sa, inv_step, hist, nonfinite);
    }
}

// NL levels in one pass: their histograms side by side in dynamic shared
// memory (NL x 32 KB); anchors and scales are the same for every level.
// (Four blocks per SM for one level: the pass waits on memory, so it wants
// the resident warps; NL > 1 is held to two by its shared memory anyway.)
template <uint32_t NL>
__global__ void __launch_bounds__(kStatsWarps * 32, NL == 1 ? 4 : 2) k_stats(EncArgs a, StepTable st, StatsLevels lv) {
    const Geom &g = a.g;
    const uint32_t grp = blockIdx.x, slice = blockIdx.y;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t c = grp * kLanes + lane;
    const uint16_t *x = a.kv + (uint64_t)slice * g.T * g.C + c;
    const float step = st.v[slice >> 1];

    extern __shared__ __align__(16) uint32_t hist[];  // [level][symbol][lane]
    __shared__ float red[kStatsWarps][kLanes];
    __shared__ float s_scale[kLanes];

    for (uint32_t i = threadIdx.x; i < NL * 256u * kLanes; i += blockDim.x) hist[i] = 0;

    // E1: absmax over this call's anchor rows -> scale = absmax / 127
    // (four independent row loads in flight per lane).
    float amax = 0.f;
    const uint32_t A = (uint32_t)g.A;
    for (uint32_t r0 = warp; r0 < A; r0 += 4u * kStatsWarps) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t r = r0 + (uint32_t)i * kStatsWarps;
            v[i] = 0.f;
            if (r < A) v[i] = ld_half(x + (uint64_t)anchor_token(g, r) * g.C);
        }
#pragma unroll
        for (int i = 0; i < 4; i++) amax = fmaxf(amax, fabsf(v[i]));
    }
    red[warp][lane] = amax;
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

    // E2 + E3 + E4: one warp per group of tokens (anchor + its deltas); the
    // 10-token groups of the CacheGen pipeline load two whole groups at once.
    bool nonfinite = false;
    const float inv_sa = __fdiv_rn(1.f, sa);  // one rounding each
    float inv_step[NL];
#pragma unroll
    for (uint32_t l = 0; l < NL; l++) inv_step[l] = __fdiv_rn(1.f, __fmul_rn(step, lv.mult[l]));
    if (g.G == 10)
        stats_groups<10, NL>(a, lv, slice, grp, x, sa, inv_sa, inv_step, hist, nonfinite);
    else
        stats_groups<0, NL>(a, lv, slice, grp, x, sa, inv_sa, inv_step, hist, nonfinite);
    if (__any_sync(kFull, nonfinite) && lane == 0) flag(a.status, CG_ERR_NONFINITE);
    __syncthreads();
    if (lv.raw_delta)  // level 0's counts, [table][symbol]
        for (uint32_t i = threadIdx.x; i < 256u * kLanes; i += blockDim.x)
            lv.raw_delta[((uint64_t)slice * g.C + grp * kLanes + (i & 31u)) * 256u + (i >> 5)] = hist[i];

    // E5: normalize each channel's counts to a 16-bit table (warp per
    // (level, channel)).
    for (uint32_t jj = warp; jj < NL * kLanes; jj += kStatsWarps) {
        const uint32_t lvl = jj / kLanes, j = jj % kLanes;
        const uint32_t *hl = hist + lvl * 256u * kLanes;
        uint16_t *ftab = lv.ftab[lvl];
        uint32_t *tlohi = lv.tlohi[lvl], *twidth = lv.twidth[lvl];
        const uint64_t table = (uint64_t)slice * g.C + grp * kLanes + j;
        uint32_t n[8], f[8];
        uint32_t N = 0, lo = 256, hi = 0;
        bool any = false;
        #pragma unroll
        for (int i = 0; i < 8; i++) {
            uint32_t s = (uint32_t)i * 32u + lane;
            n[i] = hl[s * kLanes + j];
            N += n[i];
            if (n[i]) {
                lo = min(lo, s);
                hi = max(hi, s);
                any = true;
            }
        }
        N = warp_sum(N);
        for (int o = 16; o; o >>= 1) {
            lo = min(lo, __shfl_xor_sync(kFull, lo, o));
            hi = max(hi, __shfl_xor_sync(kFull, hi, o));
        }
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
                uint64_t v = ((uint64_t)n[i] * kM) / N;
                f[i] = v < 1u ? 1u : (uint32_t)v;
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

// floor(x / f) and x mod f for 1 <= f <= 65536 and x < f * 2^16, with
// m = floor((2^32 - 1) / f) precomputed per symbol: x * m / 2^32 lies in
// (x/f - 1, x/f], so its integer part is the quotient or one less, and one
// correction makes it exact.
__device__ __forceinline__ void udiv_magic(uint32_t x, uint32_t f, uint32_t m, uint32_t &q, uint32_t &r) {
    q = __umulhi(x, m);
    r = x - q * f;
    if (r >= f) {
        q += 1u;
        r -= f;
    }
}

struct EncStream {
    uint16_t *region;
    uint32_t top, xs, e_top;
    uint64_t e_base;
    bool esc_bad;
};

// One coder step of the lane's symbol, in reverse order: emit the low half
// of the state if coding the symbol would overflow it (the warp's emitters
// write in lane order), then x = floor(x / f) * 2^16 + x mod f + c.
// etab: [symbol][lane] c | (f - 1) << 16, followed by [symbol][lane] floor((2^32 - 1) / f).
// q: the lane's quantized delta.  kHasEsc = false when no lane of the warp
// escapes in this step (the caller checked).
__device__ __forceinline__ int quantize(float v, float xa, float inv_step) {
    return __float2int_rn(__fmul_rn(__fsub_rn(v, xa), inv_step));
}

template <bool kHasEsc>
__device__ __forceinline__ void enc_step(const EncArgs &a, const uint32_t *etab, int q, uint32_t lane, uint32_t lt,
                                         EncStream &S) {
    const uint32_t s = symbol_of(q);
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
    const uint32_t e = etab[s * kLanes + lane], m = etab[kEtabWords + s * kLanes + lane];
    const uint32_t f = (e >> 16) + 1u, cs = e & 0xFFFFu;
    const bool emit = (S.xs >> 16) >= f;
    const uint32_t mb = __ballot_sync(kFull, emit);
    const uint32_t nem = __popc(mb);
    // branch-free: every lane forms the address, the emitting lanes store
    uint16_t *dst = S.region + (S.top - nem + __popc(mb & lt));
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p st.global.u16 [%0], %1;\n\t}"
                 ::"l"(dst), "h"((unsigned short)(S.xs & 0xFFFFu)), "r"((uint32_t)emit)
                 : "memory");
    S.xs = emit ? S.xs >> 16 : S.xs;
    S.top -= nem;
    uint32_t qd, rd;
    udiv_magic(S.xs, f, m, qd, rd);
    S.xs = (qd << 16) + rd + cs;
}

// Encode one stream: groups from the span's last to its first, each group's
// deltas in reverse.  Whole groups (kG deltas + anchor inside the span) are
// loaded one group ahead of the one being coded.
template <uint32_t kG>
__device__ __forceinline__ void encode_span(const EncArgs &a, const uint32_t *etab, const uint16_t *x, uint32_t slice,
                                            uint32_t grp, uint32_t ch, uint32_t span, float sa, float inv_step) {
    const Geom &g = a.g;
    const uint32_t lane = threadIdx.x & 31u, lt = lanemask_lt();
    const uint32_t c = grp * kLanes + lane;
    const uint32_t G = kG ? kG : g.G;
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
    float cur[kV], nxt[kV];
    float qa_cur = 0.f, qa_nxt = 0.f;
    auto load_group = [&](uint32_t gpos, float (&buf)[kV], float &qa) {
        const uint16_t *xp = x + (uint64_t)(c0 + gpos + 1u) * g.C;
#pragma unroll
        for (uint32_t i = 0; i < kV; i++) buf[i] = ld_half(xp + (uint64_t)i * g.C);
        qa = (float)a.anchors[g.anchor_index(slice, c0 + gpos) + c];
    };
    bool cur_full = kG > 1 && gs >= p0 && gs + G <= p1;
    if (cur_full) load_group(gs, cur, qa_cur);
    while (true) {
        const bool has_next = gs > p0;
        const uint32_t gn = has_next ? gs - G : 0u;
        const bool nxt_full = kG > 1 && has_next && gn >= p0;
        if (nxt_full) load_group(gn, nxt, qa_nxt);
        // A whole group is quantized first: one vote tells whether any of
        // its values escapes.  If none does (nearly always), its steps skip
        // the escape handling; otherwise -- and for groups cut by the span
        // -- the values are reloaded and coded one by one with it.
        bool fast = false;
        int q[kV];
        if (cur_full) {
            const float xa = __fmul_rn(qa_cur, sa);
            bool esc = false;
#pragma unroll
            for (uint32_t i = 0; i < kV; i++) {
                q[i] = quantize(cur[i], xa, inv_step);
                esc = esc || symbol_of(q[i]) == kEsc;
            }
            fast = !__any_sync(kFull, esc);
        }
        if (fast) {
#pragma unroll
            for (uint32_t i = kV; i-- > 0;) enc_step<false>(a, etab, q[i], lane, lt, S);
        } else {
            const float xa = __fmul_rn((float)a.anchors[g.anchor_index(slice, c0 + gs) + c], sa);
            const uint32_t t_lo = max(gs + 1u, p0), t_hi = min(gs + G, p1);
            for (uint32_t t = t_hi; t-- > t_lo;)
                enc_step<true>(a, etab, quantize(ld_half(x + (uint64_t)(c0 + t) * g.C), xa, inv_step), lane, lt, S);
        }
        if (!has_next) break;
        gs = gn;
        cur_full = nxt_full;
        qa_cur = qa_nxt;
#pragma unroll
        for (uint32_t i = 0; i < kV; i++) cur[i] = nxt[i];
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
// column (up to kMaxEncWarps, then warps take several).
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
        uint32_t cum = 0;
        for (uint32_t s = lo; s <= hi; s++) {
            uint32_t fm1 = a.ftab[table * 256u + s];
            etab[s * kLanes + lane] = cum | (fm1 << 16);
            etab[kEtabWords + s * kLanes + lane] = 0xFFFFFFFFu / (fm1 + 1u);
            if (fits) {
                a.tables[off + 2u + 2u * (s - lo)] = (uint8_t)(fm1 & 255u);
                a.tables[off + 3u + 2u * (s - lo)] = (uint8_t)(fm1 >> 8);
            }
            cum += fm1 + 1u;
        }
        s_scale[lane] = a.scales[(uint64_t)slice * g.C + c];
    }
    __syncthreads();
    const float sa = s_scale[lane];
    const float inv_step = __fdiv_rn(1.f, step);  // the quantizer multiplies by this rounded inverse

    for (uint64_t sp = warp; sp < g.spans_total; sp += nwarps) {
        const uint32_t ch = (uint32_t)(sp / g.spans_full), span = (uint32_t)(sp - (uint64_t)ch * g.spans_full);
        if (g.G == 10)
            encode_span<10>(a, etab, x, slice, grp, ch, span, sa, inv_step);
        else
            encode_span<0>(a, etab, x, slice, grp, ch, span, sa, inv_step);
    }
}

__global__ void __launch_bounds__(256) k_pack(EncArgs a) {
    const uint64_t k = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    if (k >= a.g.n_streams) return;
    const uint32_t cnt = a.words_count[k];
    const uint64_t off = a.stream_off[k], end = a.stream_off[k + 1];
    if (end > a.payload_cap) return;  // RANGE already flagged by the scan
    const uint16_t *src = a.scratch + k * a.region_words + (a.region_words - cnt);
    uint16_t *dst = reinterpret_cast<uint16_t *>(a.payload + off);
    const uint64_t n = (end - off) >> 1;
    for (uint64_t i = lane; i < n; i += 32) dst[i] = i < cnt ? src[i] : (uint16_t)0;
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
           (out->payload || !out->payload_cap) && (out->escapes || !out->escapes_cap) &&
           reinterpret_cast<uintptr_t>(out->payload) % 16u == 0;
}

template <uint32_t NL>
static cudaError_t launch_stats(dim3 grid, cudaStream_t s, const EncArgs &a, const StepTable &st, const StatsLevels &lv) {
    constexpr int bytes = (int)(NL * 256u * kLanes * 4u);
    // per device, so set before every launch (a host-side call)
    const cudaError_t attr = cudaFuncSetAttribute(k_stats<NL>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (attr != cudaSuccess) return attr;
    k_stats<NL><<<grid, kStatsWarps * 32, bytes, s>>>(a, st, lv);
    return cudaGetLastError();
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
    if (!kv || !ws || !outs || !sizes || reinterpret_cast<uintptr_t>(ws) % 256u) return CG_ERR_INVALID_ARG;
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
        a.region_words = L.region_words;
        a.dsizes = reinterpret_cast<cg_sizes *>(w + L.dsizes[l]);
        a.status = dev_status;
        return a;
    };
    StatsLevels lv;
    lv.raw_delta = lv.raw_anchor = nullptr;
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
    CG_CUDA_TRY(cudaFuncSetAttribute(k_encode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kEncSmemBytes));
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
        k_encode<<<grid, enc_warps * 32, kEncSmemBytes, s>>>(a, stl);
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

extern "C" cg_status cg_ablation_ws_bytes(const cg_config *cfg, size_t *ws_bytes) {
    Geom g;
    if (!make_geom(cfg, &g) || !ws_bytes) return CG_ERR_INVALID_ARG;
    *ws_bytes = ablation_ws(g).total;
    return CG_OK;
}

extern "C" cg_status cg_ablation(const cg_config *cfg, const uint16_t *kv, void *ws, size_t ws_bytes,
                                 cg_ablation_bits *out, uint32_t *dev_status, void *stream) {
    Geom g;
    if (!make_geom(cfg, &g) || !kv || !ws || !out || reinterpret_cast<uintptr_t>(ws) % 256u) return CG_ERR_INVALID_ARG;
    const AblationWs W = ablation_ws(g);
    if (ws_bytes < W.total) return CG_ERR_RANGE;
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
