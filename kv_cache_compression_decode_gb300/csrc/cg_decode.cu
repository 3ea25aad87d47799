// cg_decode.cu -- GPU decoder of the KV-cache codec (sm_103a).
//
// One thread block per (object, layer, K/V, 32-channel group).  The block's
// warps turn its 32 compact frequency tables into shared-memory symbol
// tables and a bucket table, both laid out [entry][lane]:
//   tab    [256][32] u32   c_s | (f_s - 1) << 16 (f - 1 keeps f = 65536, a
//                          single-symbol table, within 16 bits)
//   coarse [256][32] u16   bucket b (slots 256 b .. 256 b + 255):
//                          (s0 << 8 | d) - 256 b mod 2^16, s0 the symbol
//                          holding slot 256 b, d = 256 (b + 1) - (end of s0)
//                          when s0 ends inside the bucket, else 0
// Then every warp decodes whole streams (lane = channel): per step the lane
// finds its symbol as byte 1 of coarse + x (x the 32-bit state, whose low 16
// bits are the slot): that sum is (s0 << 8 | d) + (slot & 255) plus a
// multiple of 2^16, and the carry out of its low byte steps past s0 exactly
// when the slot lies beyond s0's end.  The lane then takes one
// more symbol in the rare bucket that holds a second end before the slot, and
// walks on only with three or more (each a few lane-steps in a thousand); it then
// updates its 32-bit range-ANS state, and the warp
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

#include <mutex>
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
// Registers per thread of the decode kernels: 56 x 32 lanes is a whole
// number of 256-register allocation units, so that three blocks of up to 12
// warps fit one SM.
constexpr int kDecRegs = 56;
constexpr uint32_t kSegBytes = 256;                     // one bulk copy
constexpr uint32_t kSegWords = kSegBytes / 2;           // 128 words
constexpr uint32_t kRingSegs = 8;
constexpr uint32_t kRingWords = kSegWords * kRingSegs;  // 1024 words = 2 KB per warp
constexpr uint32_t kAhead = 4;                          // segments requested ahead of the one awaited
constexpr uint32_t kMaxRun = 9;                         // steps between ring checks (<= 288 words)
constexpr uint32_t kSpinLimit = 1u << 14;               // x 64 us suspend hint: ~1 s bound per wait
// Time-out test kernel (cg_test_decode_timeout): the bulk copy of this ring
// segment of every stream is never issued, and a wait gives up after a few
// polls.
constexpr uint32_t kWithheldSeg = 1;
constexpr uint32_t kTestSpinLimit = 16;
// A run of kMaxRun steps reads words [pw, pw + R), R = 32 * kMaxRun.  The
// run waits for segment k only when pw + R > k * W (W = kSegWords), and that
// wait first requests segment k + kAhead into the slot of segment
// k + kAhead - kRingSegs, whose words end at (k + kAhead - kRingSegs + 1) W.
// The reads have passed them if pw >= that end, which pw > k W - R gives
// whenever R <= (kRingSegs - kAhead - 1) W + 1.
static_assert(kLanes * kMaxRun <= (kRingSegs - kAhead - 1) * kSegWords + 1, "ring window");
static_assert((kRingSegs & (kRingSegs - 1u)) == 0, "slot = segment & (kRingSegs - 1)");

// Dynamic shared memory of a decode block of nw warps.  Every warp's ring
// starts on a 2048-byte boundary of the shared window, so that the
// renormalization forms a word's address as ring | offset.  Dynamic shared
// memory begins either on such a boundary or 1024 bytes past one; the
// dequant table (1 KB) goes after the rings in the first case and before
// them in the second, and the rest follows both at fixed offsets from the
// tables base tb = nw * kRingBytes + 1024:
//   rings u16 [nw][1024], dq f32 [256]   or   dq f32 [256], rings u16 [nw][1024]
//   tb + kTabOff     u32 [256][32]: c | (f - 1) << 16
//   tb + kCoarseOff  u16 [256][32]: (s0 << 8 | d) - 256 b (see top)
//   tb + kHiOff      u32 [32]: lo << 16 | hi
//   tb + kScaleOff   f32 [32]
//   tb + kBadOff     int
//   tb + kBarOff     u64 [nw][kRingSegs]
constexpr uint32_t kRingBytes = kRingWords * 2;               // 2048
constexpr uint32_t kDqBytes = 256 * 4;
constexpr uint32_t kTabOff = 0;
constexpr uint32_t kCoarseOff = kTabOff + 256 * kLanes * 4;
constexpr uint32_t kHiOff = kCoarseOff + 256 * kLanes * 2;
constexpr uint32_t kScaleOff = kHiOff + kLanes * 4;
constexpr uint32_t kBadOff = kScaleOff + kLanes * 4;
constexpr uint32_t kBarOff = kBadOff + 16;
static_assert(kRingBytes == 2048u && kDqBytes == 1024u, "ring alignment and the dequant table's kilobyte");
__host__ __device__ constexpr uint32_t dec_smem_bytes(uint32_t nwarps) {
    return nwarps * kRingBytes + kDqBytes + kBarOff + nwarps * kRingSegs * 8;
}

// A block's pieces of that layout.
struct Shm {
    uint8_t *tb;  // tables base
    float *dq;
    uint16_t *ring;  // warp 0's ring; warp w's at ring + w * kRingWords
};

// False (for the whole block) when dynamic shared memory does not start on
// or 1024 bytes past a 2048-byte boundary, which the layout needs.
__device__ __forceinline__ bool shm_layout(uint8_t *smem, uint32_t nw, Shm &S) {
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem);
    const bool odd = (base & 1024u) != 0;
    S.tb = smem + nw * kRingBytes + kDqBytes;
    S.dq = reinterpret_cast<float *>(odd ? smem : smem + nw * kRingBytes);
    S.ring = reinterpret_cast<uint16_t *>(odd ? smem + kDqBytes : smem);
    return (base & 1023u) == 0;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// 1-D bulk copy global -> shared (TMA), completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(65536u)
        : "memory");
    return ok != 0;
}

// Per-warp ring of stream words, refilled 256 bytes at a time by bulk copies.
struct Ring {
    const uint16_t *buf;  // generic pointer to the warp's kRingWords words
    uint32_t buf_s;       // shared address of the ring
    uint32_t bar_s;       // shared address of bar[0] (kRingSegs consecutive u64)
    uint32_t phase;       // bit k: parity of slot k's next completion
};

// Stream-local cursor over the ring.
struct Cursor {
    const uint8_t *src;  // stream start in global memory (16-byte aligned)
    uint32_t nbytes, nw, nseg;
    uint32_t wseg;   // next segment to wait for
    uint32_t avail;  // words [0, avail) are in the ring
    bool alive;
};

// kWithhold selects the time-out test kernel: segment kWithheldSeg is never
// requested, so a wait for it runs out with nothing in flight.
template <bool kWithhold>
__device__ __forceinline__ void ring_issue(Ring &R, const Cursor &K, uint32_t k) {
    const uint32_t off = k * kSegBytes;
    if (k >= K.nseg || (kWithhold && k == kWithheldSeg)) return;
    if ((threadIdx.x & 31u) == 0) {
        const uint32_t slot = k & (kRingSegs - 1u), bytes = min(kSegBytes, K.nbytes - off);
        fence_proxy_async();
        mbar_expect_tx(R.bar_s + 8u * slot, bytes);
        bulk_g2s(R.buf_s + slot * kSegBytes, K.src + off, bytes, R.bar_s + 8u * slot);
    }
}

// Waits (bounded) for segment k; false if the wait gave up.
template <bool kWithhold>
__device__ __forceinline__ bool ring_wait(Ring &R, uint32_t k) {
    const uint32_t slot = k & (kRingSegs - 1u);
    const uint32_t par = (R.phase >> slot) & 1u;
    bool ok = false;
    for (uint32_t it = 0; it < (kWithhold ? kTestSpinLimit : kSpinLimit) && !ok; it++)
        ok = mbar_try_wait(R.bar_s + 8u * slot, par);
    R.phase ^= 1u << slot;
    return __all_sync(kFull, ok);
}

// Make words [0, need) of the stream available.  Segment k + kAhead goes
// into the slot of segment k + kAhead - kRingSegs, which the reads have
// passed (the ring-window assertion above).  Once a wait has given up no
// further segment is requested: the copies already issued are segments
// [wseg, wseg + kAhead), which the end of the span waits for.
template <bool kWithhold>
__device__ __forceinline__ void ensure(Ring &R, Cursor &K, uint32_t need) {
    while (K.alive && K.avail < need && K.wseg < K.nseg) {
        __syncwarp();
        ring_issue<kWithhold>(R, K, K.wseg + kAhead);
        K.alive = ring_wait<kWithhold>(R, K.wseg);
        K.wseg++;
        K.avail = min(K.wseg * kSegWords, K.nw);
    }
}


// The block's tables, built in three phases separated by block barriers.
// Lane = channel of the block's 32-channel group; the compact table of a
// channel holds lo, hi (a byte each) and the 16-bit values f_s - 1 for
// s = lo..hi, 2 + 2 (hi - lo + 1) bytes (2 bytes, lo > hi, when empty).
//  1. Every warp reads the lane's offsets and header; warp w takes the
//     batches j = w, w + nw, ... of 32 entries (entries 32 j .. 32 j + 31)
//     and writes their frequency sum into a scratch row (the bucket table's
//     space, which phase 3 fills).
//  2. Each warp writes its batches' entries c_s | (f_s - 1) << 16, starting
//     from the sum of the batches before them; warp 0 checks that the lane's
//     frequencies add up to 65536 and writes lo / hi, the anchor scale and
//     the block's verdict.
//  3. Every warp fills a share of the bucket table.
// The offsets alone bound every read (entries at even offsets inside the
// section), so a malformed table is flagged, never read out of bounds.
constexpr uint32_t kBatches = 256u / kLanes;

__device__ __forceinline__ bool table_span(const DecObj &o, uint64_t table, uint64_t &at, uint32_t &n) {
    const uint64_t b = o.table_off[table], e = o.table_off[table + 1];
    const bool ok = e >= b + 2u && e <= o.tables_cap && ((b | e) & 1u) == 0 && e - b <= 2u + 2u * 256u;
    at = b;
    n = ok ? (uint32_t)((e - b - 2u) >> 1) : 0u;
    return ok;
}

__device__ __forceinline__ bool prepare_tables(const DecObj &o, uint32_t slice, uint32_t grp, float step,
                                               const Shm &S, uint32_t *status) {
    uint8_t *const smem = S.tb;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const uint64_t table = (uint64_t)slice * o.g.C + grp * kLanes + lane;
    uint32_t *tab = reinterpret_cast<uint32_t *>(smem + kTabOff) + lane;
    uint32_t *part = reinterpret_cast<uint32_t *>(smem + kCoarseOff) + lane;  // [kBatches][32] scratch
    for (uint32_t s = threadIdx.x; s < 256u; s += blockDim.x) S.dq[s] = __fmul_rn(__int2float_rn((int)s - 127), step);

    // phase 1
    uint64_t at;
    uint32_t n;
    bool ok = table_span(o, table, at, n);
    const uint16_t *fm = reinterpret_cast<const uint16_t *>(o.tables + at);  // header, then the entries
    const uint32_t h = ok ? fm[0] : 0u;
    const float sa = warp == 0 ? o.scales[table] : 0.f;
    for (uint32_t j = warp; j < kBatches; j += nw) {
        uint32_t sum = 0;
#pragma unroll
        for (uint32_t h0 = 0; h0 < kLanes; h0 += kLanes / 2) {
            uint32_t v[kLanes / 2];
#pragma unroll
            for (uint32_t t = 0; t < kLanes / 2; t++) {
                const uint32_t i = j * kLanes + h0 + t;
                v[t] = i < n ? fm[1u + i] + 1u : 0u;
            }
#pragma unroll
            for (uint32_t t = 0; t < kLanes / 2; t++) sum += v[t];
        }
        part[j * kLanes] = sum;
    }
    uint32_t lo = h & 255u, hi = h >> 8;
    ok = ok && (lo <= hi ? n == hi - lo + 1u : n == 0u);
    __syncthreads();

    // phase 2
    for (uint32_t j = warp; j < kBatches && ok && j * kLanes < n; j += nw) {
        uint32_t cum = 0;
        for (uint32_t i = 0; i < j; i++) cum += part[i * kLanes];
#pragma unroll
        for (uint32_t h0 = 0; h0 < kLanes; h0 += kLanes / 2) {
            uint32_t v[kLanes / 2];
#pragma unroll
            for (uint32_t t = 0; t < kLanes / 2; t++) {
                const uint32_t i = j * kLanes + h0 + t;
                v[t] = i < n ? fm[1u + i] : 0u;
            }
#pragma unroll
            for (uint32_t t = 0; t < kLanes / 2; t++) {
                const uint32_t i = j * kLanes + h0 + t;
                if (i < n) tab[(lo + i) * kLanes] = (cum & 0xFFFFu) | (v[t] << 16);
                cum += v[t] + 1u;
            }
        }
    }
    if (warp == 0) {
        uint32_t total = 0;
#pragma unroll
        for (uint32_t i = 0; i < kBatches; i++) total += part[i * kLanes];
        ok = ok && (lo > hi || total == kM);
        if (!ok || lo > hi) {
            // empty (no delta token in this call) or invalid: any slot resolves to
            // symbol 0 with f = 65536, and the block is skipped if invalid
            tab[0] = 0xFFFF0000u;
            lo = hi = 0;
        }
        reinterpret_cast<uint32_t *>(smem + kHiOff)[lane] = lo << 16 | hi;
        reinterpret_cast<float *>(smem + kScaleOff)[lane] = sa;
        const bool all_ok = __all_sync(kFull, ok);
        if (lane == 0) {
            *reinterpret_cast<int *>(smem + kBadOff) = !all_ok;
            if (!all_ok) flag_why(status, CG_ERR_CORRUPT, kWhyTable);
        }
    }
    __syncthreads();
    if (*reinterpret_cast<const int *>(smem + kBadOff)) return false;

    // phase 3: bucket b (slots 256 b .. 256 b + 255) holds (s0 << 8 | d) -
    // 256 b mod 2^16, s0 the symbol containing slot 256 b -- the largest s in
    // [lo, hi] with c_s <= 256 b, found by a fixed 8-step binary search over
    // the lane's symbol table -- and d = 256 (b + 1) - (end of s0) when s0
    // ends inside the bucket, else 0.  (s0 << 8 | d) + (slot & 255) stays
    // below 2^16: only symbol 255 could carry past it, and it ends at 2^16.
    // Four searches run side by side.
    {
        constexpr uint32_t kU = 4;
        const uint32_t lh = reinterpret_cast<const uint32_t *>(smem + kHiOff)[lane];
        const uint32_t lo3 = lh >> 16, hi3 = lh & 0xFFFFu;
        uint16_t *coarse = reinterpret_cast<uint16_t *>(smem + kCoarseOff) + lane;
        for (uint32_t b0 = warp; b0 < 256u; b0 += kU * nw) {
            uint32_t sym[kU];
#pragma unroll
            for (uint32_t u = 0; u < kU; u++) sym[u] = lo3;  // c_lo = 0 <= any slot
#pragma unroll
            for (uint32_t st = 128u; st; st >>= 1) {
#pragma unroll
                for (uint32_t u = 0; u < kU; u++) {
                    const uint32_t slot = (b0 + u * nw) * 256u;
                    if (sym[u] + st <= hi3 && (tab[(sym[u] + st) * kLanes] & 0xFFFFu) <= slot) sym[u] += st;
                }
            }
#pragma unroll
            for (uint32_t u = 0; u < kU; u++) {
                const uint32_t b = b0 + u * nw;
                if (b < 256u) {
                    const uint32_t e = tab[sym[u] * kLanes];
                    const uint32_t end = (e & 0xFFFFu) + (e >> 16) + 1u, bend = b * 256u + 256u;
                    coarse[b * kLanes] = (uint16_t)((sym[u] << 8 | (end < bend ? bend - end : 0u)) - (b << 8));
                }
            }
        }
    }
    __syncthreads();
    return true;
}

// Lane-private view of the block's tables.
struct Lut {
    const uint32_t *tab;     // this lane's column: tab[s * 32]
    const uint16_t *coarse;  // this lane's column: coarse[b * 32]
    const float *dq;
    uint32_t hi, lane, lt;
    uint32_t tab_s, coarse_s, dq_s;  // the same three as shared-window addresses
};

// Loads from the shared window by 32-bit address.  The tables are written
// before the block's barrier and only read afterwards.
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
    uint32_t v;
    asm("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

// The warp's renormalization of the updated state xn into x: lanes whose
// state fell below 2^16 take the next words of the stream in lane order.
// Written in PTX so that the state takes its word under the predicate
// (x = (x << 16) | w for the lanes that need one) instead of a select; the
// ring load is unconditional.  pb counts the stream bytes taken; the ring
// starts on a 2048-byte boundary, so a word's address is ring | (byte
// offset mod 2048).
static_assert(kStateLow == 65536u && kRingWords == 1024u, "renorm constants");
__device__ __forceinline__ void renorm(uint32_t &x, uint32_t xn, uint32_t &pb, const Lut &T, const uint16_t *ring) {
    const uint32_t rs = (uint32_t)__cvta_generic_to_shared(ring);
    x = xn;
    asm("{\n\t.reg .pred p;\n\t.reg .b32 b, t, i, w;\n\t"
        "setp.lt.u32 p, %0, 65536;\n\t"           // need = x < 2^16
        "vote.sync.ballot.b32 b, p, 0xffffffff;\n\t"
        "and.b32 t, b, %2;\n\t"                     // needing lanes below this one
        "popc.b32 t, t;\n\t"
        "mad.lo.u32 i, t, 2, %1;\n\t"               // the lane's word: stream byte offset
        "and.b32 i, i, 2047;\n\t"
        "or.b32 i, i, %3;\n\t"                      // ... in the ring
        "ld.shared.u16 w, [i];\n\t"
        "@p mad.lo.u32 %0, %0, 65536, w;\n\t"       // (x << 16) | w
        "popc.b32 t, b;\n\t"
        "mad.lo.u32 %1, t, 2, %1;\n\t}"             // bytes taken by the warp
        : "+r"(x), "+r"(pb)
        : "r"(T.lt), "r"(rs)
        : "memory");
}

// State update for the lane's symbol (r = slot - c_s, fm1 = f_s - 1, a
// form that also holds for f = 65536) and renormalization.
__device__ __forceinline__ void update(uint32_t &x, uint32_t &pb, const Lut &T, const uint16_t *ring, uint32_t r,
                                       uint32_t fm1) {
    const uint32_t xh = x >> 16;
    renorm(x, xh * fm1 + xh + r, pb, T, ring);
}

__device__ __forceinline__ uint16_t to_half(float v) { return __half_as_ushort(__float2half_rn(v)); }

// One decode step of the lane's coder: symbol lookup, state update, the
// warp's renormalization (lanes take the next words in lane order) and the
// symbol's dequantized delta.  Symbols past a second end inside their bucket
// and escapes are rare: one vote sends the warp to the path that handles
// both, and that path walks with a uniform loop so the common path carries
// no divergence bookkeeping.
template <bool kHasEsc>
__device__ __forceinline__ float rans_step(uint32_t &x, uint32_t &pb, const Lut &T, const uint16_t *ring, float step,
                                           const int32_t *escapes, uint32_t &ep, uint32_t ee) {
    const uint32_t e0 = T.coarse[((x >> 8) & 0xFFu) * kLanes];
    uint32_t s = __byte_perm(e0 + x, 0, 0x4441);
    uint32_t e = T.tab[s * kLanes];
    uint32_t r = (x - e) & 0xFFFFu;  // slot - c_s: the slot never lies before c_s
    uint32_t fm1 = e >> 16;
    bool wk = r > fm1;
    float dq;
    if (__any_sync(kFull, kHasEsc ? (wk || s == kEsc) : wk)) {
        while (__any_sync(kFull, wk)) {
            if (wk) {
                s++;
                e = T.tab[s * kLanes];
                r = (x - e) & 0xFFFFu;
                fm1 = e >> 16;
                wk = r > fm1 && s < T.hi;
            }
        }
        dq = T.dq[s];
        if (kHasEsc) {
            const uint32_t esb = __ballot_sync(kFull, s == kEsc);
            if (s == kEsc) {
                const uint32_t idx = ep + __popc(esb & T.lt);
                dq = __fmul_rn(__int2float_rn(idx < ee ? escapes[idx] : 0), step);
            }
            ep += __popc(esb);
        }
    } else {
        dq = T.dq[s];
    }
    update(x, pb, T, ring, r, fm1);
    return dq;
}

// Output rows of one (layer, K/V) slice for the lane's channel.  Row k of a
// group is token t + k; seek() places t, advance() moves it on.  C is the
// row length of the [T][C] layout (a compile-time constant where known).
// [L][2][T][C] layout, shifted by a token offset (chunk destinations).
template <bool kShift>
struct LinearOut {
    uint16_t *base;  // token 0 of the slice
    int64_t shift;   // destination token = object token + shift (kShift only)
    uint32_t c;      // lane's channel
    uint16_t *p;
    __device__ __forceinline__ void seek(uint32_t tok, uint32_t C) {
        p = base + ((int64_t)tok + (kShift ? shift : 0)) * (int64_t)C + c;
    }
    __device__ __forceinline__ uint16_t *row(uint32_t k, uint32_t C) const { return p + (size_t)k * C; }
    __device__ __forceinline__ void advance(uint32_t n, uint32_t C) { p += (size_t)n * C; }
    __device__ __forceinline__ bool ok() const { return true; }
};

// Device view of a cg_paged_kv destination.
struct PagedDst {
    uint16_t *pool;
    const uint32_t *table;
    uint32_t n_blocks, n_pool, bshift;
    uint64_t layer_stride, kv_stride, block_stride, token_stride;
};

// Paged layout: token t lives in block table[t >> bshift], row t & mask.
// A group (at most G <= block_tokens rows) touches at most two blocks, whose
// bases are looked up when the group starts: rows k < kb of the group lie in
// token t's block at r0 + k * stride, the rest in the next block at q1 + k *
// stride (q1 = that block's row 0 less kb rows).  kTsC: the token stride is
// the row length C, a compile-time constant where C is, so a row's offset is
// too.  A physical block outside the pool stops the span (ok() turns false)
// before anything is written there.
template <bool kTsC>
struct PagedOut {
    uint16_t *slice;  // pool + layer and K/V offsets + lane's channel
    const uint32_t *table;
    uint32_t n_blocks, n_pool, bshift;
    uint64_t block_stride, ts;
    uint32_t t, kb;
    uintptr_t r0, q1;
    bool good;
    __device__ __forceinline__ uint16_t *block(uint32_t lb) {
        if (lb >= n_blocks) return slice;  // past the last token: never a row's block
        const uint32_t pb = table[lb];
        if (pb >= n_pool) {
            good = false;
            return slice;
        }
        return slice + (uint64_t)pb * block_stride;
    }
    __device__ __forceinline__ void seek(uint32_t tok, uint32_t C) {
        const uint64_t stride = kTsC ? C : ts;
        const uint32_t lb = tok >> bshift, off = tok & ((1u << bshift) - 1u);
        t = tok;
        kb = (1u << bshift) - off;
        r0 = reinterpret_cast<uintptr_t>(block(lb)) + (uint64_t)off * stride * 2u;
        q1 = reinterpret_cast<uintptr_t>(block(lb + 1u)) - (uint64_t)kb * stride * 2u;
    }
    __device__ __forceinline__ uint16_t *row(uint32_t k, uint32_t C) const {
        const uint64_t stride = kTsC ? C : ts;
        return reinterpret_cast<uint16_t *>((k < kb ? r0 : q1) + (uint64_t)k * stride * 2u);
    }
    __device__ __forceinline__ void advance(uint32_t n, uint32_t C) { seek(t + n, C); }
    __device__ __forceinline__ bool ok() const { return good; }
};

// Decode stream (slice, grp, span sp) of object o into the rows of `O`.
// kG = 10 / kC = 1024 select compile-time group size / row stride (0: runtime).
template <bool kHasEsc, uint32_t kG, uint32_t kC, class Out, bool kW>
__device__ __forceinline__ bool decode_span_impl(const DecObj &o, uint32_t slice, uint32_t grp, uint32_t sp,
                                                 float step, const Shm &S, Ring &R, Out O, uint32_t *status,
                                                 uint64_t sb, uint64_t se, uint32_t eb, uint32_t ee,
                                                 uint32_t nsteps) {
    const Geom &g = o.g;
    const uint32_t G = kG ? kG : g.G;
    const uint32_t C = kC ? kC : g.C;
    Lut T;
    T.lane = threadIdx.x & 31u;
    T.lt = lanemask_lt();
    T.tab = reinterpret_cast<const uint32_t *>(S.tb + kTabOff) + T.lane;
    T.coarse = reinterpret_cast<const uint16_t *>(S.tb + kCoarseOff) + T.lane;
    T.dq = S.dq;
    T.hi = reinterpret_cast<const uint32_t *>(S.tb + kHiOff)[T.lane] & 0xFFFFu;
    T.tab_s = smem_addr(T.tab);
    T.coarse_s = smem_addr(T.coarse);
    T.dq_s = smem_addr(T.dq);
    const uint32_t c = grp * kLanes + T.lane;
    const uint32_t ch = sp / g.spans_full, span = sp - ch * g.spans_full;
    const uint32_t c0 = ch * g.chunk, len = g.chunk_len(ch);
    const uint32_t p0 = span * g.tps, p1 = min(p0 + g.tps, len);
    const float sa = reinterpret_cast<const float *>(S.tb + kScaleOff)[T.lane];
    const uint16_t *ring = R.buf;

    Cursor K;
    K.src = o.payload + sb;
    K.nbytes = (uint32_t)(se - sb);
    K.nw = K.nbytes >> 1;
    K.nseg = (K.nbytes + kSegBytes - 1u) / kSegBytes;
    K.wseg = 0;
    K.avail = 0;
    K.alive = true;
    uint32_t x = 0, pb = 0, ep = eb;  // pb: stream bytes taken (words: pb / 2)
    if (nsteps) {
        for (uint32_t k = 0; k < kAhead; k++) ring_issue<kW>(R, K, k);
        ensure<kW>(R, K, 2u * kLanes);
        x = ((uint32_t)ring[2 * T.lane] << 16) | ring[2 * T.lane + 1];
        pb = 4u * kLanes;
    }

    uint32_t p = p0;
    const int8_t *arow = o.anchors + g.anchor_index(slice, c0 + p0) + c;  // row of p0's group
    O.seek(c0 + p0, C);
    float xa = __fmul_rn((float)*arow, sa);
    const uint32_t gp0 = p0 % G;
    if (gp0) {  // head: the rest of a group whose anchor lies before the span
        const uint32_t cnt = min(G - gp0, p1 - p);
        for (uint32_t k = 0; k < cnt && K.alive && O.ok(); k++) {
            if (k % kMaxRun == 0) ensure<kW>(R, K, (pb >> 1) + kLanes * min(kMaxRun, cnt - k));
            *O.row(k, C) = to_half(__fadd_rn(xa, rans_step<kHasEsc>(x, pb, T, ring, step, o.escapes, ep, ee)));
        }
        p += cnt;
        O.advance(cnt, C);
        arow += C;
    }
    // whole groups: anchor + G - 1 steps with one ring check
    int8_t qa_next = p < p1 ? *arow : 0;
    while (p + G <= p1 && K.alive && O.ok()) {
        xa = __fmul_rn((float)qa_next, sa);
        if (p + G < p1) qa_next = arow[C];  // prefetch the next group's anchor
        *O.row(0, C) = to_half(xa);
        if (kG) ensure<kW>(R, K, (pb >> 1) + kLanes * (kG - 1u));  // kG - 1 <= kMaxRun
        if constexpr (kG == 10) {
            // The nine delta steps written out.  Per step: the bucket lookup,
            // then one vote for the rare cases -- a slot past the end of the
            // bucket's carry symbol (a second end inside its bucket) or an
            // escape.  A lane past a second end takes the next symbol inline;
            // if a lane is still past its symbol's end (three or more ends),
            // or one holds an escape, the step jumps, with nothing changed,
            // to the full steps, which finish the group.  Keeping the walk
            // out of the written-out run leaves it free of loops, and the
            // direct jump keeps the common path to the one vote's branch.
            uint32_t k;
#define CG_STEP(K)                                                                                          \
    {                                                                                                       \
        const uint32_t e0 = lds_u16(T.coarse_s + __byte_perm(x, 0, 0x4441) * (kLanes * 2u));                \
        uint32_t s = __byte_perm(e0 + x, 0, 0x4441);                                                        \
        uint32_t e = lds_u32(T.tab_s + s * (kLanes * 4u));                                                  \
        float dq = lds_f32(T.dq_s + s * 4u);                                                                \
        uint32_t r = (x - e) & 0xFFFFu, fm1 = e >> 16;                                                      \
        if (__any_sync(kFull, kHasEsc ? (r > fm1 || s == kEsc) : r > fm1)) {                                \
            if (r > fm1) {                                                                                  \
                s++;                                                                                        \
                e = lds_u32(T.tab_s + s * (kLanes * 4u));                                                   \
                r = (x - e) & 0xFFFFu;                                                                      \
                fm1 = e >> 16;                                                                              \
            }                                                                                               \
            if (__any_sync(kFull, r > fm1 || s > T.hi || (kHasEsc && s == kEsc))) {                         \
                k = K;                                                                                      \
                goto cg_slow;                                                                               \
            }                                                                                               \
            dq = lds_f32(T.dq_s + s * 4u);                                                                  \
        }                                                                                                   \
        update(x, pb, T, ring, r, fm1);                                                                     \
        *O.row(K, C) = to_half(__fadd_rn(xa, dq));                                                          \
    }
            CG_STEP(1) CG_STEP(2) CG_STEP(3) CG_STEP(4) CG_STEP(5) CG_STEP(6) CG_STEP(7) CG_STEP(8) CG_STEP(9)
#undef CG_STEP
            goto cg_done;
        cg_slow:
#pragma unroll 1
            for (; k < kG; k++)
                *O.row(k, C) = to_half(__fadd_rn(xa, rans_step<kHasEsc>(x, pb, T, ring, step, o.escapes, ep, ee)));
        cg_done:;
        } else {
            for (uint32_t k = 1; k < G; k++) {
                if ((k - 1u) % kMaxRun == 0) ensure<kW>(R, K, (pb >> 1) + kLanes * min(kMaxRun, G - k));
                *O.row(k, C) = to_half(__fadd_rn(xa, rans_step<kHasEsc>(x, pb, T, ring, step, o.escapes, ep, ee)));
            }
        }
        p += G;
        O.advance(G, C);
        arow += C;
    }
    if (p < p1 && K.alive && O.ok()) {  // tail: a group cut by the span end
        xa = __fmul_rn((float)qa_next, sa);
        *O.row(0, C) = to_half(xa);
        const uint32_t cnt = p1 - p - 1u;
        for (uint32_t k = 1; k <= cnt && K.alive; k++) {
            if ((k - 1u) % kMaxRun == 0) ensure<kW>(R, K, (pb >> 1) + kLanes * min(kMaxRun, cnt - k + 1u));
            *O.row(k, C) = to_half(__fadd_rn(xa, rans_step<kHasEsc>(x, pb, T, ring, step, o.escapes, ep, ee)));
        }
    }
    // drain the copies still in flight (also after a wait gave up) before the
    // ring is reused or the block exits
    for (uint32_t k = K.wseg; k < K.nseg && k < K.wseg + kAhead; k++) K.alive = ring_wait<kW>(R, k) && K.alive;
    if (!K.alive) {
        if (T.lane == 0) flag_why(status, CG_ERR_TIMEOUT, kWhyWait);
        return false;
    }
    if (!O.ok()) {  // a destination block outside the pool: the span stopped
        if (T.lane == 0) flag(status, CG_ERR_RANGE);
        return true;
    }
    uint32_t why = ep == ee ? 0u : kWhyEscapes;
    const uint32_t pw = pb >> 1;  // words taken
    if (nsteps) {
        if (!__all_sync(kFull, x == kStateLow)) why |= kWhyState;
        if (!(pw <= K.nw && K.nw - pw < 8u)) why |= kWhyLength;
        const uint16_t *wg = reinterpret_cast<const uint16_t *>(K.src);
        bool zero = true;
        for (uint32_t i = pw + T.lane; i < K.nw && i >= pw; i += 32) zero = zero && wg[i] == 0;
        if (!__all_sync(kFull, zero)) why |= kWhyPadding;
    }
    if (why && T.lane == 0) flag_why(status, CG_ERR_CORRUPT, why);
    return true;
}

// Returns false once a bounded wait of this warp has given up: the warp has
// then waited (again bounded) for the copies it had issued, and it takes no
// further stream.
template <class Out, bool kW = false>
__device__ bool decode_span(const DecObj &o, uint32_t slice, uint32_t grp, uint32_t sp, float step,
                            const Shm &S, Ring &R, Out O, uint32_t *status) {
    const Geom &g = o.g;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t ch = sp / g.spans_full, span = sp - ch * g.spans_full;
    const uint32_t len = g.chunk_len(ch);
    const uint32_t p0 = span * g.tps, p1 = min(p0 + g.tps, len);
    const uint64_t k = g.stream_index(ch, slice, span, grp);
    const uint64_t sb = o.stream_off[k], se = o.stream_off[k + 1];
    const uint32_t eb = o.esc_off[k], ee = o.esc_off[k + 1];
    const uint32_t nsteps = g.steps_in(p0, p1);
    const uint64_t nw = (se - sb) >> 1;
    const bool bad = se < sb || (sb & 15u) || (se & 15u) || se > o.payload_cap || ee < eb || ee > o.escapes_cap ||
                     (nsteps == 0 && nw != 0) || (nsteps != 0 && nw < 2u * kLanes) || nw > 0xFFFFFFFull;
    if (bad) {
        if (lane == 0) flag_why(status, CG_ERR_CORRUPT, kWhyOffsets);
        return true;
    }
#define CG_SPAN(E, GG, CC) \
    decode_span_impl<E, GG, CC, Out, kW>(o, slice, grp, sp, step, S, R, O, status, sb, se, eb, ee, nsteps)
    // compile-time row strides for the two common widths: 8 and 32 heads of 128
    if (g.G == 10 && g.C == 1024) return ee != eb ? CG_SPAN(true, 10, 1024) : CG_SPAN(false, 10, 1024);
    if (g.G == 10 && g.C == 4096) return ee != eb ? CG_SPAN(true, 10, 4096) : CG_SPAN(false, 10, 4096);
    if (g.G == 10) return ee != eb ? CG_SPAN(true, 10, 0) : CG_SPAN(false, 10, 0);
    return ee != eb ? CG_SPAN(true, 0, 0) : CG_SPAN(false, 0, 0);
#undef CG_SPAN
}

__device__ __forceinline__ Ring make_ring(const Shm &S) {
    const uint32_t warp = threadIdx.x >> 5;
    Ring R;
    R.buf = S.ring + warp * kRingWords;
    R.buf_s = smem_addr(R.buf);
    R.bar_s = smem_addr(S.tb + kBarOff) + warp * kRingSegs * 8u;
    R.phase = 0;
    if ((threadIdx.x & 31u) == 0) {
        for (uint32_t k = 0; k < kRingSegs; k++) mbar_init(R.bar_s + 8u * k);
        fence_barrier_init();
        fence_proxy_async();  // the initialized barriers are seen by the bulk-copy unit
    }
    __syncwarp();
    return R;
}

// kPaged: rows go to the blocks of `pd` (kTsC: its token stride is C), else
// to out[L][2][T][C].  kW: the
// time-out test kernel (a withheld ring segment, short waits).
template <bool kPaged, bool kW = false, bool kTsC = false>
__global__ void __maxnreg__(kDecRegs) k_decode_all(DecObj o, StepTable st, uint16_t *out, PagedDst pd,
                                                   uint32_t *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t grp = blockIdx.x, slice = blockIdx.y, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const uint32_t c = grp * kLanes + (threadIdx.x & 31u);
    const float step = st.v[slice >> 1];
    Shm S;
    if (!shm_layout(smem, nw, S)) {
        if (threadIdx.x == 0) flag_why(status, CG_ERR_CUDA, kWhyLayout);
        return;
    }
    Ring R = make_ring(S);
    if (!prepare_tables(o, slice, grp, step, S, status)) return;
    for (uint64_t sp = warp; sp < o.g.spans_total; sp += nw) {
        bool alive;
        if (kPaged) {
            PagedOut<kTsC> O;
            O.slice = pd.pool + (uint64_t)(slice >> 1) * pd.layer_stride + (uint64_t)(slice & 1u) * pd.kv_stride + c;
            O.table = pd.table;
            O.n_blocks = pd.n_blocks;
            O.n_pool = pd.n_pool;
            O.bshift = pd.bshift;
            O.block_stride = pd.block_stride;
            O.ts = pd.token_stride;
            O.good = true;
            alive = decode_span<PagedOut<kTsC>, kW>(o, slice, grp, (uint32_t)sp, step, S, R, O, status);
        } else {
            const LinearOut<false> O{out + (uint64_t)slice * o.g.T * o.g.C, 0, c, nullptr};
            alive = decode_span<LinearOut<false>, kW>(o, slice, grp, (uint32_t)sp, step, S, R, O, status);
        }
        if (!alive) break;
    }
}

__global__ void __maxnreg__(kDecRegs) k_decode_jobs(const DecObj *objs, const DecJob *jobs,
                                                                       const SpanRef *spans, const RefDst *refs,
                                                                       uint32_t *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const DecJob job = jobs[blockIdx.x];
    const DecObj &o = objs[job.obj];
    const uint32_t warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const float step = o.step[job.slice >> 1];
    Shm S;
    if (!shm_layout(smem, nw, S)) {
        if (threadIdx.x == 0) flag_why(status, CG_ERR_CUDA, kWhyLayout);
        return;
    }
    Ring R = make_ring(S);
    if (!prepare_tables(o, job.slice, job.grp, step, S, status)) return;
    for (uint32_t i = warp; i < job.span_count; i += nw) {
        const SpanRef sr = spans[job.span_begin + i];
        const RefDst rd = refs[sr.ref];
        const LinearOut<true> O{rd.dst + (uint64_t)job.slice * rd.dst_tokens * o.g.C, rd.shift,
                                job.grp * kLanes + (threadIdx.x & 31u), nullptr};
        if (!decode_span(o, job.slice, job.grp, sr.span, step, S, R, O, status)) break;
    }
}

// The kernels' dynamic shared memory limit, set on the current device before
// each launch (the attribute is per device; setting it is a host-side call).
static cudaError_t set_smem_attrs() {
    cudaError_t e = cudaFuncSetAttribute(k_decode_all<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)dec_smem_bytes(kMaxDecWarps));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_decode_all<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dec_smem_bytes(kMaxDecWarps));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_decode_all<true, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dec_smem_bytes(kMaxDecWarps));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_decode_jobs, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dec_smem_bytes(kMaxDecWarps));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_decode_all<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dec_smem_bytes(kMaxDecWarps));
    return e;
}

static bool fill_obj(const cg_config *cfg, const cg_encoded *enc, DecObj *o) {
    if (!make_geom(cfg, &o->g) || !enc) return false;
    if (!enc->anchors || !enc->scales || !enc->tables || !enc->table_off || !enc->stream_off || !enc->esc_off)
        return false;
    if ((!enc->payload && enc->payload_cap) || (!enc->escapes && enc->escapes_cap)) return false;
    if (!sections_aligned(*enc)) return false;
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
    CG_CUDA_TRY(set_smem_attrs());
    const uint32_t nwarps = warps_for(o.g.spans_total);
    k_decode_all<false><<<grid, nwarps * 32, dec_smem_bytes(nwarps), static_cast<cudaStream_t>(stream)>>>(
        o, st, kv_out, PagedDst{}, dev_status);
    CG_CUDA_TRY(cudaGetLastError());
    return CG_OK;
}

extern "C" cg_status cg_test_decode_timeout(const cg_config *cfg, const cg_encoded *enc, uint16_t *kv_out,
                                            uint32_t *dev_status, void *stream) {
    DecObj o;
    if (!fill_obj(cfg, enc, &o) || !kv_out) return CG_ERR_INVALID_ARG;
    StepTable st;
    for (uint32_t l = 0; l < o.g.L; l++) st.v[l] = cfg->step[l];
    const dim3 grid(o.g.NG, o.g.n_slices);
    CG_CUDA_TRY(set_smem_attrs());
    const uint32_t nwarps = warps_for(o.g.spans_total);
    k_decode_all<false, true><<<grid, nwarps * 32, dec_smem_bytes(nwarps), static_cast<cudaStream_t>(stream)>>>(
        o, st, kv_out, PagedDst{}, dev_status);
    CG_CUDA_TRY(cudaGetLastError());
    return CG_OK;
}

extern "C" cg_status cg_decode_paged(const cg_config *cfg, const cg_encoded *enc, const cg_paged_kv *dst,
                                     uint32_t *dev_status, void *stream) {
    DecObj o;
    if (!fill_obj(cfg, enc, &o) || !dst || !dst->pool || !dst->block_table) return CG_ERR_INVALID_ARG;
    const uint32_t bt = dst->block_tokens;
    if (bt == 0 || (bt & (bt - 1u)) || bt < o.g.G || dst->n_pool_blocks == 0) return CG_ERR_INVALID_ARG;
    if ((uint64_t)dst->n_blocks * bt < o.g.T) return CG_ERR_INVALID_ARG;
    PagedDst pd;
    pd.pool = dst->pool;
    pd.table = dst->block_table;
    pd.n_blocks = dst->n_blocks;
    pd.n_pool = dst->n_pool_blocks;
    pd.bshift = (uint32_t)__builtin_ctz(bt);
    pd.layer_stride = dst->layer_stride;
    pd.kv_stride = dst->kv_stride;
    pd.block_stride = dst->block_stride;
    pd.token_stride = dst->token_stride;
    StepTable st;
    for (uint32_t l = 0; l < o.g.L; l++) st.v[l] = cfg->step[l];
    const dim3 grid(o.g.NG, o.g.n_slices);
    CG_CUDA_TRY(set_smem_attrs());
    const uint32_t nwarps = warps_for(o.g.spans_total);
    auto k = pd.token_stride == o.g.C ? k_decode_all<true, false, true> : k_decode_all<true>;
    k<<<grid, nwarps * 32, dec_smem_bytes(nwarps), static_cast<cudaStream_t>(stream)>>>(o, st, nullptr, pd,
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
    CG_CUDA_TRY(set_smem_attrs());
    const uint32_t nwarps = warps_for(P.max_spans);
    k_decode_jobs<<<(unsigned)P.jobs.size(), nwarps * 32, dec_smem_bytes(nwarps), s>>>(
        reinterpret_cast<const DecObj *>(w + P.off_objs), reinterpret_cast<const DecJob *>(w + P.off_jobs),
        reinterpret_cast<const SpanRef *>(w + P.off_spans), reinterpret_cast<const RefDst *>(w + P.off_refs),
        dev_status);
    CG_CUDA_TRY(cudaGetLastError());
    return CG_OK;
}

// ---------------------------------------------------------------------------
// Chunk decode that allocates nothing: descriptors live in a file-scope
// device array instead of a caller workspace.
// ---------------------------------------------------------------------------
namespace cg {

// One call's descriptors (objects, destinations, span list, jobs, steps).
static __device__ __align__(256) uint8_t g_noalloc_desc[CG_NOALLOC_DESC_BYTES];
// Host staging for those descriptors (static storage, guarded by the mutex).
static __align__(256) uint8_t h_noalloc_stage[CG_NOALLOC_DESC_BYTES];
static std::mutex g_noalloc_mu;
constexpr int kNoAllocMaxDevices = 64;
static uint8_t *g_noalloc_dev[kNoAllocMaxDevices];  // device address of g_noalloc_desc, per device

// Same descriptor layout as plan_chunks, written straight into `buf`
// (host) for the device address `dev`, with no heap use.  Objects are the
// distinct `enc` pointers in order of first appearance.
struct StaticPlan {
    uint64_t bytes, off_objs, off_refs, off_spans, off_jobs;
    uint32_t n_jobs, max_spans;
};

static cg_status plan_chunks_static(const cg_chunk_ref *refs, uint32_t n, uint8_t *buf, size_t cap, uint8_t *dev,
                                    StaticPlan *P) {
    if (!refs || n == 0) return CG_ERR_INVALID_ARG;
    auto first_of = [&](uint32_t i) {
        uint32_t j = 0;
        while (refs[j].enc != refs[i].enc) j++;
        return j;
    };
    uint64_t n_obj = 0, n_spans = 0, jobs = 0, steps_bytes = 0;
    for (uint32_t i = 0; i < n; i++) {
        const cg_chunk_ref &r = refs[i];
        DecObj o;
        if (!fill_obj(r.cfg, r.enc, &o) || !r.dst) return CG_ERR_INVALID_ARG;
        if (r.chunk >= o.g.n_chunks) return CG_ERR_INVALID_ARG;
        if ((uint64_t)r.dst_token0 + o.g.chunk_len(r.chunk) > r.dst_tokens) return CG_ERR_INVALID_ARG;
        const uint32_t f = first_of(i);
        if (f == i) {
            n_obj++;
            jobs += (uint64_t)o.g.n_slices * o.g.NG;
            steps_bytes = round_up(steps_bytes + 4ull * o.g.L, 256);
        } else {
            DecObj o0;
            fill_obj(refs[f].cfg, refs[f].enc, &o0);
            const Geom &a = o0.g, &b = o.g;
            if (a.L != b.L || a.T != b.T || a.C != b.C || a.G != b.G || a.chunk != b.chunk || a.tps != b.tps)
                return CG_ERR_INVALID_ARG;
        }
        n_spans += o.g.spc(r.chunk);
    }
    uint64_t o = 0;
    auto take = [&](uint64_t nb) {
        uint64_t at = o;
        o = round_up(o + nb, 256);
        return at;
    };
    const uint64_t off_objs = take(n_obj * sizeof(DecObj)), off_refs = take((uint64_t)n * sizeof(RefDst));
    const uint64_t off_spans = take(n_spans * sizeof(SpanRef)), off_jobs = take(jobs * sizeof(DecJob));
    const uint64_t off_steps = o;
    o += steps_bytes;
    if (o > cap || jobs > 0x7FFFFFFFull) return CG_ERR_RANGE;
    DecObj *objs = reinterpret_cast<DecObj *>(buf + off_objs);
    RefDst *rd = reinterpret_cast<RefDst *>(buf + off_refs);
    SpanRef *sp = reinterpret_cast<SpanRef *>(buf + off_spans);
    DecJob *jb = reinterpret_cast<DecJob *>(buf + off_jobs);
    uint64_t so = off_steps, si = 0, ji = 0;
    uint32_t k = 0, mx = 1;
    for (uint32_t i = 0; i < n; i++) {
        const cg_chunk_ref &r = refs[i];
        DecObj ob;
        fill_obj(r.cfg, r.enc, &ob);
        rd[i].dst = r.dst;
        rd[i].dst_tokens = r.dst_tokens;
        rd[i].shift = (int64_t)r.dst_token0 - (int64_t)r.chunk * ob.g.chunk;
        if (first_of(i) != i) continue;
        // object k: its steps, its span list (all refs sharing this enc), its jobs
        ob.step = reinterpret_cast<const float *>(dev + so);
        memcpy(buf + so, r.cfg->step, 4ull * r.cfg->L);
        so = round_up(so + 4ull * r.cfg->L, 256);
        objs[k] = ob;
        const uint32_t sb = (uint32_t)si;
        for (uint32_t m = i; m < n; m++) {
            if (refs[m].enc != r.enc) continue;
            for (uint32_t q = 0; q < ob.g.spc(refs[m].chunk); q++) sp[si++] = SpanRef{refs[m].chunk * ob.g.spans_full + q, m};
        }
        const uint32_t cnt = (uint32_t)si - sb;
        mx = cnt > mx ? cnt : mx;
        for (uint32_t slice = 0; slice < ob.g.n_slices; slice++)
            for (uint32_t grp = 0; grp < ob.g.NG; grp++) jb[ji++] = DecJob{k, slice, grp, sb, cnt};
        k++;
    }
    P->bytes = o;
    P->off_objs = off_objs;
    P->off_refs = off_refs;
    P->off_spans = off_spans;
    P->off_jobs = off_jobs;
    P->n_jobs = (uint32_t)jobs;
    P->max_spans = mx;
    return CG_OK;
}

}  // namespace cg

extern "C" cg_status cg_decode_chunks_noalloc(const cg_chunk_ref *refs, uint32_t n, uint32_t *dev_status,
                                              void *stream) {
    int dev = 0;
    CG_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kNoAllocMaxDevices) return CG_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_dev[dev]) {  // first call on this device: find the array's device address
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_desc) != cudaSuccess || !p) return CG_ERR_CUDA;
        g_noalloc_dev[dev] = static_cast<uint8_t *>(p);
    }
    uint8_t *d = g_noalloc_dev[dev];
    StaticPlan P;
    cg_status st = plan_chunks_static(refs, n, h_noalloc_stage, sizeof(h_noalloc_stage), d, &P);
    if (st != CG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Pageable source: staged before cudaMemcpyAsync returns, so the static
    // host buffer is free again when the lock is released.
    CG_CUDA_TRY(cudaMemcpyAsync(d, h_noalloc_stage, P.bytes, cudaMemcpyHostToDevice, s));
    CG_CUDA_TRY(set_smem_attrs());
    const uint32_t nwarps = warps_for(P.max_spans);
    k_decode_jobs<<<P.n_jobs, nwarps * 32, dec_smem_bytes(nwarps), s>>>(
        reinterpret_cast<const DecObj *>(d + P.off_objs), reinterpret_cast<const DecJob *>(d + P.off_jobs),
        reinterpret_cast<const SpanRef *>(d + P.off_spans), reinterpret_cast<const RefDst *>(d + P.off_refs),
        dev_status);
    CG_CUDA_TRY(cudaGetLastError());
    return CG_OK;
}
