/*
 * cg.h -- C ABI of the GB300 KV-cache codec (CacheGen-style tensor codec).
 *
 * The codec turns a fp16 KV cache kv[L][2][T][C] (layers x {K,V} x tokens x
 * heads*head_dim) into a compact bitstream and back.  It follows the method
 * the CacheGen pages describe:
 *   - tokens are cut into groups of `group_size` (10); the first token of a
 *     group is the anchor, kept at 8 bits, and the other tokens are coded as
 *     deltas against it ("CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试",
 *     §2.1, compression pipeline stage 1);
 *   - deltas are quantized with a per-layer step, finer for shallow layers
 *     (0.5 / 1.0 / 1.5 for the layer thirds; same page, §1 and §2.1 stage 2);
 *   - the symbols are arithmetic-coded with separate statistics per (layer,
 *     channel) (same page, §1; "CacheGen: KV Cache Compression and Streaming
 *     for Fast Large Language Model Serving", sciencestack page, TL;DR and
 *     Figure 5), here a 32-bit range-ANS coder with 16-bit tables;
 *   - long contexts are cut into ~1.5K-token chunks that decode on their own
 *     and can each be stored at several quality levels (same page, §2.2);
 *   - decoding runs on the GPU and can be pipelined with the transfer of the
 *     compressed chunks (gptget.net page on the same paper, method details).
 *
 * Conventions for every entry point:
 *   - The library allocates no device memory: every buffer is owned by the
 *     caller.  "device" pointers are CUDA device memory of the current
 *     device, "host" pointers are CPU memory.  Host-side state and scratch,
 *     where a call has any, is said at the call: cg_decode_chunks plans its
 *     descriptors in host heap memory that it frees before returning;
 *     cg_decode_chunks_noalloc keeps a fixed device array, a static host
 *     staging buffer and, per device, the array's device address for the
 *     life of the process.  Every other call keeps no state between calls.
 *   - GPU work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: outputs are valid after the stream is
 *     synchronized.
 *   - A status returned by the call itself means nothing was enqueued
 *     (CG_ERR_INVALID_ARG, CG_ERR_RANGE for a buffer found too small on the
 *     host) or a launch failed (CG_ERR_CUDA).
 *   - Data-dependent errors found on the GPU are OR-ed into `*dev_status`
 *     (a device uint32_t the caller clears beforehand) as the bit
 *     (1u << code): CG_ERR_NONFINITE, CG_ERR_RANGE, CG_ERR_CORRUPT,
 *     CG_ERR_TIMEOUT.  Read it after synchronizing; cg_status_from_flags()
 *     turns it into a status.  Outputs are undefined when it is non-zero.
 *     Bits 16..23 say which check failed (diagnostics only): 16 malformed
 *     table, 17 stream/escape offsets out of range, 18 coder end state,
 *     19 stream length, 20 non-zero padding, 21 escape count, 22 a bounded
 *     device wait gave up, 23 a decode block's shared memory was not placed
 *     where the decoder's layout needs it (reported with CG_ERR_CUDA; the
 *     block writes nothing).
 *   - fp16 tensors are passed as their 16-bit patterns (uint16_t).
 *
 * Encoded object (all sections little-endian; per-chunk sections are
 * chunk-major so one chunk is one contiguous range of each):
 *   anchors    int8   [n_chunks][L][2][anchor rows of the chunk][C]
 *   scales     float  [L][2][C]          anchor scale per (layer, K/V, channel)
 *   tables     bytes  per (l, kv, c) in that order: u8 lo, u8 hi, then u16
 *                     (f_s - 1) for s = lo..hi; an empty table is lo=1, hi=0
 *   table_off  u32    [L*2*C + 1]        byte offsets into `tables`
 *   payload    bytes  streams ordered (chunk, l, kv, span, channel group);
 *                     a stream is its u16 words then zero words up to a
 *                     multiple of 8 words (16 bytes)
 *   stream_off u64    [n_streams + 1]    byte offsets into `payload` (x16)
 *   escapes    int32  quantized deltas outside [-127, 127], per stream in
 *                     (step, lane) order
 *   esc_off    u32    [n_streams + 1]    indices into `escapes`
 */
#ifndef CG_H
#define CG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CG_OK = 0,
    CG_ERR_INVALID_ARG = 1, /* bad configuration, pointer or size; nothing enqueued */
    CG_ERR_NONFINITE = 2,   /* the input cache holds NaN or Inf */
    CG_ERR_RANGE = 3,       /* an output or workspace buffer is too small */
    CG_ERR_CORRUPT = 4,     /* an encoded object failed its integrity checks */
    CG_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up */
    CG_ERR_CUDA = 6         /* a CUDA call or kernel launch failed */
} cg_status;

/* Codec configuration.  Checked on the host by every call:
 *   L >= 1, L <= CG_MAX_LAYERS; T >= 1; C >= 32 and C % 32 == 0;
 *   group_size >= 1; chunk_tokens >= 1 (groups restart at every chunk);
 *   tokens_per_stream >= 1 (a stream covers at most this many tokens of one
 *   chunk); step: host array of L floats, each finite and > 2^-10. */
#define CG_MAX_LAYERS 1024u
typedef struct {
    uint32_t L, T, C, group_size, chunk_tokens, tokens_per_stream;
    const float *step; /* host, L entries: quantization step per layer */
} cg_config;

/* Sizes derived from a configuration (cg_encode_bounds). */
typedef struct {
    uint64_t A;                 /* anchor rows per (layer, K/V) */
    uint64_t n_chunks, spans_total, n_streams, n_tables;
    uint64_t anchors_bytes;     /* int8 anchor plane */
    uint64_t scales_bytes;      /* float scales */
    uint64_t table_off_bytes;   /* u32 [n_tables + 1] */
    uint64_t tables_max_bytes;  /* worst-case compact tables */
    uint64_t stream_off_bytes;  /* u64 [n_streams + 1] */
    uint64_t payload_max_bytes; /* worst-case payload */
    uint64_t esc_off_bytes;     /* u32 [n_streams + 1] */
    uint64_t escapes_max_count; /* worst-case escapes (every delta) */
    uint64_t workspace_bytes;   /* device workspace cg_encode needs */
} cg_bounds;

/* An encoded object.  For cg_encode these are device pointers to
 * caller-allocated outputs with the given capacities; for cg_decode they
 * point to a complete object in device memory; for cg_serialize /
 * cg_deserialize they point to host memory.  The encode and decode calls
 * take each section at an address aligned to its element type (2 bytes for
 * tables, whose 16-bit entries sit at even offsets; 16 bytes for the payload)
 * and refuse any other with CG_ERR_INVALID_ARG before anything is enqueued. */
typedef struct {
    int8_t *anchors;
    float *scales;
    uint8_t *tables;
    uint32_t *table_off;
    uint8_t *payload;
    uint64_t *stream_off;
    int32_t *escapes;
    uint32_t *esc_off;
    uint64_t tables_cap;  /* bytes available at `tables` */
    uint64_t payload_cap; /* bytes available at `payload` */
    uint64_t escapes_cap; /* int32 entries available at `escapes` */
} cg_encoded;

/* Actual sizes of an encoded object. */
typedef struct {
    uint64_t payload_bytes, tables_bytes, n_escapes, total_bytes;
} cg_sizes;

/* Text for a status code.  Never NULL.  (Status helper of this library; no
 * passage of the CacheGen pages defines it.) */
const char *cg_status_string(cg_status s);

/* First error code set in a device status word (CG_OK when zero).  (Status
 * helper of this library; no passage defines it.) */
cg_status cg_status_from_flags(uint32_t flags);

/* Fill *b with the sizes of every section and of the encode workspace for
 * `cfg`.  Sizing helper of this library (no passage of the pages defines it;
 * the sections are those of the encoded object above).  Host only; no CUDA
 * call.  CG_ERR_INVALID_ARG on a bad config,
 * CG_ERR_RANGE if an offset section would overflow its integer type. */
cg_status cg_encode_bounds(const cg_config *cfg, cg_bounds *b);

/*
 * Encode kv (fp16 bits, [L][2][T][C] contiguous, 16-byte aligned: it is read
 * in 16-byte pieces) into `out`.  kv is memory of the current device, managed
 * memory, or page-locked host memory mapped into the device's address space
 * (cudaHostAlloc / cudaHostRegister): the kernels then read the cache straight
 * from host memory, at the mapping's device address (cg_cache_source).  Any
 * other pointer (unregistered host memory, another device's memory) is
 * refused with CG_ERR_INVALID_ARG before any work is enqueued.
 * Implements the whole encoder: anchor scale and int8 anchors, delta
 * quantization with the layer's step (escape symbol 255 for |q| > 127),
 * per-(layer, K/V, channel) histograms normalized to 16-bit frequency tables,
 * interleaved range-ANS coding of every stream, and the prefix-sum pack of
 * the streams into one payload (the compression pipeline of
 * "CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §2.1).
 *   ws, ws_bytes: device workspace, at least cg_bounds.workspace_bytes,
 *                 256-byte aligned; contents on entry do not matter.  The
 *                 workspace and every output section must be memory the
 *                 device can use at that address (CG_ERR_INVALID_ARG
 *                 otherwise, checked on the host before any work).
 *   out:          host struct of device pointers; anchors, scales, table_off,
 *                 stream_off and esc_off must hold their full sections,
 *                 tables/payload/escapes at least *_cap bytes/entries.
 *   sizes:        host memory (pinned for a truly asynchronous call) that
 *                 receives the actual sizes once the stream has completed.
 *   dev_status:   device word; NONFINITE on NaN/Inf input, RANGE when a
 *                 capacity in `out` is exceeded.
 */
cg_status cg_encode(const cg_config *cfg, const uint16_t *kv, void *ws, size_t ws_bytes, const cg_encoded *out,
                    cg_sizes *sizes, uint32_t *dev_status, void *stream);

/*
 * Where the encoder's kernels would read a cache at kv (host query, no work
 * enqueued): *mem_type receives the CUDA memory type of kv (0 unregistered
 * host memory, 1 page-locked host memory, 2 device memory, 3 managed) and
 * *device_view the address the kernels read, or NULL.  CG_OK when the
 * current device can read it; CG_ERR_INVALID_ARG for null arguments or memory
 * it cannot read; CG_ERR_CUDA when the query itself fails (no device).
 * (Query helper of this library; no passage of the pages defines it.)
 */
cg_status cg_cache_source(const void *kv, int *mem_type, const void **device_view);

/*
 * Encode one cache at several quality levels in one call (at most 4): level
 * l uses cfg->step[k] * mult[l] for layer k, the way the CacheGen pages keep
 * every chunk at a high, medium and low quality ("CacheGen vs 传统量化KV缓存
 * 压缩技术深度对比与性能测试", §2.2).  One statistics pass reads the cache once
 * for every level: anchors and scales (the same at every level) and each
 * level's tables.  The levels are then coded and packed one after another
 * in one shared scratch region.  outs[l] / sizes[l] are level l's object and
 * sizes, each exactly what cg_encode gives with the level's steps.  outs[l]
 * may share the anchors and scales buffers of outs[0]; otherwise they get a
 * copy.  Every level's steps must be valid steps (> 2^-10, finite).
 *   ws: device, cg_encode_levels_ws_bytes() bytes, 256-byte aligned
 *       (cg_encode_levels_ws_bytes is its sizing helper, host only).
 */
cg_status cg_encode_levels_ws_bytes(const cg_config *cfg, uint32_t n_levels, size_t *ws_bytes);
cg_status cg_encode_levels(const cg_config *cfg, uint32_t n_levels, const float *mult, const uint16_t *kv, void *ws,
                           size_t ws_bytes, const cg_encoded *outs, cg_sizes *sizes, uint32_t *dev_status,
                           void *stream);

/*
 * Decode a whole encoded object (device pointers in *enc) into kv_out
 * (device, fp16 bits, [L][2][T][C]).  One thread block per (layer, K/V,
 * 32-channel group) loads its 32 frequency tables into shared memory; each
 * warp decodes one stream (one lane per channel), dequantizes and adds the
 * anchor in fp32 and stores fp16 (the GPU decoder of the CacheGen pages,
 * gptget.net page, method details).  Reconstruction is
 * fp16_rn(q_a * s) for anchors and fp16_rn(q_a * s + q * step) for deltas,
 * every fp32 operation rounded separately.
 *   dev_status: CORRUPT when a table, offset, escape count, end state or
 *               padding check fails.
 */
cg_status cg_decode(const cg_config *cfg, const cg_encoded *enc, uint16_t *kv_out, uint32_t *dev_status,
                    void *stream);

/*
 * Test hook for the device-side time-out path; no passage of the CacheGen
 * pages defines it.  Every wait of the decoder on a bulk copy is bounded;
 * this call makes such a wait run out on purpose, without a GPU fault or a
 * hang, so that the path can be tested.  It decodes like cg_decode, except
 * that the kernel never requests the bulk copy of ring segment 1 (stream
 * bytes 256..511) of any stream, and each wait gives up after a few short
 * polls instead of about a second.  A warp whose stream is longer than 256
 * bytes therefore sees its wait run out: it ORs CG_ERR_TIMEOUT and
 * diagnostic bit 22 into *dev_status, waits (bounded) for the copies it has
 * issued, and takes no further stream; the kernel then returns.  Nothing is
 * left in flight.  kv_out is undefined afterwards; the object, the
 * destination and the context stay usable (a cg_decode of the same object
 * that follows gives the normal output).  Arguments and host checks as for
 * cg_decode.
 */
cg_status cg_test_decode_timeout(const cg_config *cfg, const cg_encoded *enc, uint16_t *kv_out,
                                 uint32_t *dev_status, void *stream);

/* One chunk to decode: chunk `chunk` of object `enc` (configured by `cfg`)
 * is written to dst, a device fp16 tensor [L][2][dst_tokens][C], at token
 * rows dst_token0 .. dst_token0 + chunk length - 1.  The encoded object's
 * sections may be the full object or just device copies whose per-chunk
 * ranges for this chunk are present (see cg_chunk_ranges). */
typedef struct {
    const cg_config *cfg;
    const cg_encoded *enc;
    uint32_t chunk;
    uint16_t *dst;
    uint32_t dst_tokens;
    uint32_t dst_token0;
} cg_chunk_ref;

/* Workspace bytes cg_decode_chunks needs for these refs.  Sizing helper of
 * this library (no passage defines it).  Host only. */
cg_status cg_decode_chunks_ws_bytes(const cg_chunk_ref *refs, uint32_t n, size_t *ws_bytes);

/*
 * Decode a batch of chunks, possibly from different objects (e.g. the
 * quality level chosen per chunk, "CacheGen vs 传统量化KV缓存压缩技术深度对比
 * 与性能测试", §2.2), in one launch.  Chunks of the same object share the
 * thread blocks that load that object's tables.
 *   ws: device workspace of cg_decode_chunks_ws_bytes bytes, 256-aligned;
 *       it receives the job descriptors (copied from host memory that is
 *       released before the call returns).
 */
cg_status cg_decode_chunks(const cg_chunk_ref *refs, uint32_t n, void *ws, size_t ws_bytes, uint32_t *dev_status,
                           void *stream);

/*
 * Chunked decode for callers that cannot allocate device memory.  The CacheGen
 * pages have no counterpart to this; it exists for users of this library.
 *
 * cg_decode_chunks needs a device workspace for its job descriptors.  Some
 * callers cannot provide one: code that runs where every device byte is
 * owned by someone else (a serving engine's pre-sized KV pool, a plugin that
 * may not call cudaMalloc or a caching allocator), or a hot path that must not
 * pay for allocation.  This entry point takes the same refs but keeps the
 * descriptors in a fixed device array inside libcg, CG_NOALLOC_DESC_BYTES
 * (4 MiB) long, which every GPU that loads the library holds until the
 * process exits.  It calls no cudaMalloc or cudaFree and no allocating
 * routine; the host side plans into static storage as well.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and keeps it for the life of the process.  The
 *     kept address belongs to the device's primary context: after
 *     cudaDeviceReset on that device the library must be loaded again before
 *     this call is used.
 *   - Every call rewrites the array, so calls that overlap on the GPU race:
 *     issue them on one stream, or order them with events.  Calls from
 *     several host threads are serialized by a lock.
 *   - CG_ERR_RANGE if the refs need more descriptor bytes than the array
 *     holds (cg_decode_chunks_ws_bytes reports the need; a few hundred
 *     objects' worth of jobs fit), CG_ERR_INVALID_ARG / CG_ERR_CUDA as for
 *     cg_decode_chunks.  Outputs and dev_status behave as in
 *     cg_decode_chunks.
 */
#define CG_NOALLOC_DESC_BYTES (4u << 20)
cg_status cg_decode_chunks_noalloc(const cg_chunk_ref *refs, uint32_t n, uint32_t *dev_status, void *stream);

/*
 * Paged destination: the fp16 cache as fixed-size token blocks scattered in
 * a pool, as a serving engine keeps it (the decoded cache goes straight into
 * the engine's blocks; "CacheGen: KV Cache Compression and Streaming for
 * Fast Large Language Model Serving", gptget.net page, method details: the
 * decoded KV is handed to the serving LLM).  Element (layer l, K/V kv,
 * token t, channel c) is
 *     pool[l * layer_stride + kv * kv_stride + block_table[t / block_tokens] * block_stride
 *          + (t % block_tokens) * token_stride + c]
 * (strides in fp16 elements; a token's C channels are contiguous).  For the
 * per-layer layout [L][n_pool][2][block_tokens][C], for instance:
 * layer_stride = n_pool * 2 * block_tokens * C, block_stride = 2 * block_tokens
 * * C, kv_stride = block_tokens * C, token_stride = C.
 */
typedef struct {
    uint16_t *pool;              /* device */
    const uint32_t *block_table; /* device [n_blocks]: physical block of logical block i */
    uint32_t n_blocks;           /* logical blocks; n_blocks * block_tokens >= T */
    uint32_t n_pool_blocks;      /* physical blocks in the pool */
    uint32_t block_tokens;       /* a power of two, >= group_size */
    uint64_t layer_stride, kv_stride, block_stride, token_stride;
} cg_paged_kv;

/* cg_decode into a paged destination: the same decode, every token row
 * stored through the block table.  A block-table entry >= n_pool_blocks
 * sets CG_ERR_RANGE in *dev_status and the streams that reach it stop
 * before writing to it.  Host checks (CG_ERR_INVALID_ARG): null pointers,
 * block_tokens not a power of two or below group_size, too few blocks. */
cg_status cg_decode_paged(const cg_config *cfg, const cg_encoded *enc, const cg_paged_kv *dst, uint32_t *dev_status,
                          void *stream);

/* Where chunk `chunk` lives inside the per-chunk sections: byte ranges of
 * payload and anchors, entry range of escapes, and entry ranges of
 * stream_off / esc_off that describe it.  Chunks are the unit that is stored
 * and streamed ("CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §2.2:
 * ~1.5K-token chunks sent one by one); the byte layout is this library's
 * (per-chunk sections chunk-major, see the top of this file).  Host only; `off` arrays are host
 * copies of stream_off (u64) and esc_off (u32) of the object. */
typedef struct {
    uint64_t stream_begin, stream_end;   /* stream indices */
    uint64_t payload_begin, payload_end; /* bytes */
    uint64_t escape_begin, escape_end;   /* entries */
    uint64_t anchor_begin, anchor_end;   /* bytes */
} cg_chunk_range;
cg_status cg_chunk_ranges(const cg_config *cfg, uint32_t chunk, const uint64_t *stream_off, const uint32_t *esc_off,
                          cg_chunk_range *r);

/*
 * Serialized object, the stored form of an encoded context (the pages keep
 * every chunk pre-encoded and stored until it is requested: "CacheGen vs
 * 传统量化KV缓存压缩技术深度对比与性能测试", §2.2; the format itself is this
 * library's).  A header (magic "CGKV", version, L, T, C, group_size,
 * chunk_tokens, tokens_per_stream, the L steps, section sizes) followed by
 * the sections of `obj` (host pointers) in the order listed at the top of
 * this file.  cg_serialize with buf == NULL reports the size in *len.
 */
cg_status cg_serialize(const cg_config *cfg, const cg_encoded *obj, const cg_sizes *sizes, void *buf, size_t *len);

/* Read a serialized header: fills cfg (cfg->step is set to `step`, which
 * must hold CG_MAX_LAYERS floats or at least L) and *sizes. */
cg_status cg_deserialize_header(const void *buf, size_t len, cg_config *cfg, float *step, cg_sizes *sizes);

/* Copy the sections of a serialized object into `obj` (host pointers with
 * capacities at least the sizes from cg_deserialize_header). */
cg_status cg_deserialize(const void *buf, size_t len, const cg_encoded *obj);

/*
 * Grouping ablation: ideal coded bits, the sum over symbols of
 * n_s log2(N / n_s), of the call's delta symbols under three groupings of
 * the statistics -- one table per (layer, K/V, channel) as the codec does,
 * one per (layer, K/V), one for the whole cache -- and of the int8 anchors
 * kept raw (8 bits) or entropy-coded per (layer, K/V, channel).  The
 * CacheGen pages motivate per-(layer, channel) statistics this way
 * ("CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §1; sciencestack page,
 * Figure 5: entropy by grouping strategy).  Escaped values add 32 bits each
 * in every grouping (escape_bits).  Bits per value of a variant =
 * (its delta bits + escape_bits + its anchor bits) / values.
 */
typedef struct {
    double values;              /* L * 2 * T * C */
    double delta_bits_channel;  /* one table per (layer, K/V, channel) */
    double delta_bits_slice;    /* one table per (layer, K/V) */
    double delta_bits_global;   /* one table */
    double escape_bits;         /* 32 per escaped delta */
    double anchor_bits_raw;     /* 8 per anchor */
    double anchor_bits_channel; /* anchors entropy-coded per (layer, K/V, channel) */
} cg_ablation_bits;

/* kv as for cg_encode (16-byte aligned); ws: device, cg_ablation_ws_bytes()
 * bytes (its sizing helper, host only), 256-byte aligned; out: device, valid
 * once the stream has completed; dev_status as for cg_encode. */
cg_status cg_ablation_ws_bytes(const cg_config *cfg, size_t *ws_bytes);
cg_status cg_ablation(const cg_config *cfg, const uint16_t *kv, void *ws, size_t ws_bytes, cg_ablation_bits *out,
                      uint32_t *dev_status, void *stream);

/*
 * Bandwidth-adaptive quality level per chunk (host only).
 * ("CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §2.2: every chunk is
 * stored at several quality levels, and the sender picks a level chunk by
 * chunk from the bandwidth it sees, so that transfer plus decode meets the
 * service-level deadline.)
 *
 * Chunks go out in order over one link and are decoded in order on the GPU;
 * the decode of a chunk overlaps the transfer of the next.  For chunk i the
 * planner predicts the bandwidth as the throughput the link gave chunk i - 1
 * (the trace's first entry for chunk 0).  It takes the highest quality (the
 * lowest level index) whose predicted completion of the whole context --
 * chunk i at that level and every later chunk at the lowest quality, at the
 * predicted bandwidth -- is within slo_s; when no level fits it takes the
 * lowest quality.  The chunk's transfer is then played against the trace
 * (piecewise constant, slot_s seconds per entry, the last entry holding on).
 */
typedef struct {
    uint32_t n_chunks, n_levels; /* levels: 0 = highest quality */
    const uint64_t *bytes;       /* host [n_chunks][n_levels]: bytes sent for chunk c at level q */
    const double *decode_s;      /* host [n_chunks][n_levels]: GPU decode seconds of chunk c at level q */
    const double *bw;            /* host [n_slots]: link bandwidth in bytes per second, > 0 */
    uint32_t n_slots;
    double slot_s;               /* seconds per trace entry, > 0 */
    double slo_s;                /* deadline, seconds from the first byte sent */
} cg_level_plan;

typedef struct {
    double arrive_s; /* last byte of the chunk received */
    double done_s;   /* decode of the chunk finished */
} cg_chunk_time;

/* Fills level[n_chunks] and time[n_chunks] (host, caller-owned) with the plan
 * and its timeline under the trace, and *finish_s with the time the last
 * chunk is decoded.  CG_ERR_INVALID_ARG for null pointers, zero counts, or
 * sizes, times and bandwidths that are negative, non-finite or (bandwidth,
 * slot length) zero. */
cg_status cg_plan_levels(const cg_level_plan *p, uint32_t *level, cg_chunk_time *time, double *finish_s);

#ifdef __cplusplus
}
#endif

#endif /* CG_H */
