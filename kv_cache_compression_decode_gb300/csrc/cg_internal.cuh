// cg_internal.cuh -- geometry, layout and status helpers shared by the
// encoder and decoder kernels of libcg (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/cg.h"

namespace cg {

constexpr uint32_t kLanes = 32;       // channels per stream = lanes per warp
constexpr uint32_t kM = 65536;        // total of a normalized table
constexpr uint32_t kStateLow = 65536; // coder state interval [2^16, 2^32)
constexpr uint32_t kEsc = 255;        // escape symbol
constexpr uint32_t kFull = 0xFFFFFFFFu;

__host__ __device__ inline uint32_t ceil_div(uint32_t a, uint32_t b) { return (a + b - 1u) / b; }
__host__ __device__ inline uint64_t round_up(uint64_t a, uint64_t b) { return (a + b - 1u) / b * b; }

// Chunk / group / span geometry of one configuration.
struct Geom {
    uint32_t L, T, C, G, chunk, tps;
    uint32_t n_chunks, last_len;
    uint32_t apc_full;   // anchor rows in a full chunk
    uint32_t spans_full; // spans in a full chunk
    uint32_t NG;         // 32-channel groups
    uint32_t n_slices;   // L * 2
    uint64_t A;          // anchor rows per slice
    uint64_t spans_total, n_streams, n_tables;

    __host__ __device__ uint32_t chunk_len(uint32_t ch) const { return ch + 1 == n_chunks ? last_len : chunk; }
    __host__ __device__ uint32_t apc(uint32_t ch) const { return ceil_div(chunk_len(ch), G); }
    __host__ __device__ uint32_t spc(uint32_t ch) const { return ceil_div(chunk_len(ch), tps); }
    // First anchor row (over all slices) of chunk ch in the chunk-major plane.
    __host__ __device__ uint64_t chunk_anchor_row0(uint32_t ch) const {
        return (uint64_t)ch * apc_full * n_slices;
    }
    // Element index of (slice, anchor of token t, channel 0) in the plane
    // [chunk][slice][rows of the chunk][C].
    __host__ __device__ uint64_t anchor_index(uint32_t slice, uint32_t t) const {
        uint32_t ch = t / chunk, pos = t - ch * chunk;
        return (chunk_anchor_row0(ch) + (uint64_t)slice * apc(ch) + pos / G) * C;
    }
    // First stream of chunk ch.
    __host__ __device__ uint64_t chunk_stream0(uint32_t ch) const {
        return (uint64_t)ch * spans_full * n_slices * NG;
    }
    // Stream index of (chunk, slice, span in chunk, group).
    __host__ __device__ uint64_t stream_index(uint32_t ch, uint32_t slice, uint32_t span, uint32_t g) const {
        return chunk_stream0(ch) + ((uint64_t)slice * spc(ch) + span) * NG + g;
    }
    // Number of non-anchor tokens ("steps") in chunk-relative [p0, p1).
    __host__ __device__ uint32_t steps_in(uint32_t p0, uint32_t p1) const {
        return (p1 - p0) - (ceil_div(p1, G) - ceil_div(p0, G));
    }
};

inline bool make_geom(const cg_config *cfg, Geom *g) {
    if (!cfg || !cfg->step) return false;
    if (cfg->L == 0 || cfg->L > CG_MAX_LAYERS || cfg->T == 0 || cfg->C == 0 || cfg->C % kLanes) return false;
    if (cfg->group_size == 0 || cfg->chunk_tokens == 0 || cfg->tokens_per_stream == 0) return false;
    for (uint32_t l = 0; l < cfg->L; l++) {
        float s = cfg->step[l];
        if (!(s > 0x1p-10f) || !(s < 3.0e38f)) return false;
    }
    g->L = cfg->L;
    g->T = cfg->T;
    g->C = cfg->C;
    g->G = cfg->group_size;
    g->chunk = cfg->chunk_tokens < cfg->T ? cfg->chunk_tokens : cfg->T;
    g->tps = cfg->tokens_per_stream < g->chunk ? cfg->tokens_per_stream : g->chunk;
    g->n_chunks = ceil_div(g->T, g->chunk);
    g->last_len = g->T - (g->n_chunks - 1) * g->chunk;
    g->apc_full = ceil_div(g->chunk, g->G);
    g->spans_full = ceil_div(g->chunk, g->tps);
    g->NG = g->C / kLanes;
    g->n_slices = g->L * 2;
    g->A = (uint64_t)(g->n_chunks - 1) * g->apc_full + ceil_div(g->last_len, g->G);
    g->spans_total = (uint64_t)(g->n_chunks - 1) * g->spans_full + ceil_div(g->last_len, g->tps);
    g->n_streams = (uint64_t)g->n_slices * g->spans_total * g->NG;
    g->n_tables = (uint64_t)g->n_slices * g->C;
    return true;
}

// Device status word: errors are OR-ed in as (1 << code).
__device__ inline void flag(uint32_t *status, cg_status code) {
    if (status) atomicOr(status, 1u << (uint32_t)code);
}

// Diagnostic bits above the status codes: which check failed.
constexpr uint32_t kWhyTable = 1u << 16;    // a frequency table is malformed
constexpr uint32_t kWhyOffsets = 1u << 17;  // stream / escape offsets out of range
constexpr uint32_t kWhyState = 1u << 18;    // a coder state did not end at 2^16
constexpr uint32_t kWhyLength = 1u << 19;   // words consumed do not match the stream length
constexpr uint32_t kWhyPadding = 1u << 20;  // non-zero padding after the stream
constexpr uint32_t kWhyEscapes = 1u << 21;  // escapes consumed do not match the count
constexpr uint32_t kWhyWait = 1u << 22;     // a bounded wait gave up
constexpr uint32_t kWhyLayout = 1u << 23;   // a decode block's shared memory was not placed as its layout needs

__device__ inline void flag_why(uint32_t *status, cg_status code, uint32_t why) {
    if (status) atomicOr(status, (1u << (uint32_t)code) | why);
}

// Each section of an object at an address aligned to its element type, the
// payload to 16 bytes (the decoder's bulk copies): the kernels read and
// write them by element.
inline bool sections_aligned(const cg_encoded &o) {
    const auto mis = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1u)) != 0; };
    return !(mis(o.scales, 4) || mis(o.tables, 2) || mis(o.table_off, 4) || mis(o.payload, 16) ||
             mis(o.stream_off, 8) || mis(o.escapes, 4) || mis(o.esc_off, 4));
}

__device__ inline uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace cg

#define CG_CUDA_TRY(expr)                               \
    do {                                                \
        cudaError_t _e = (expr);                        \
        if (_e != cudaSuccess) return CG_ERR_CUDA;      \
    } while (0)
