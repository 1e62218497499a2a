// Stable in-place compaction of SoA row arrays by eviction flags, staged
// through shared memory by one CTA (BlockServe page, Algorithm 1 and section
// II-E: finished requests leave the batch, survivors keep their order).
// Used by the single-CTA commit of pack.cu and by the last CTA of the step
// kernel's fused commit.
//
// Rows are compacted in chunks of rows in increasing order: a chunk's
// surviving rows are first staged in shared memory (every array's slice of a
// row, in 16-, 4- or 1-byte elements), then written to their new rows.  A destination is never
// above its source, so it lies in a chunk already staged (this one or an
// earlier one) and nothing is overwritten before it is read.  Survivors
// ahead of the first evicted row keep their index and are not moved.
#pragma once

#include <stdint.h>

#include <algorithm>

#include "common.cuh"

namespace dllm {

constexpr int kCompactMapWords = 2048;   // elements per staged row the element maps cover
constexpr int kCompactBatch = 8;         // global loads (and stores) in flight per thread and element size

// How the rows move: every array's row slice is moved in elements of 16
// bytes (when the slice and its array are 16-byte aligned), 4 bytes, or 1
// byte.  A staged row holds the 16-byte part of every array first, then the
// 4-byte part, then the byte part.
struct CompactPlan {
    int n_arrays, chunk_rows;
    unsigned char* arrays[DLLM_COMPACT_MAX_ARRAYS];
    long long row_bytes[DLLM_COMPACT_MAX_ARRAYS];
    int unit[DLLM_COMPACT_MAX_ARRAYS];          // element size of each array: 16, 4 or 1
    int per_row[3];                             // elements per staged row of each size (16, 4, 1 bytes)
    long long row_total;                        // staged bytes per row
    FastDiv div_row[3];                         // division by per_row[]
    int* new_index;
    int* src_row;
    int* A_out;
};

// Host: fill a plan from dllm_compact_args for `threads` threads and
// `stage_bytes` of staging.  DLLM_OK, DLLM_ERR_INVAL or
// DLLM_ERR_UNSUPPORTED (a row wider than the staging or the element maps).
inline int make_compact_plan(const dllm_compact_args* c, int threads, long long stage_bytes, CompactPlan* P) {
    if (c->n_arrays < 0 || c->n_arrays > DLLM_COMPACT_MAX_ARRAYS || !c->A_out) return DLLM_ERR_INVAL;
    P->n_arrays = c->n_arrays;
    P->per_row[0] = P->per_row[1] = P->per_row[2] = 0;
    for (int k = 0; k < c->n_arrays; ++k) {
        if ((c->A > 0 && !c->arrays[k]) || c->row_bytes[k] <= 0) return DLLM_ERR_INVAL;
        P->arrays[k] = static_cast<unsigned char*>(c->arrays[k]);
        P->row_bytes[k] = c->row_bytes[k];
        const uintptr_t base = reinterpret_cast<uintptr_t>(c->arrays[k]);
        const int u = (c->row_bytes[k] % 16 == 0 && base % 16 == 0) ? 16
                      : (c->row_bytes[k] % 4 == 0 && base % 4 == 0) ? 4 : 1;
        P->unit[k] = u;
        const long long n = c->row_bytes[k] / u;
        if (n > kCompactMapWords) return DLLM_ERR_UNSUPPORTED;
        P->per_row[u == 16 ? 0 : u == 4 ? 1 : 2] += (int)n;
    }
    for (int z = 0; z < 3; ++z)
        if (P->per_row[z] > kCompactMapWords) return DLLM_ERR_UNSUPPORTED;
    P->row_total = 16LL * P->per_row[0] + 4LL * P->per_row[1] + P->per_row[2];
    if (P->row_total > stage_bytes) return DLLM_ERR_UNSUPPORTED;
    P->chunk_rows = P->row_total > 0 ? (int)std::min<long long>(threads, stage_bytes / P->row_total) : threads;
    for (int z = 0; z < 3; ++z) P->div_row[z] = make_fastdiv((uint32_t)std::max(1, P->per_row[z]));
    P->new_index = c->new_index;
    P->src_row = c->src_row;
    P->A_out = c->A_out;
    return DLLM_OK;
}

// Shared-memory scratch of one compaction: per element size, the element
// map of a staged row (array << 24 | byte offset in that array's row), the
// arrays' addresses and row sizes, and per-chunk row indices (NT threads).
template <int NT>
struct CompactScratch {
    int map[3][kCompactMapWords];
    unsigned char* arrays[DLLM_COMPACT_MAX_ARRAYS];
    long long row_bytes[DLLM_COMPACT_MAX_ARRAYS];
    int src[NT], dst[NT];
    int wsum[NT / 32];
    int skip;
};

// The element maps of a staged row, and the arrays' addresses and row sizes.
template <int NT>
__device__ __forceinline__ void compact_map(const CompactPlan& P, CompactScratch<NT>& S, int tid) {
    for (int z = 0; z < 3; ++z) {
        const int u = z == 0 ? 16 : z == 1 ? 4 : 1;
        for (int w = tid; w < P.per_row[z]; w += NT) {
            // the w-th element of size u in a row: arrays in order, each its row_bytes / u elements
            int rem = w, arr = 0;
            for (int a = 0; a < P.n_arrays; ++a) {
                if (P.unit[a] != u) continue;
                const int n = (int)(P.row_bytes[a] / u);
                if (rem < n) {
                    arr = a;
                    break;
                }
                rem -= n;
            }
            S.map[z][w] = (arr << 24) | (rem * u);
        }
    }
    if (tid < P.n_arrays) {
        S.arrays[tid] = P.arrays[tid];
        S.row_bytes[tid] = P.row_bytes[tid];
    }
}

// Element (k, w) of one element size: staged at stage[k * per_row + w].
template <typename E, int NT>
__device__ __forceinline__ void compact_load(const CompactScratch<NT>& S, const int* map, int per_row,
                                             const FastDiv& div, const int* s_src, E* stage, int kept, int tid) {
    const int total = per_row * kept;
    for (int t0 = tid; t0 < total; t0 += kCompactBatch * NT) {
        E v[kCompactBatch];
#pragma unroll
        for (int u = 0; u < kCompactBatch; ++u) {
            const int t = t0 + u * NT;
            if (t < total) {
                const int k = fast_div(t, div);
                const int m = map[t - k * per_row];
                const int a = m >> 24;
                v[u] = __ldcg(reinterpret_cast<const E*>(S.arrays[a] + (long long)s_src[k] * S.row_bytes[a] +
                                                         (m & 0xffffff)));
            }
        }
#pragma unroll
        for (int u = 0; u < kCompactBatch; ++u) {
            const int t = t0 + u * NT;
            if (t < total) stage[t] = v[u];
        }
    }
}

template <typename E, int NT>
__device__ __forceinline__ void compact_store(const CompactScratch<NT>& S, const int* map, int per_row,
                                              const FastDiv& div, const int* s_dst, const E* stage, int kept,
                                              int tid) {
    const int total = per_row * kept;
    for (int t0 = tid; t0 < total; t0 += kCompactBatch * NT) {
#pragma unroll
        for (int u = 0; u < kCompactBatch; ++u) {
            const int t = t0 + u * NT;
            if (t < total) {
                const int k = fast_div(t, div);
                const int m = map[t - k * per_row];
                const int a = m >> 24;
                *reinterpret_cast<E*>(S.arrays[a] + (long long)s_dst[k] * S.row_bytes[a] + (m & 0xffffff)) = stage[t];
            }
        }
    }
}

// Move `kept` rows from s_src[k] to s_dst[k] through the stage: every load of
// every element size first, then a barrier, then the stores.
template <int NT>
__device__ __forceinline__ void compact_move(const CompactPlan& P, const CompactScratch<NT>& S, unsigned char* stage,
                                             const int* s_src, const int* s_dst, int kept, int tid) {
    uint4* s16 = reinterpret_cast<uint4*>(stage);
    uint32_t* s4 = reinterpret_cast<uint32_t*>(stage + 16LL * P.per_row[0] * kept);
    uint8_t* s1 = reinterpret_cast<uint8_t*>(stage + 16LL * P.per_row[0] * kept + 4LL * P.per_row[1] * kept);
    if (P.per_row[0]) compact_load<uint4, NT>(S, S.map[0], P.per_row[0], P.div_row[0], s_src, s16, kept, tid);
    if (P.per_row[1]) compact_load<uint32_t, NT>(S, S.map[1], P.per_row[1], P.div_row[1], s_src, s4, kept, tid);
    if (P.per_row[2]) compact_load<uint8_t, NT>(S, S.map[2], P.per_row[2], P.div_row[2], s_src, s1, kept, tid);
    __syncthreads();
    if (P.per_row[0]) compact_store<uint4, NT>(S, S.map[0], P.per_row[0], P.div_row[0], s_dst, s16, kept, tid);
    if (P.per_row[1]) compact_store<uint32_t, NT>(S, S.map[1], P.per_row[1], P.div_row[1], s_dst, s4, kept, tid);
    if (P.per_row[2]) compact_store<uint8_t, NT>(S, S.map[2], P.per_row[2], P.div_row[2], s_dst, s1, kept, tid);
}

// Compact A rows by evict[i] (nonzero: the row leaves), all NT threads of
// the CTA.  The element map must be built (compact_map) and the evict flags
// and rows visible to the whole CTA.  Rows and flags are read from L2 (they
// may have been written by other SMs while this one cached older lines).
// Writes new_index / src_row when given and *A_out; ends with a barrier.
template <int NT>
__device__ __forceinline__ void compact_rows(const CompactPlan& P, CompactScratch<NT>& S, unsigned char* stage,
                                             const uint8_t* evict, int A, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    int base = 0;      // survivors before the chunk
    for (int c0 = 0; c0 < A; c0 += P.chunk_rows) {
        const int i = c0 + tid;
        const bool in = tid < P.chunk_rows && i < A;
        const bool keep = in && __ldcg(evict + i) == 0;
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (lane == 0) S.wsum[warp] = __popc(bal);
        if (tid == 0) S.skip = 0x7fffffff;
        __syncthreads();
        int before = 0, kept = 0;
        for (int w = 0; w < NT / 32; ++w) {
            const int c = S.wsum[w];
            if (w < warp) before += c;
            kept += c;
        }
        const int rank = before + __popc(bal & ((1u << lane) - 1u));
        // survivors ahead of the first evicted row keep their index: they
        // are a prefix of the chunk's survivors and need no move
        const bool moves = keep && base + rank != i;
        const unsigned mv = __ballot_sync(0xffffffffu, moves);
        if (mv && lane == __ffs(mv) - 1) atomicMin(&S.skip, rank);
        if (in) {
            const int ni = keep ? base + rank : -1;
            if (P.new_index) P.new_index[i] = ni;
            if (keep) {
                if (P.src_row) P.src_row[ni] = i;
                S.src[rank] = i;
                S.dst[rank] = ni;
            }
        }
        __syncthreads();
        const int skip = min(S.skip, kept);
        compact_move<NT>(P, S, stage, S.src + skip, S.dst + skip, kept - skip, tid);
        __syncthreads();
        base += kept;
    }
    if (tid == 0) *P.A_out = base;
}

}  // namespace dllm
