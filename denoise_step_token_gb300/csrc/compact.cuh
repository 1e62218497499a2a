// Stable in-place compaction of SoA row arrays by eviction flags, staged
// through shared memory by one CTA (BlockServe page, Algorithm 1 and section
// II-E: finished requests leave the batch, survivors keep their order).
// Used by the single-CTA commit of pack.cu and by the last CTA of the step
// kernel's fused commit.
//
// Rows are compacted in chunks of rows in increasing order: a chunk's
// surviving rows are first staged in shared memory (every array's slice of a
// row side by side), then written to their new rows.  A destination is never
// above its source, so it lies in a chunk already staged (this one or an
// earlier one) and nothing is overwritten before it is read.  Survivors
// ahead of the first evicted row keep their index and are not moved.
#pragma once

#include <stdint.h>

#include <algorithm>

#include "common.cuh"

namespace dllm {

constexpr int kCompactMapWords = 2048;   // elements per staged row the element map covers
constexpr int kCompactBatch = 16;        // global loads (and stores) in flight per thread

struct CompactPlan {
    int n_arrays, chunk_rows, word;   // word: 4-byte elements (else bytes)
    unsigned char* arrays[DLLM_COMPACT_MAX_ARRAYS];
    long long row_bytes[DLLM_COMPACT_MAX_ARRAYS];
    long long stage_off[DLLM_COMPACT_MAX_ARRAYS];   // per-row offset of each array in a staged row
    long long row_total;                            // staged bytes per row
    FastDiv div_row;                                // division by the staged elements per row
    int* new_index;
    int* src_row;
    int* A_out;
};

// Host: fill a plan from dllm_compact_args for `threads` threads and
// `stage_bytes` of staging.  DLLM_OK, DLLM_ERR_INVAL or
// DLLM_ERR_UNSUPPORTED (a row wider than the staging or the element map).
inline int make_compact_plan(const dllm_compact_args* c, int threads, long long stage_bytes, CompactPlan* P) {
    if (c->n_arrays < 0 || c->n_arrays > DLLM_COMPACT_MAX_ARRAYS || !c->A_out) return DLLM_ERR_INVAL;
    P->n_arrays = c->n_arrays;
    P->row_total = 0;
    bool word = true;
    for (int k = 0; k < c->n_arrays; ++k) {
        if ((c->A > 0 && !c->arrays[k]) || c->row_bytes[k] <= 0) return DLLM_ERR_INVAL;
        P->arrays[k] = static_cast<unsigned char*>(c->arrays[k]);
        P->row_bytes[k] = c->row_bytes[k];
        word = word && (c->row_bytes[k] % 4 == 0) && (reinterpret_cast<uintptr_t>(c->arrays[k]) % 4 == 0);
    }
    for (int k = 0; k < c->n_arrays; ++k) {
        P->stage_off[k] = P->row_total;
        P->row_total += (c->row_bytes[k] + 3) & ~3ll;   // 4-byte aligned slots
    }
    if (P->row_total > stage_bytes) return DLLM_ERR_UNSUPPORTED;
    P->word = word ? 1 : 0;
    if (P->row_total / (word ? 4 : 1) > kCompactMapWords) return DLLM_ERR_UNSUPPORTED;
    P->chunk_rows = P->row_total > 0 ? (int)std::min<long long>(threads, stage_bytes / P->row_total) : threads;
    P->div_row = make_fastdiv((uint32_t)std::max<long long>(1, P->row_total / (word ? 4 : 1)));
    P->new_index = c->new_index;
    P->src_row = c->src_row;
    P->A_out = c->A_out;
    return DLLM_OK;
}

// Shared-memory scratch of one compaction: the element map (per element of
// a staged row, its array << 24 | its byte offset in that array's row, -1
// in padding), the arrays' addresses and row sizes, and per-chunk row
// indices (NT threads).
template <int NT>
struct CompactScratch {
    int map[kCompactMapWords];
    unsigned char* arrays[DLLM_COMPACT_MAX_ARRAYS];
    long long row_bytes[DLLM_COMPACT_MAX_ARRAYS];
    int src[NT], dst[NT];
    int wsum[NT / 32];
    int skip;
};

// The element map of a staged row, and the arrays' addresses and row sizes.
template <int NT>
__device__ __forceinline__ void compact_map(const CompactPlan& P, CompactScratch<NT>& S, int tid) {
    const int es = P.word ? 4 : 1;
    const int per_row = (int)(P.row_total / es);
    for (int w = tid; w < per_row; w += NT) {
        const long long off = (long long)w * es;
        int arr = -1, o = 0;
        for (int a = P.n_arrays - 1; a >= 0; --a) {
            if (off >= P.stage_off[a]) {
                if (off - P.stage_off[a] < P.row_bytes[a]) {
                    arr = a;
                    o = (int)(off - P.stage_off[a]);
                }
                break;
            }
        }
        S.map[w] = arr < 0 ? -1 : (arr << 24) | o;
    }
    if (tid < P.n_arrays) {
        S.arrays[tid] = P.arrays[tid];
        S.row_bytes[tid] = P.row_bytes[tid];
    }
}

template <int NT, typename E>
__device__ __forceinline__ void compact_move(const CompactPlan& P, const CompactScratch<NT>& S, unsigned char* stage,
                                             const int* s_src, const int* s_dst, int kept, int tid) {
    // Staged row k (all arrays side by side) at stage + k * row_total.  The
    // chunk's elements over every array form one flat range (32-bit indices:
    // the stage is at most a few hundred KiB); the element map gives each
    // place in a staged row its array and byte offset.  kCompactBatch loads
    // per thread are in flight before their stores, and the same number of
    // stores after the barrier.
    const int per_row = (int)(P.row_total / (long long)sizeof(E));
    const int total = per_row * kept;
    for (int t0 = tid; t0 < total; t0 += kCompactBatch * NT) {
        E v[kCompactBatch];
#pragma unroll
        for (int u = 0; u < kCompactBatch; ++u) {
            const int t = t0 + u * NT;
            v[u] = E(0);
            if (t < total) {
                const int k = fast_div(t, P.div_row);
                const int m = S.map[t - k * per_row];
                if (m >= 0) {
                    const int a = m >> 24;
                    v[u] = __ldcg(reinterpret_cast<const E*>(S.arrays[a] + (long long)s_src[k] * S.row_bytes[a] +
                                                             (m & 0xffffff)));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kCompactBatch; ++u) {
            const int t = t0 + u * NT;
            if (t < total) reinterpret_cast<E*>(stage)[t] = v[u];
        }
    }
    __syncthreads();
    for (int t0 = tid; t0 < total; t0 += kCompactBatch * NT) {
#pragma unroll
        for (int u = 0; u < kCompactBatch; ++u) {
            const int t = t0 + u * NT;
            if (t < total) {
                const int k = fast_div(t, P.div_row);
                const int m = S.map[t - k * per_row];
                if (m >= 0) {
                    const int a = m >> 24;
                    *reinterpret_cast<E*>(S.arrays[a] + (long long)s_dst[k] * S.row_bytes[a] + (m & 0xffffff)) =
                        reinterpret_cast<const E*>(stage)[t];
                }
            }
        }
    }
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
        if (P.word) compact_move<NT, uint32_t>(P, S, stage, S.src + skip, S.dst + skip, kept - skip, tid);
        else compact_move<NT, uint8_t>(P, S, stage, S.src + skip, S.dst + skip, kept - skip, tid);
        __syncthreads();
        base += kept;
    }
    if (tid == 0) *P.A_out = base;
}

}  // namespace dllm
