// Mixed-state batch management around the step (S7-S9):
//   dllm_pack_plan / dllm_admit  host planning by eq. (1) and sand-fill,
//   dllm_pack                    the left-padded bounding box,
//   dllm_pack_block              its active-block columns only (in-place re-loop),
//   dllm_advance                 block commit, b += 1, eviction flags,
//   dllm_compact                 stable in-place compaction of row arrays,
//   dllm_advance_compact         both of the last two in one launch,
//   dllm_refill                  appending admitted requests.
// BlockServe page ("BlockServe: 块粒度连续批处理实现高吞吐扩散大语言模型服务"),
// sections II-C (Algorithm 1), II-D (eq. (1), sand-fill admission) and II-E
// (logical position alignment, gather/scatter of the active block); FDFO page,
// section "FDFO 的核心思想" (finished requests leave at once).
//
// These kernels move a few MB per call and are latency-bound; they are written
// for coalesced access (consecutive threads, consecutive columns) and a grid
// capped at a few CTAs per SM.

#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "common.cuh"
#include "compact.cuh"

namespace dllm {
namespace {

// ---------------------------------------------------------------------------
// dllm_pack
// ---------------------------------------------------------------------------
struct PackParams {
    int A, L, W, pad_id;
    const int* p;
    const int* b;
    const int* rid;
    const long long* prompt_off;
    const int* prompt_tokens;
    const int* gen_tokens;
    long long ld_gen;
    const int* block_ids;
    int* ids;
    uint8_t* attn;
    int* pos;
    int* pad;
    int* blk_start;
    int* err;
};

__global__ void __launch_bounds__(256) pack_kernel(const __grid_constant__ PackParams P) {
    pdl_wait();
    pdl_release();
    const long long total = (long long)P.A * P.W;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(idx / P.W);
        const int c = (int)(idx - (long long)i * P.W);
        // the row's scalars together: the token source below hangs off rid
        const int p = __ldg(P.p + i);
        const int b = __ldg(P.b + i);
        const int r = __ldg(P.rid + i);
        const long long width = (long long)p + (long long)(b + 1) * P.L;
        if (p < 0 || b < 0 || width > P.W || (p > 0 && !P.prompt_tokens) || (b > 0 && !P.gen_tokens)) {
            if (c == 0) set_error(P.err, DLLM_DEVERR_ROW_WIDTH);
            continue;
        }
        const int pad = P.W - (int)width;
        int tok, a, ps;
        if (c < pad) {
            tok = P.pad_id;
            a = 0;
            ps = 0;
        } else {
            const int k = c - pad;   // logical position: cumulative index over the mask
            a = 1;
            ps = k;
            if (k < p) {
                tok = __ldg(P.prompt_tokens + __ldg(P.prompt_off + r) + k);
            } else if (k < p + b * P.L) {
                tok = __ldg(P.gen_tokens + (long long)r * P.ld_gen + (k - p));
            } else {
                tok = __ldg(P.block_ids + (long long)i * P.L + (k - p - b * P.L));
            }
        }
        P.ids[idx] = tok;
        if (P.attn) P.attn[idx] = (uint8_t)a;
        if (P.pos) P.pos[idx] = ps;
        if (c == 0) {
            if (P.pad) P.pad[i] = pad;
            if (P.blk_start) P.blk_start[i] = p + b * P.L;
        }
    }
}

// ---------------------------------------------------------------------------
// dllm_advance: one warp per row
// ---------------------------------------------------------------------------
struct AdvanceParams {
    int A, L, mask_id;
    const uint8_t* advance;
    const int* rid;
    const int* K;
    int* b;
    int* ids;
    float* cs;
    int* gen;
    long long ld_gen;
    uint8_t* evict;
    int* err;
};

__global__ void __launch_bounds__(256) advance_kernel(const __grid_constant__ AdvanceParams P) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (i >= P.A) return;
    if (!P.advance[i]) {
        if (lane == 0) P.evict[i] = 0;
        return;
    }
    const int r = P.rid[i];
    const int b = P.b[i];
    const int K = P.K[i];
    if (b < 0 || b >= K || (long long)(b + 1) * P.L > P.ld_gen) {
        if (lane == 0) {
            set_error(P.err, DLLM_DEVERR_BLOCK_INDEX);
            P.evict[i] = 0;
        }
        return;
    }
    const long long src = (long long)i * P.L;
    const long long dst = (long long)r * P.ld_gen + (long long)b * P.L;
    for (int j = lane; j < P.L; j += 32) P.gen[dst + j] = P.ids[src + j];
    const bool ev = b + 1 >= K;
    __syncwarp();
    if (!ev) {
        const float qnan = __int_as_float(0x7fc00000);
        for (int j = lane; j < P.L; j += 32) {
            P.ids[src + j] = P.mask_id;
            P.cs[src + j] = qnan;
        }
    }
    if (lane == 0) {
        P.b[i] = b + 1;
        P.evict[i] = ev ? 1 : 0;
    }
}

// ---------------------------------------------------------------------------
// dllm_compact: scatter kept rows into the workspace, then copy back
// ---------------------------------------------------------------------------
constexpr int kCompactRows = 256;   // rows per CTA, one per thread for the scan

struct CompactParams {
    int A, n_arrays;
    const uint8_t* evict;
    int* new_index;
    int* src_row;
    int* A_out;
    unsigned char* arrays[DLLM_COMPACT_MAX_ARRAYS];
    unsigned char* stage[DLLM_COMPACT_MAX_ARRAYS];
    long long row_bytes[DLLM_COMPACT_MAX_ARRAYS];
};

// Copy `rows` rows of one array.  Thread t of nt handles 32-bit words (or
// bytes, when a row is not word-sized or the pointers are not word-aligned)
// t, t + nt, ... of the flattened rows, four loads in flight before their
// stores.  dst_row(r) < 0 skips row r.
template <typename T, typename DstRow>
__device__ __forceinline__ void copy_rows_t(T* __restrict__ dst, const T* __restrict__ src, int per_row, int rows,
                                            DstRow dst_row, int src_row0, int t, int nt) {
    const int total = per_row * rows;
    for (int k0 = t; k0 < total; k0 += 4 * nt) {
        T v[4];
        int d[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + u * nt;
            d[u] = -1;
            if (k < total) {
                const int r = k / per_row;
                const int w = k - r * per_row;
                const int dr = dst_row(r);
                if (dr >= 0) {
                    d[u] = dr * per_row + w;
                    v[u] = src[(src_row0 + r) * per_row + w];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (d[u] >= 0) dst[d[u]] = v[u];
    }
}

template <typename DstRow>
__device__ __forceinline__ void copy_rows(unsigned char* dst, const unsigned char* src, long long rb, int rows,
                                          DstRow dst_row, int src_row0, int t, int nt) {
    const uintptr_t al = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src);
    if ((rb & 3) == 0 && (al & 3) == 0)
        copy_rows_t(reinterpret_cast<uint32_t*>(dst), reinterpret_cast<const uint32_t*>(src), (int)(rb >> 2), rows,
                    dst_row, src_row0, t, nt);
    else
        copy_rows_t(dst, src, (int)rb, rows, dst_row, src_row0, t, nt);
}

// grid: (row tiles of kCompactRows, arrays); CTA (x, 0) also writes the maps
__global__ void __launch_bounds__(kCompactRows) compact_scatter_kernel(const __grid_constant__ CompactParams P) {
    __shared__ int s_warp[kCompactRows / 32];
    __shared__ int s_before;
    __shared__ int s_new[kCompactRows];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int i0 = blockIdx.x * kCompactRows;
    // kept rows before this CTA's range
    int pre = 0;
    for (int k = t; k < i0; k += kCompactRows) pre += P.evict[k] ? 0 : 1;
    for (int off = 16; off; off >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, off);
    if (lane == 0) s_warp[warp] = pre;
    __syncthreads();
    if (t == 0) {
        int acc = 0;
        for (int w = 0; w < kCompactRows / 32; ++w) acc += s_warp[w];
        s_before = acc;
    }
    __syncthreads();
    // stable rank inside the range
    const int i = i0 + t;
    const bool keep = i < P.A && !P.evict[i];
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_warp[warp] = __popc(bal);
    __syncthreads();
    int wbefore = 0, total = 0;
    for (int w = 0; w < kCompactRows / 32; ++w) {
        if (w < warp) wbefore += s_warp[w];
        total += s_warp[w];
    }
    const int ni = keep ? s_before + wbefore + __popc(bal & ((1u << lane) - 1u)) : -1;
    if (blockIdx.y == 0) {
        if (i < P.A) {
            if (P.new_index) P.new_index[i] = ni;
            if (keep && P.src_row) P.src_row[ni] = i;
        }
        if (i0 + kCompactRows >= P.A && t == 0) *P.A_out = s_before + total;   // last row tile
    }
    s_new[t] = ni;
    __syncthreads();
    // scatter the kept rows of array blockIdx.y into its staging copy
    const int a = blockIdx.y;
    if (a < P.n_arrays) {
        const int rows = min(kCompactRows, P.A - i0);
        copy_rows(P.stage[a], P.arrays[a], P.row_bytes[a], rows, [&](int r) { return s_new[r]; }, i0, t,
                  kCompactRows);
    }
}

// grid: (row-word blocks, arrays)
__global__ void __launch_bounds__(256) compact_copyback_kernel(const __grid_constant__ CompactParams P) {
    const int n = *P.A_out;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int nt = gridDim.x * blockDim.x;
    const int a = blockIdx.y;
    copy_rows(P.arrays[a], P.stage[a], P.row_bytes[a], n, [](int r) { return r; }, 0, t, nt);
}

// ---------------------------------------------------------------------------
// dllm_refill: initialise appended rows
// ---------------------------------------------------------------------------
struct RefillParams {
    int A0, n, L, mask_id;
    const int* new_rid;
    const int* new_p;
    const int* new_K;
    const float* new_thr;
    int* rid;
    int* p;
    int* b;
    int* K;
    float* thr;
    int* ids;
    float* cs;
};

__global__ void __launch_bounds__(256) refill_kernel(const __grid_constant__ RefillParams P) {
    const long long total = (long long)P.n * P.L;
    for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < total;
         k += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(k / P.L);
        const long long dst = (long long)(P.A0 + r) * P.L + (k - (long long)r * P.L);
        P.ids[dst] = P.mask_id;
        P.cs[dst] = __int_as_float(0x7fc00000);
        if (k - (long long)r * P.L == 0) {
            const int row = P.A0 + r;
            P.rid[row] = P.new_rid[r];
            P.p[row] = P.new_p[r];
            P.b[row] = 0;
            P.K[row] = P.new_K[r];
            P.thr[row] = P.new_thr[r];
        }
    }
}

inline size_t compact_ws_bytes(int A, int n, const int64_t* rb) {
    size_t total = 0;
    for (int k = 0; k < n; ++k) total += (size_t(A) * size_t(rb[k]) + 255) & ~size_t(255);
    return total + 256;
}

// Disjoint-set "nearest free slot" finder used by the admission planner.
struct NextFree {
    std::vector<int> parent;
    explicit NextFree(int n) : parent(n + 1) {
        for (int i = 0; i <= n; ++i) parent[i] = i;
    }
    int find(int i) {
        int r = i;
        while (parent[r] != r) r = parent[r];
        while (parent[i] != r) {
            const int nx = parent[i];
            parent[i] = r;
            i = nx;
        }
        return r;
    }
};

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" int dllm_pack_plan(int32_t A, const int32_t* p, const int32_t* b, int32_t L, int32_t* W, int64_t* cost) {
    if (A < 0 || L < 1) return DLLM_ERR_INVAL;
    if (A > 0 && (!p || !b)) return DLLM_ERR_INVAL;
    long long w = 0;
    for (int i = 0; i < A; ++i) {
        if (p[i] < 0 || b[i] < 0) return DLLM_ERR_INVAL;
        w = std::max(w, (long long)p[i] + ((long long)b[i] + 1) * L);
    }
    if (w > 0x7fffffffLL) return DLLM_ERR_UNSUPPORTED;
    if (W) *W = (int32_t)w;
    if (cost) *cost = (int64_t)A * w;
    return DLLM_OK;
}

extern "C" int dllm_admit(int32_t n_pending, const int32_t* pending_p, int32_t A, const int32_t* active_p,
                          const int32_t* active_b, int32_t L, int64_t budget, int32_t* admit_idx, int32_t* n_admit) {
    if (n_pending < 0 || A < 0 || L < 1 || !n_admit) return DLLM_ERR_INVAL;
    if (n_pending > 0 && (!pending_p || !admit_idx)) return DLLM_ERR_INVAL;
    if (A > 0 && (!active_p || !active_b)) return DLLM_ERR_INVAL;
    for (int k = 0; k < n_pending; ++k) {
        if (pending_p[k] < 0 || (k > 0 && pending_p[k] < pending_p[k - 1])) return DLLM_ERR_INVAL;
    }
    long long w_cur = 0;
    for (int i = 0; i < A; ++i) {
        if (active_p[i] < 0 || active_b[i] < 0) return DLLM_ERR_INVAL;
        w_cur = std::max(w_cur, (long long)active_p[i] + ((long long)active_b[i] + 1) * L);
    }
    long long count = A;
    // left: slot k + 1 stands for queue entry k, slot 0 for "none"; find()
    // gives the nearest free slot at or below.  right: find() gives the
    // nearest free entry at or above (n_pending for "none").
    NextFree left(n_pending), right(n_pending);
    auto take = [&](int k) {
        left.parent[k + 1] = k;
        right.parent[k] = k + 1;
    };
    auto free_at_or_below = [&](int k) { return left.find(k + 1) - 1; };
    auto free_at_or_above = [&](int k) { return right.find(k); };
    int n = 0;
    while (true) {
        const int head = free_at_or_above(0);
        if (head >= n_pending) break;
        int cand = -1;
        const long long lim = w_cur - L;   // fits without widening: p + L <= w_cur
        if (lim >= 0) {
            const int hi = int(std::upper_bound(pending_p, pending_p + n_pending, lim) - pending_p) - 1;
            const int k = hi >= 0 ? free_at_or_below(hi) : -1;
            if (k >= 0) {
                const int lo = int(std::lower_bound(pending_p, pending_p + n_pending, pending_p[k]) - pending_p);
                cand = free_at_or_above(lo);   // earliest free entry of the same length
            }
        }
        if (cand < 0) cand = head;
        const long long w_new = std::max(w_cur, (long long)pending_p[cand] + L);
        if ((count + 1) * w_new > budget) break;
        take(cand);
        admit_idx[n++] = cand;
        ++count;
        w_cur = w_new;
    }
    *n_admit = n;
    return DLLM_OK;
}

extern "C" int dllm_pack(const dllm_pack_args* a, void* stream) {
    if (!a || a->A < 0 || a->L < 1 || a->W < 0) return DLLM_ERR_INVAL;
    if (a->A == 0 || a->W == 0) return DLLM_OK;
    if (!a->p || !a->b || !a->rid || !a->prompt_off || !a->block_ids || !a->ids) return DLLM_ERR_INVAL;
    if (a->ld_gen < 0) return DLLM_ERR_INVAL;
    PackParams P;
    P.A = a->A; P.L = a->L; P.W = a->W; P.pad_id = a->pad_id;
    P.p = a->p; P.b = a->b; P.rid = a->rid; P.prompt_off = reinterpret_cast<const long long*>(a->prompt_off);
    P.prompt_tokens = a->prompt_tokens; P.gen_tokens = a->gen_tokens; P.ld_gen = a->ld_gen;
    P.block_ids = a->block_ids; P.ids = a->ids; P.attn = a->attn; P.pos = a->pos; P.pad = a->pad;
    P.blk_start = a->blk_start;
    P.err = error_word_ptr();
    if (!P.err) return DLLM_ERR_CUDA;
    const long long total = (long long)a->A * a->W;
    const int sms = sm_count();
    long long blocks = (total + 255) / 256;
    blocks = std::min<long long>(blocks, (long long)std::max(sms, 1) * 8);
    DLLM_CUDA_TRY(launch_dependent(pack_kernel, dim3((unsigned)blocks), dim3(256), 0, as_stream(stream), P));
    return DLLM_OK;
}

// ---------------------------------------------------------------------------
// dllm_pack_block: rewrite the active-block columns [W - L, W) of a packed
// box from the rows' current blocks (FDFO page, "工程设计四": with no block
// completed, the next step runs on the same batch).  One thread per token.
// ---------------------------------------------------------------------------
namespace dllm {
namespace {

__global__ void __launch_bounds__(256) pack_block_kernel(int A, int L, int W, const int* __restrict__ block_ids,
                                                         int* __restrict__ ids) {
    const long long n = (long long)A * L;
    for (long long t = blockIdx.x * 256ll + threadIdx.x; t < n; t += (long long)gridDim.x * 256) {
        const int i = (int)(t / L), j = (int)(t - (long long)i * L);
        ids[(long long)i * W + (W - L) + j] = block_ids[t];
    }
}

}  // namespace
}  // namespace dllm

extern "C" int dllm_pack_block(const dllm_pack_args* a, void* stream) {
    if (!a || a->A < 0 || a->L < 1) return DLLM_ERR_INVAL;
    if (a->A == 0) return DLLM_OK;
    if (a->W < a->L || !a->block_ids || !a->ids) return DLLM_ERR_INVAL;
    const long long total = (long long)a->A * a->L;
    const int sms = sm_count();
    long long blocks = (total + 255) / 256;
    blocks = std::min<long long>(blocks, (long long)std::max(sms, 1) * 8);
    pack_block_kernel<<<(unsigned)blocks, 256, 0, as_stream(stream)>>>(a->A, a->L, a->W, a->block_ids, a->ids);
    DLLM_CUDA_TRY(cudaGetLastError());
    return DLLM_OK;
}

extern "C" int dllm_advance(const dllm_advance_args* a, void* stream) {
    if (!a || a->A < 0 || a->L < 1 || a->L > DLLM_MAX_L || a->ld_gen < 0) return DLLM_ERR_INVAL;
    if (a->A == 0) return DLLM_OK;
    if (!a->advance || !a->rid || !a->K || !a->b || !a->input_ids || !a->conf_state || !a->gen_tokens || !a->evict)
        return DLLM_ERR_INVAL;
    AdvanceParams P;
    P.A = a->A; P.L = a->L; P.mask_id = a->mask_id;
    P.advance = a->advance; P.rid = a->rid; P.K = a->K; P.b = a->b; P.ids = a->input_ids;
    P.cs = a->conf_state; P.gen = a->gen_tokens; P.ld_gen = a->ld_gen; P.evict = a->evict;
    P.err = error_word_ptr();
    if (!P.err) return DLLM_ERR_CUDA;
    const int wpb = 8;
    advance_kernel<<<(a->A + wpb - 1) / wpb, wpb * 32, 0, as_stream(stream)>>>(P);
    DLLM_CUDA_TRY(cudaGetLastError());
    return DLLM_OK;
}

// ---------------------------------------------------------------------------
// dllm_advance_compact: dllm_advance then dllm_compact by its evict flags, in
// one launch of one CTA (the compaction itself: compact.cuh).
// ---------------------------------------------------------------------------
namespace dllm {
namespace {

constexpr int kFusedThreads = 1024;
constexpr int kFusedStageBytes = 96 * 1024;
constexpr int kFusedBatch = kCompactBatch;   // global loads in flight per thread

struct FusedParams {
    AdvanceParams adv;
    CompactPlan cp;
};

// The block commit of dllm_advance for all rows, by one CTA, 1024 rows at a
// time: one thread per row reads its row's state and writes b and evict,
// then every thread copies block tokens, one element each.
__device__ __forceinline__ void advance_rows(const AdvanceParams& P, long long* s_dst, uint8_t* s_ev, int tid) {
    for (int c0 = 0; c0 < P.A; c0 += kFusedThreads) {
        const int i = c0 + tid;
        long long dst = -1;
        bool ev = false;
        if (i < P.A) {
            // all four loads in flight together
            const int adv = P.advance[i];
            const int r = P.rid[i];
            const int b = P.b[i];
            const int K = P.K[i];
            if (adv) {
                if (b < 0 || b >= K || (long long)(b + 1) * P.L > P.ld_gen) {
                    set_error(P.err, DLLM_DEVERR_BLOCK_INDEX);
                } else {
                    dst = (long long)r * P.ld_gen + (long long)b * P.L;
                    ev = b + 1 >= K;
                    P.b[i] = b + 1;
                }
            }
            P.evict[i] = ev ? 1 : 0;
        }
        s_dst[tid] = dst;
        s_ev[tid] = ev ? 1 : 0;
        __syncthreads();
        const int rows = min(kFusedThreads, P.A - c0);
        const int n = rows * P.L;   // <= 1024 * DLLM_MAX_L
        int* ids = P.ids + (long long)c0 * P.L;
        float* cs = P.cs + (long long)c0 * P.L;
        const float qnan = __int_as_float(0x7fc00000);
        // kFusedBatch tokens per thread in flight: every load, then the stores
        for (int t0 = tid; t0 < n; t0 += kFusedBatch * kFusedThreads) {
            int v[kFusedBatch];
#pragma unroll
            for (int u = 0; u < kFusedBatch; ++u) {
                const int t = t0 + u * kFusedThreads;
                v[u] = (t < n && s_dst[t / P.L] >= 0) ? ids[t] : 0;
            }
#pragma unroll
            for (int u = 0; u < kFusedBatch; ++u) {
                const int t = t0 + u * kFusedThreads;
                if (t >= n) break;
                const int row = t / P.L;
                const long long d = s_dst[row];
                if (d < 0) continue;
                P.gen[d + (t - row * P.L)] = v[u];
                if (!s_ev[row]) {
                    ids[t] = P.mask_id;
                    cs[t] = qnan;
                }
            }
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kFusedThreads) advance_compact_kernel(const __grid_constant__ FusedParams P) {
    extern __shared__ __align__(16) unsigned char stage[];
    __shared__ CompactScratch<kFusedThreads> s_cp;
    __shared__ long long s_gen_dst[kFusedThreads];
    __shared__ uint8_t s_ev[kFusedThreads];
    const int tid = threadIdx.x;
    // the element map depends on launch parameters only: built before
    // waiting on the previous kernel
    compact_map<kFusedThreads>(P.cp, s_cp, tid);
    pdl_wait();
    pdl_release();
    advance_rows(P.adv, s_gen_dst, s_ev, tid);   // ends with a barrier: evict, ids, cs, b visible CTA-wide
    compact_rows<kFusedThreads>(P.cp, s_cp, stage, P.adv.evict, P.adv.A, tid);
}

}  // namespace
}  // namespace dllm

extern "C" int dllm_advance_compact(const dllm_advance_args* a, const dllm_compact_args* c, void* stream) {
    if (!a || !c || a->A < 0 || a->L < 1 || a->L > DLLM_MAX_L || a->ld_gen < 0 || c->A != a->A) return DLLM_ERR_INVAL;
    if (a->A > 0 && (!a->advance || !a->rid || !a->K || !a->b || !a->input_ids || !a->conf_state ||
                     !a->gen_tokens || !a->evict))
        return DLLM_ERR_INVAL;
    FusedParams P;
    P.adv.A = a->A; P.adv.L = a->L; P.adv.mask_id = a->mask_id;
    P.adv.advance = a->advance; P.adv.rid = a->rid; P.adv.K = a->K; P.adv.b = a->b; P.adv.ids = a->input_ids;
    P.adv.cs = a->conf_state; P.adv.gen = a->gen_tokens; P.adv.ld_gen = a->ld_gen; P.adv.evict = a->evict;
    P.adv.err = error_word_ptr();
    if (!P.adv.err) return DLLM_ERR_CUDA;
    const int prc = make_compact_plan(c, kFusedThreads, kFusedStageBytes, &P.cp);
    if (prc != DLLM_OK) return prc;
    // rows beyond one staging chunk: one CTA would serialise them; with a
    // compaction workspace, run the multi-CTA advance and compaction instead
    if ((long long)a->A * P.cp.row_total > kFusedStageBytes && c->workspace &&
        c->workspace_bytes >= dllm_compact_workspace_size(c->A, c->n_arrays, c->row_bytes)) {
        const int rc = dllm_advance(a, stream);
        if (rc != DLLM_OK) return rc;
        dllm_compact_args c2 = *c;
        c2.evict = a->evict;
        return dllm_compact(&c2, stream);
    }
    int dev = 0;
    DLLM_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return DLLM_ERR_UNSUPPORTED;
    static std::atomic<bool> configured[64];
    if (!configured[dev].load(std::memory_order_acquire)) {
        DLLM_CUDA_TRY(cudaFuncSetAttribute(advance_compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kFusedStageBytes));
        configured[dev].store(true, std::memory_order_release);
    }
    DLLM_CUDA_TRY(launch_dependent(advance_compact_kernel, dim3(1), dim3(kFusedThreads), (size_t)kFusedStageBytes,
                                   as_stream(stream), P));
    return DLLM_OK;
}

extern "C" size_t dllm_compact_workspace_size(int32_t A, int32_t n_arrays, const int64_t* row_bytes) {
    if (A < 0 || n_arrays < 0 || n_arrays > DLLM_COMPACT_MAX_ARRAYS) return 0;
    if (n_arrays > 0 && !row_bytes) return 0;
    for (int k = 0; k < n_arrays; ++k)
        if (row_bytes[k] <= 0) return 0;
    return compact_ws_bytes(A, n_arrays, row_bytes);
}

extern "C" int dllm_compact(const dllm_compact_args* a, void* stream) {
    if (!a || a->A < 0 || a->n_arrays < 0 || a->n_arrays > DLLM_COMPACT_MAX_ARRAYS) return DLLM_ERR_INVAL;
    if (!a->A_out) return DLLM_ERR_INVAL;
    cudaStream_t s = as_stream(stream);
    if (a->A == 0) {
        DLLM_CUDA_TRY(cudaMemsetAsync(a->A_out, 0, sizeof(int32_t), s));
        return DLLM_OK;
    }
    if (!a->evict) return DLLM_ERR_INVAL;
    for (int k = 0; k < a->n_arrays; ++k)
        if (!a->arrays[k] || a->row_bytes[k] <= 0) return DLLM_ERR_INVAL;
    const size_t need = compact_ws_bytes(a->A, a->n_arrays, a->row_bytes);
    if (a->n_arrays > 0 && (!a->workspace || a->workspace_bytes < need)) return DLLM_ERR_WORKSPACE;
    CompactParams P;
    P.A = a->A; P.n_arrays = a->n_arrays; P.evict = a->evict; P.new_index = a->new_index;
    P.src_row = a->src_row; P.A_out = a->A_out;
    size_t off = 0;
    unsigned char* ws = static_cast<unsigned char*>(a->workspace);
    for (int k = 0; k < DLLM_COMPACT_MAX_ARRAYS; ++k) {
        P.arrays[k] = nullptr;
        P.stage[k] = nullptr;
        P.row_bytes[k] = 0;
        if (k < a->n_arrays) {
            P.arrays[k] = static_cast<unsigned char*>(a->arrays[k]);
            P.row_bytes[k] = a->row_bytes[k];
            P.stage[k] = ws + off;
            off += (size_t(a->A) * size_t(a->row_bytes[k]) + 255) & ~size_t(255);
        }
    }
    for (int k = 0; k < a->n_arrays; ++k)
        if ((long long)a->A * a->row_bytes[k] > 0x7fffffffLL) return DLLM_ERR_UNSUPPORTED;
    const dim3 grid((a->A + kCompactRows - 1) / kCompactRows, std::max(a->n_arrays, 1));
    compact_scatter_kernel<<<grid, kCompactRows, 0, s>>>(P);
    DLLM_CUDA_TRY(cudaGetLastError());
    if (a->n_arrays > 0) {
        long long words = 0;
        for (int k = 0; k < a->n_arrays; ++k)
            words = std::max(words, (long long)a->A * ((a->row_bytes[k] + 3) / 4));
        const int sms = std::max(sm_count(), 1);
        const int cbx = (int)std::max(1LL, std::min((words + 1023) / 1024, (long long)sms));
        compact_copyback_kernel<<<dim3(cbx, a->n_arrays), 256, 0, s>>>(P);
        DLLM_CUDA_TRY(cudaGetLastError());
    }
    return DLLM_OK;
}

extern "C" int dllm_refill(const dllm_refill_args* a, void* stream) {
    if (!a || a->A0 < 0 || a->n < 0 || a->L < 1 || a->L > DLLM_MAX_L) return DLLM_ERR_INVAL;
    if (a->n == 0) return DLLM_OK;
    if (!a->new_rid || !a->new_p || !a->new_K || !a->new_thr || !a->rid || !a->p || !a->b || !a->K || !a->thr ||
        !a->input_ids || !a->conf_state)
        return DLLM_ERR_INVAL;
    RefillParams P;
    P.A0 = a->A0; P.n = a->n; P.L = a->L; P.mask_id = a->mask_id;
    P.new_rid = a->new_rid; P.new_p = a->new_p; P.new_K = a->new_K; P.new_thr = a->new_thr;
    P.rid = a->rid; P.p = a->p; P.b = a->b; P.K = a->K; P.thr = a->thr; P.ids = a->input_ids; P.cs = a->conf_state;
    const long long total = (long long)a->n * a->L;
    const int sms = std::max(sm_count(), 1);
    const int blocks = (int)std::max(1LL, std::min((total + 255) / 256, (long long)sms * 4));
    refill_kernel<<<blocks, 256, 0, as_stream(stream)>>>(P);
    DLLM_CUDA_TRY(cudaGetLastError());
    return DLLM_OK;
}
