// dllm_step and dllm_features: the denoise step of block-wise diffusion-LLM
// serving (S1-S6), one fused, persistent kernel per call.
//
// Method (FDFO page "FDFO: 让 dLLM 推理从「整批等最慢」变成「谁先完成谁先走」",
// sections "工程设计一" and "工程设计二"; DiLaServe review, sections 3.1 and
// 4.2 item ③): for every masked position read the bf16 logits row, take the
// softmax probability of the argmax token as its confidence, unmask the
// positions above the request's threshold (or the single most confident one),
// write the tokens, report done / accept_length and the confidence features.
//
// Kernel design (GB300: 152 SMs, one CTA per SM, warp-specialised):
//   S1  every CTA scans input_ids once into shared bitmasks, ranks the masked
//       rows and takes an equal share of the element stream of all but the
//       last min(M/4, 1024) masked rows; those (the tail) are shared by all
//       CTAs.
//   S2  work unit = one fixed 8192-element chunk of one masked row.  Each
//       streaming warp takes chunks from the CTA's pool (a shared counter),
//       then from the shared tail (tickets on a global counter), and runs
//       its own ring of bulk copies (cp.async.bulk, the TMA engine, L2
//       evict-first) into shared memory; being the only reader of its ring,
//       it sees every barrier phase in order.  Each lane folds its elements
//       into an online (max, sum of exp, first argmax batch) with a packed
//       bf16x2 max and one FFMA + MUFU.EX2 + FADD per element; the warp then
//       writes each chunk partial as one 64-bit word and counts the chunks
//       on the row's counter, both relaxed (no fence on the streaming path).
//   Rows: the add that completes a row queues it for the CTA's finisher
//       warps, which read the row's partial words (polling any still in
//       flight), fold them in a fixed order, write conf = 1/s,
//       lse = m + ln s and the argmax token, and count the row towards its
//       request; the request's last row runs S3-S6 for it (selection,
//       fallback, update, done, quantile features by rank).
// The chunk split, lane mapping and fold order depend only on V, so a
// request's results are bit-identical whatever else is in the batch.  No
// CTA waits for another to make progress: counters elect the last arriver,
// and a finisher waits only for stores already issued to land.  input_ids is
// written only after every CTA has finished scanning it (otherwise the
// grid's last CTA to exit writes it), so a CTA that starts late still sees
// the entry state.  Every wait inside a CTA is bounded in time.

#include <math.h>
#include <stdint.h>

#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "compact.cuh"

namespace dllm {
namespace {

// Pipeline shape (tunable at build time; the defaults are the measured best).
#ifndef DLLM_STEP_WARPS
#define DLLM_STEP_WARPS 14
#endif
#ifndef DLLM_STEP_FINISHERS
#define DLLM_STEP_FINISHERS 1
#endif
#ifndef DLLM_STEP_STAGES
#define DLLM_STEP_STAGES 3
#endif
#ifndef DLLM_STEP_COPY_ELEMS
#define DLLM_STEP_COPY_ELEMS 2048
#endif
#ifndef DLLM_STEP_CHUNK_ELEMS
#define DLLM_STEP_CHUNK_ELEMS 8192
#endif
#ifndef DLLM_STEP_GROUP
#define DLLM_STEP_GROUP 2
#endif
#ifndef DLLM_STEP_TAIL_DEN
#define DLLM_STEP_TAIL_DEN 4
#endif
#ifndef DLLM_STEP_IDLE_NS
#define DLLM_STEP_IDLE_NS 64  // a warp with an empty finish queue sleeps this long between polls
#endif
#ifndef DLLM_STEP_F32X2
#define DLLM_STEP_F32X2 1     // packed f32x2 FMA / add in the element loop
#endif

constexpr int kStreamWarps = DLLM_STEP_WARPS;         // warps streaming logits
constexpr int kFinishWarps = DLLM_STEP_FINISHERS;     // warps finishing rows and requests
constexpr int kFirstFinisher = kStreamWarps;
constexpr int kWarpsTotal = kStreamWarps + kFinishWarps;
constexpr int kThreads = kWarpsTotal * 32;
constexpr int kStages = DLLM_STEP_STAGES;             // bulk copies in flight per streaming warp
constexpr int kCopyElems = DLLM_STEP_COPY_ELEMS;      // one bulk copy
constexpr int kCopyBytes = kCopyElems * 2;
constexpr int kChunkElems = DLLM_STEP_CHUNK_ELEMS;    // fixed reduction chunk of a row
constexpr int kGroup = DLLM_STEP_GROUP;               // chunks of one row taken at once
constexpr int kTailDen = DLLM_STEP_TAIL_DEN;          // up to 1/kTailDen of the masked rows ...
constexpr int kTailRowsMax = 1024;                    // ... and at most this many are shared by all CTAs
constexpr int kBatchVecs = 8;                         // 16-byte vectors per lane per batch
constexpr int kBatchElems = kBatchVecs * 8 * 32;      // 2048 contiguous elements
constexpr int kBatchesPerCopy = kCopyElems / kBatchElems;
constexpr int kBatchesPerChunk = kChunkElems / kBatchElems;
constexpr float kLog2e = 1.4426950408889634f;
#ifndef DLLM_STEP_WAIT_LIMIT_NS
#define DLLM_STEP_WAIT_LIMIT_NS 1000000000ull          // 1 s for any single wait
#endif
constexpr uint64_t kWaitLimitNs = DLLM_STEP_WAIT_LIMIT_NS;

static_assert(kCopyElems % kBatchElems == 0, "a copy holds whole batches");
static_assert(kChunkElems % kCopyElems == 0, "a chunk holds whole copies");
static_assert(kStages >= 1 && kStages <= 8, "pipeline depth");
static_assert(kTailDen >= 1 && kTailDen <= 64, "tail share");

// A chunk partial in one 64-bit word, written with a single relaxed store:
// low half = the chunk max m (a bf16 value, so the low 16 bits of its fp32
// pattern are zero) with (first batch holding m) + 1 in those 16 bits; high
// half = sum of exp(x - m) over the chunk.  A zero word is "not yet written":
// partial words are zero at rest and the row finisher clears them.
__device__ __forceinline__ unsigned long long pack_partial(float m, float s, int kb) {
    const uint32_t lo = (__float_as_uint(m) & 0xffff0000u) | (uint32_t)(kb + 1);
    return ((unsigned long long)__float_as_uint(s) << 32) | lo;
}
__device__ __forceinline__ void unpack_partial(unsigned long long w, float& m, float& s, int& kb) {
    const uint32_t lo = (uint32_t)w;
    m = __uint_as_float(lo & 0xffff0000u);
    kb = (int)(lo & 0xffffu) - 1;
    s = __uint_as_float((uint32_t)(w >> 32));
}

// A finished row in one 64-bit word: low half = conf, high half = the
// argmax token with the top bit set (so the word is never zero); token
// 0x7fffffff stands for "none found" (-1).
__device__ __forceinline__ unsigned long long pack_row(float conf, int tok) {
    const uint32_t hi = 0x80000000u | ((uint32_t)tok & 0x7fffffffu);
    return ((unsigned long long)hi << 32) | __float_as_uint(conf);
}
__device__ __forceinline__ void unpack_row(unsigned long long w, float& conf, int& tok) {
    conf = __uint_as_float((uint32_t)w);
    const int t = (int)((uint32_t)(w >> 32) & 0x7fffffffu);
    tok = (t == 0x7fffffff) ? -1 : t;
}

// Poll a zero-at-rest word until its (already issued) store lands; bounded.
__device__ __noinline__ unsigned long long poll_word(const unsigned long long* p, int* err) {
    const uint64_t t0 = globaltimer_ns();
    uint32_t spins = 0;
    unsigned long long w;
    while ((w = ld_relaxed_gpu_u64(p)) == 0ull) {
        __nanosleep(32);
        if ((++spins & 63u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            set_error(err, DLLM_DEVERR_TIMEOUT);
            break;
        }
    }
    return w;
}

struct StepParams {
    int B, L, V, NC, BL, mask_id, list_cap, static_cap, zero_cap;
    int compact;              // logits rows hold only the masked positions, by rank
    long long logits_rows;    // rows of a compact logits array
    int shard;                // S2 only, over a vocabulary shard starting at token v0
    int v0;
    float* trip_m;            // [BL] shard max, sum of exp, global argmax
    float* trip_s;
    int* trip_i;
    FastDiv div_nc, div_g;   // division by NC and by the grid size
    long long ldv;
    const uint16_t* logits;
    int* ids;
    const float* thr;
    const int* quota;   // [B] positions to unmask (fixed-steps rule), or null (threshold rule)
    float* cs;
    uint8_t* done;
    int* accept;
    int* n_new;
    float* feats;
    float* conf_out;
    float* lse_out;
    int* tok_out;
    int* ctl;        // [0] CTAs done scanning, [1] CTAs exited (low 16 bits) and deferred
                     // commits (high bits), [2] tail tickets drawn
    int* cnt;        // [BL] row counters, [B] request counters, [B] deferred-commit list
    unsigned long long* part;   // [BL * NC] packed chunk partials, zero at rest
    unsigned long long* row_word;   // [BL] a finished row's conf and token, zero at rest
    int* row_tok;
    uint8_t* sel;
    int* err;
    // fused commit (dllm_step_commit); commit == 0 otherwise
    int commit;
    const int* c_rid;   // [B] request id of each row
    const int* c_K;     // [B] blocks of each request
    int* c_b;           // [B] current block index (in/out)
    int* c_gen;         // committed tokens, row rid at c_gen + rid * c_ld_gen
    long long c_ld_gen;
    uint8_t* c_evict;   // [B] out: the row leaves the batch
    CompactPlan cp;     // stable compaction of the caller's row arrays by c_evict
    // vocabulary shards in one launch (dllm_step_vocab_shards); n_shards == 0
    // otherwise.  A row's chunks are shard 0's, then shard 1's, ...: shard k
    // holds chunks [sh_c0[k], sh_c0[k + 1]).
    int n_shards;
    const uint16_t* sh_logits[DLLM_MAX_VOCAB_SHARDS];
    long long sh_ldv[DLLM_MAX_VOCAB_SHARDS];
    int sh_v0[DLLM_MAX_VOCAB_SHARDS];
    int sh_V[DLLM_MAX_VOCAB_SHARDS];
    int sh_c0[DLLM_MAX_VOCAB_SHARDS + 1];
};

// Where chunk c of a row lives: its logits array and row stride, its first
// element within that array's row, its length, and its vocabulary shard
// (-1 without shards).
struct ChunkRef {
    const uint16_t* base;
    long long ldv;
    int start, len, shard;
};
__device__ __forceinline__ ChunkRef chunk_ref(const StepParams& P, int c) {
    if (P.n_shards == 0) return ChunkRef{P.logits, P.ldv, c * kChunkElems, min(kChunkElems, P.V - c * kChunkElems), -1};
    int k = 0;
#pragma unroll
    for (int i = 1; i < DLLM_MAX_VOCAB_SHARDS; ++i)
        if (i < P.n_shards && c >= P.sh_c0[i]) k = i;
    const int start = (c - P.sh_c0[k]) * kChunkElems;
    return ChunkRef{P.sh_logits[k], P.sh_ldv[k], start, min(kChunkElems, P.sh_V[k] - start), k};
}

// A deferred commit's list entry: the request, and whether its block is
// reset for the next one (fused commit) rather than given its new tokens.
constexpr int kDeferReset = 0x40000000;

// The fused commit's compaction scratch and staging, in the copy rings.
constexpr int kCommitScratchBytes = (int)((sizeof(CompactScratch<kThreads>) + 127) & ~size_t(127));
constexpr long long kCommitStageBytes = (long long)kStreamWarps * kStages * kCopyBytes - kCommitScratchBytes;
static_assert(kCommitStageBytes >= 16384, "the copy rings hold the commit's scratch and a useful stage");

// Workspace layout.  The first quarter holds everything that must be zero
// between calls (control words, counters, chunk partials); per-call data
// sits at the end, so calls of different shapes never put data on each
// other's zero-at-rest words.
struct WsLayout {
    size_t front, counters_bytes, data_bytes;
    size_t off_part, off_row;   // from the workspace start, inside the front quarter
    size_t off_tok, off_sel;    // from the data start
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline bool ws_layout_nc(long long B, long long L, long long NC, size_t bytes, WsLayout* w) {
    const long long BL = B * L;
    w->off_part = align256(64 + 4 * size_t(BL + 2 * B));
    w->off_row = align256(w->off_part + size_t(BL * NC) * 8);
    w->counters_bytes = w->off_row + size_t(BL) * 8;
    size_t d = 0;
    w->off_tok = d;  d = align256(d + size_t(BL) * 4);
    w->off_sel = d;  d = align256(d + size_t(BL));
    w->data_bytes = d;
    w->front = (bytes / 4) & ~size_t(255);
    return w->counters_bytes <= w->front && w->data_bytes + w->front <= bytes;
}

inline bool ws_layout(long long B, long long L, long long V, size_t bytes, WsLayout* w) {
    return ws_layout_nc(B, L, (V + kChunkElems - 1) / kChunkElems, bytes, w);
}

inline size_t ws_required(long long B, long long L, long long V) {
    WsLayout w;
    ws_layout(B, L, V, 0, &w);
    size_t need = w.counters_bytes * 4;
    const size_t need_data = (w.data_bytes * 4 + 2) / 3 + 256;
    if (need_data > need) need = need_data;
    need = align256(need + 256);
    while (!ws_layout(B, L, V, need, &w)) need += 256;
    return need;
}

// ---------------------------------------------------------------------------
// Per-lane batch processing.
// ---------------------------------------------------------------------------
// Packed per-vector maxima of a lane's batch, and the batch maximum.
__device__ __forceinline__ float batch_max(const uint4 (&v)[kBatchVecs], uint32_t (&vm)[kBatchVecs]) {
#pragma unroll
    for (int k = 0; k < kBatchVecs; ++k) vm[k] = bf16x2_max(bf16x2_max(v[k].x, v[k].y), bf16x2_max(v[k].z, v[k].w));
    uint32_t a = vm[0];
#pragma unroll
    for (int k = 1; k < kBatchVecs; ++k) a = bf16x2_max(a, vm[k]);
    return fmaxf(bf16_lo(a), bf16_hi(a));
}

// Fold one batch into the lane's running (m, s, kb): kb is the chunk batch
// holding the lane's first element equal to m.  A lane visits its batches
// in increasing position, so only a strictly larger maximum moves kb.
__device__ __forceinline__ void fold_batch(const uint4 (&v)[kBatchVecs], int kbatch, float& m, float& s, int& kb) {
    uint32_t vm[kBatchVecs];
    const float bm = batch_max(v, vm);
    if (bm > m) {
        s *= ex2_approx((m - bm) * kLog2e);
        m = bm;
        kb = kbatch;
    }
    if (m == -INFINITY) return;   // nothing finite seen yet: the batch adds 0
    const float nb = -m * kLog2e;
#if DLLM_STEP_F32X2
    // Two elements per instruction: (lo, hi) of a bf16 pair as an f32x2,
    // one packed FMA for the exponent arguments, two ex2, one packed add.
    // Per lane the accumulators, their order and every rounding are those
    // of the scalar loop below (a0 and a1 share one pair, a2 and a3 the
    // other), so the two loops give bit-identical sums.
    const unsigned long long s2 = f32x2_splat(kLog2e), n2 = f32x2_splat(nb);
    unsigned long long p01 = 0ull, p23 = 0ull;
#pragma unroll
    for (int k = 0; k < kBatchVecs; ++k) {
        acc_exp2_bf16x2(p01, v[k].x, s2, n2);
        acc_exp2_bf16x2(p23, v[k].y, s2, n2);
        acc_exp2_bf16x2(p01, v[k].z, s2, n2);
        acc_exp2_bf16x2(p23, v[k].w, s2, n2);
    }
    const float a0 = __uint_as_float((uint32_t)p01), a1 = __uint_as_float((uint32_t)(p01 >> 32));
    const float a2 = __uint_as_float((uint32_t)p23), a3 = __uint_as_float((uint32_t)(p23 >> 32));
#else
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int k = 0; k < kBatchVecs; ++k) {
        a0 += ex2_approx(fmaf(bf16_lo(v[k].x), kLog2e, nb));
        a1 += ex2_approx(fmaf(bf16_hi(v[k].x), kLog2e, nb));
        a2 += ex2_approx(fmaf(bf16_lo(v[k].y), kLog2e, nb));
        a3 += ex2_approx(fmaf(bf16_hi(v[k].y), kLog2e, nb));
        a0 += ex2_approx(fmaf(bf16_lo(v[k].z), kLog2e, nb));
        a1 += ex2_approx(fmaf(bf16_hi(v[k].z), kLog2e, nb));
        a2 += ex2_approx(fmaf(bf16_lo(v[k].w), kLog2e, nb));
        a3 += ex2_approx(fmaf(bf16_hi(v[k].w), kLog2e, nb));
    }
#endif
    s += (a0 + a1) + (a2 + a3);
}

// Replace the elements of a bf16 pair that lie beyond the row by -inf.
// `valid`: how many of the pair's two elements are inside the row.
__device__ __forceinline__ uint32_t mask_word(uint32_t w, int valid) {
    if (valid <= 0) return 0xff80ff80u;
    if (valid == 1) return (w & 0x0000ffffu) | 0xff800000u;
    return w;
}

// One copy (up to kCopyElems elements) from shared memory; q is the copy's
// index inside its chunk.
template <bool kFull>
__device__ __forceinline__ void process_copy(const uint4* buf, int lane, int q, int nel, float& m, float& s,
                                             int& kb) {
#pragma unroll
    for (int h = 0; h < kBatchesPerCopy; ++h) {
        uint4 v[kBatchVecs];
#pragma unroll
        for (int k = 0; k < kBatchVecs; ++k) {
            const int vi = lane + 32 * (h * kBatchVecs + k);
            if (kFull) {
                v[k] = buf[vi];
            } else {
                const int valid = nel - vi * 8;   // elements of this vector inside the copy
                if (valid >= 8) {
                    v[k] = buf[vi];
                } else if (valid <= 0) {
                    v[k] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
                } else {
                    uint4 t = buf[vi];
                    t.x = mask_word(t.x, valid);
                    t.y = mask_word(t.y, valid - 2);
                    t.z = mask_word(t.z, valid - 4);
                    t.w = mask_word(t.w, valid - 6);
                    v[k] = t;
                }
            }
        }
        fold_batch(v, q * kBatchesPerCopy + h, m, s, kb);
    }
}

// Combine two (max, sum) pairs; exact when one side is empty (-inf, 0).
__device__ __forceinline__ void combine(float& m, float& s, float mo, float so) {
    const float mn = fmaxf(m, mo);
    const float a = (m == mn) ? s : s * ex2_approx((m - mn) * kLog2e);
    const float b = (mo == mn) ? so : so * ex2_approx((mo - mn) * kLog2e);
    s = a + b;
    m = mn;
}

// ---------------------------------------------------------------------------
// Features of one block (warp-cooperative), DiLaServe review section 4.2 ③.
// val[k] / inU[k] describe position j = lane + 32 k (k < NK, j < L).
// Writes feats[0..5].  NK is a compile-time bound so that every array
// index is a constant and the arrays stay in registers.
// ---------------------------------------------------------------------------
// Order-preserving 32-bit image of a float (for sorting): negative values
// have every bit flipped, non-negative ones only the sign bit.
__device__ __forceinline__ uint32_t float_order_key(float v) {
    const uint32_t b = __float_as_uint(v + 0.0f);   // -0 sorts as +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float float_from_order_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Features of a block of at most 32 positions (one per lane): the unmasked
// values are sorted by a 32-lane bitonic network on their order-preserving
// bits -- positions outside U carry the largest key and sort last -- and the
// order statistics are read from their lanes.  Equal values are
// interchangeable, so no tie-break is needed; the results are those of the
// general rank count below.
__device__ __forceinline__ void warp_features_32(float val, bool inU, int L, int lane, float* feats_out) {
    const int n = __reduce_add_sync(0xffffffffu, inU ? 1u : 0u);
    float sum = inU ? val : 0.f;
#pragma unroll
    for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    float f[6];
    if (n == 0) {
        f[0] = f[1] = f[2] = f[3] = f[4] = __int_as_float(0x7fc00000);
        f[5] = 0.f;
    } else {
        uint32_t key = inU ? float_order_key(val) : 0xffffffffu;
#pragma unroll
        for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
            for (int j = k >> 1; j > 0; j >>= 1) {
                const uint32_t other = __shfl_xor_sync(0xffffffffu, key, j);
                const bool take_min = ((lane & k) == 0) == ((lane & j) == 0);
                key = take_min ? min(other, key) : max(other, key);
            }
        }
        const uint32_t hi = key;   // lane r: the r-th smallest value of U
        const float qs[3] = {0.25f, 0.5f, 0.75f};
        float lo_v[3], hi_v[3], frac[3];
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            const float h = qs[t] * float(n - 1);
            const int lo = int(floorf(h));
            frac[t] = h - float(lo);
            lo_v[t] = float_from_order_key(__shfl_sync(0xffffffffu, hi, lo));
            hi_v[t] = float_from_order_key(__shfl_sync(0xffffffffu, hi, min(lo + 1, n - 1)));
        }
        f[0] = float_from_order_key(__shfl_sync(0xffffffffu, hi, 0));
        f[1] = lo_v[0] + frac[0] * (hi_v[0] - lo_v[0]);
        f[2] = lo_v[1] + frac[1] * (hi_v[1] - lo_v[1]);
        f[3] = sum / float(n);
        f[4] = lo_v[2] + frac[2] * (hi_v[2] - lo_v[2]);
        f[5] = float(n) / float(L);
    }
    if (lane < 6) feats_out[lane] = f[lane];
}

template <int NK>
__device__ __forceinline__ void warp_features(const float (&val)[NK], const bool (&inU)[NK], int L, int lane,
                                              float* feats_out) {
    if constexpr (NK == 1) {
        warp_features_32(val[0], inU[0], L, lane, feats_out);
        return;
    }
    int n = 0;
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        if (inU[k]) {
            ++n;
            sum += val[k];
        }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        n += __shfl_xor_sync(0xffffffffu, n, off);
        sum += __shfl_xor_sync(0xffffffffu, sum, off);
    }
    float f[6];
    if (n == 0) {
        f[0] = f[1] = f[2] = f[3] = f[4] = __int_as_float(0x7fc00000);
        f[5] = 0.f;
    } else {
        // rank of each of my values among U (ties broken by position); the
        // update is branch-free so the shuffles of successive sources
        // overlap instead of waiting one by one
        int rank[NK];
#pragma unroll
        for (int k = 0; k < NK; ++k) rank[k] = 0;
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
#pragma unroll (NK == 1 ? 32 : 4)
            for (int src = 0; src < 32; ++src) {
                const int jj = src + 32 * kk;
                const float vo = __shfl_sync(0xffffffffu, val[kk], src);
                const bool uo = (__shfl_sync(0xffffffffu, inU[kk] ? 1 : 0, src) != 0) && jj < L;
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    const int j = lane + 32 * k;
                    rank[k] += (uo && inU[k] && (vo < val[k] || (vo == val[k] && jj < j))) ? 1 : 0;
                }
            }
        }
        // order statistics needed: rank 0 and lo / hi of the three quantiles
        const float qs[3] = {0.25f, 0.5f, 0.75f};
        int want[7];
        float frac[3];
        want[0] = 0;
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            const float h = qs[t] * float(n - 1);
            const int lo = int(floorf(h));
            frac[t] = h - float(lo);
            want[1 + 2 * t] = lo;
            want[2 + 2 * t] = min(lo + 1, n - 1);
        }
        float got[7];
#pragma unroll
        for (int t = 0; t < 7; ++t) {
            float mine = 0.f;
            bool have = false;
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                if (inU[k] && rank[k] == want[t]) {
                    mine = val[k];
                    have = true;
                }
            }
            const unsigned bal = __ballot_sync(0xffffffffu, have);
            got[t] = __shfl_sync(0xffffffffu, mine, __ffs(bal) - 1);
        }
        f[0] = got[0];
        f[1] = got[1] + frac[0] * (got[2] - got[1]);
        f[2] = got[3] + frac[1] * (got[4] - got[3]);
        f[3] = sum / float(n);
        f[4] = got[5] + frac[2] * (got[6] - got[5]);
        f[5] = float(n) / float(L);
    }
    if (lane < 6) feats_out[lane] = f[lane];
}

// ---------------------------------------------------------------------------
// S3-S6 for request b (one warp), for L <= 32 * NK.  has_masked: b had masked
// rows at entry (then every one of them has its row results in the
// workspace).
// ---------------------------------------------------------------------------
// Set once a warp of this CTA has seen every CTA's scan signal (with a
// gpu-scope acquire); later finalisations in the CTA read it with a CTA-scope
// acquire instead, which does not hold back their stores.
__shared__ int s_all_scanned;

template <int NK>
__device__ __noinline__ void finalize_request_t(const StepParams& P, int b, bool has_masked, int lane, bool direct) {
    // Row results arrive as zero-at-rest words (polled until they land);
    // requests without masked rows read only the launch's inputs.
    const int L = P.L;
    const long long base = (long long)b * L;
    const float t = P.quota ? 0.f : P.thr[b];
    const int q = P.quota ? P.quota[b] : 0;

    int id[NK], tk[NK];
    float c[NK], cs_old[NK];
    unsigned long long rw[NK];
    bool msk[NK];
    bool any_masked = false, any_pass = false;
    float best_c = -INFINITY;
    int best_j = 0x7fffffff;
    // issue every load of the block first, then decide
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        const int j = lane + 32 * k;
        const bool valid = j < L;
        id[k] = valid ? P.ids[base + j] : 0;
        cs_old[k] = valid ? P.cs[base + j] : 0.f;
        rw[k] = (valid && has_masked) ? ld_relaxed_gpu_u64(P.row_word + base + j) : 0ull;
    }
    // the row's commit state (fused commit): issued with the block's loads
    int c_blk = 0, c_K = 0, c_r = 0;
    if (P.commit) {
        c_blk = P.c_b[b];
        c_K = P.c_K[b];
        c_r = P.c_rid[b];
    }
    // the scan count guards only the commit at the end: loaded after the
    // block's loads so that its acquire does not hold them back, and only
    // until the CTA has seen it complete
    int scanned = 0;
    if (lane == 0 && (has_masked || P.commit) && !direct) {
        if (ld_acquire_cta_shared(&s_all_scanned)) {
            scanned = (int)gridDim.x;
        } else {
            scanned = ld_acquire_gpu(P.ctl);
            if (scanned == (int)gridDim.x) st_release_cta_shared(&s_all_scanned, 1);
        }
    }
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        const int j = lane + 32 * k;
        msk[k] = j < L && id[k] == P.mask_id;
        c[k] = 0.f;
        tk[k] = -1;
        if (msk[k]) {
            if (rw[k] == 0ull) rw[k] = poll_word(P.row_word + base + j, P.err);
            P.row_word[base + j] = 0ull;
            unpack_row(rw[k], c[k], tk[k]);
            any_masked = true;
            if (c[k] > t) any_pass = true;
            // j grows with k, so a strict > keeps the lowest position on ties
            if (best_j == 0x7fffffff || c[k] > best_c) {
                best_c = c[k];
                best_j = j;
            }
        } else {
            c[k] = 0.f;
            tk[k] = -1;
        }
    }
    any_masked = __any_sync(0xffffffffu, any_masked);
    any_pass = __any_sync(0xffffffffu, any_pass);
    int fb_j = -1;
    if (!P.quota && any_masked && !any_pass) {
        // most confident masked position, lowest position on ties
        float bc = best_c;
        int bj = best_j;
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const float oc = __shfl_xor_sync(0xffffffffu, bc, off);
            const int oj = __shfl_xor_sync(0xffffffffu, bj, off);
            if (oj != 0x7fffffff && (bj == 0x7fffffff || oc > bc || (oc == bc && oj < bj))) {
                bc = oc;
                bj = oj;
            }
        }
        fb_j = bj;
    }

    // fixed-steps rule: a masked position is taken when fewer than q masked
    // positions beat it (higher confidence, or equal and lower position)
    int qrank[NK];
#pragma unroll
    for (int k = 0; k < NK; ++k) qrank[k] = 0;
    if (P.quota) {
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
#pragma unroll (NK == 1 ? 32 : 4)
            for (int src = 0; src < 32; ++src) {
                const int jj = src + 32 * kk;
                const float co = __shfl_sync(0xffffffffu, c[kk], src);
                const bool mo = __shfl_sync(0xffffffffu, msk[kk] ? 1 : 0, src) != 0;
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    const int j = lane + 32 * k;
                    qrank[k] += (mo && msk[k] && (co > c[k] || (co == c[k] && jj < j))) ? 1 : 0;
                }
            }
        }
    }

    float val[NK];
    bool inU[NK];
    bool selk[NK];
    int n_sel = 0;
    bool still = false;
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        const int j = lane + 32 * k;
        const bool valid = j < L;
        const bool s = msk[k] && (P.quota ? qrank[k] < q : (c[k] > t || j == fb_j));
        selk[k] = s;
        const int new_id = s ? tk[k] : id[k];
        float new_cs = 0.f;
        if (valid) {
            new_cs = s ? c[k] : cs_old[k];
            if (s) P.cs[base + j] = c[k];
            if (has_masked) P.sel[base + j] = s ? 1 : 0;
            if (!msk[k]) {
                if (P.conf_out) P.conf_out[base + j] = __int_as_float(0x7fc00000);
                if (P.lse_out) P.lse_out[base + j] = __int_as_float(0x7fc00000);
                if (P.tok_out) P.tok_out[base + j] = -1;
            }
        }
        n_sel += s ? 1 : 0;
        still |= valid && new_id == P.mask_id;
        inU[k] = valid && new_id != P.mask_id;
        val[k] = new_cs;
        id[k] = new_id;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) n_sel += __shfl_xor_sync(0xffffffffu, n_sel, off);
    const bool done = !__any_sync(0xffffffffu, still);
    if (lane == 0) {
        P.done[b] = done ? 1 : 0;
        P.accept[b] = done ? L : 0;
        P.n_new[b] = n_sel;
    }
    if (P.feats) warp_features<NK>(val, inU, L, lane, P.feats + (long long)b * DLLM_NUM_FEATURES);

    // Fused commit (dllm_step_commit): a finished block joins the request's
    // committed tokens and the request moves to its next block, which
    // starts fully masked, or leaves the batch after its last one (FDFO
    // page, section "FDFO 的核心思想": a finished request commits at once;
    // BlockServe page, Algorithm 1: b_i <- b_i + 1, evict when b_i >= K_i).
    // Exactly dllm_advance with the step's done flags as its advance flags.
    bool reset = false;
    if (P.commit) {
        bool ev = false;
        if (done) {
            if (c_blk < 0 || c_blk >= c_K || (long long)(c_blk + 1) * L > P.c_ld_gen) {
                if (lane == 0) set_error(P.err, DLLM_DEVERR_BLOCK_INDEX);
            } else {
                int* g = P.c_gen + (long long)c_r * P.c_ld_gen + (long long)c_blk * L;
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    const int j = lane + 32 * k;
                    if (j < L) g[j] = id[k];
                }
                ev = c_blk + 1 >= c_K;
                reset = !ev;
                if (lane == 0) P.c_b[b] = c_blk + 1;
            }
        }
        if (lane == 0) P.c_evict[b] = ev ? 1 : 0;
        if (reset) {
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                const int j = lane + 32 * k;
                if (j < L) P.cs[base + j] = __int_as_float(0x7fc00000);
            }
        }
    }

    // S4 commit of input_ids: only once every CTA has finished its scan;
    // before that the request goes on the deferred list, which the grid's
    // last CTA commits (the add's high half counts the list's entries).
    if (!has_masked && !reset) return;
    __syncwarp();   // lane 0's acquire of the scan count orders the warp's writes
    if (direct || __shfl_sync(0xffffffffu, scanned, 0) == (int)gridDim.x) {
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const int j = lane + 32 * k;
            if (reset) {
                if (j < L) P.ids[base + j] = P.mask_id;
            } else if (selk[k]) {
                P.ids[base + j] = id[k];
            }
        }
    } else if (lane == 0) {
        const int slot = (int)((unsigned)atomicAdd(P.ctl + 1, 1 << 16) >> 16);
        P.cnt[P.BL + P.B + slot] = b | (reset ? kDeferReset : 0);
    }
    if (lane == 0 && has_masked) P.cnt[P.BL + b] = 0;   // request counter back to rest
}

// direct: input_ids may be written at once (no other CTA still scans them).
__device__ __forceinline__ void finalize_request(const StepParams& P, int b, bool has_masked, int lane,
                                                 bool direct = false) {
    const int nk = (P.L + 31) >> 5;
    if (nk <= 1) finalize_request_t<1>(P, b, has_masked, lane, direct);
    else if (nk <= 2) finalize_request_t<2>(P, b, has_masked, lane, direct);
    else if (nk <= 4) finalize_request_t<4>(P, b, has_masked, lane, direct);
    else finalize_request_t<32>(P, b, has_masked, lane, direct);
}

// ---------------------------------------------------------------------------
// The fold of a row's chunk partials [c0, c1) (a whole row, or one
// vocabulary shard of it): each lane folds chunks c0 + lane, c0 + lane + 32,
// ... in order, then the lanes combine in a fixed butterfly; the order
// depends only on c1 - c0.  key: (chunk - c0) * batches + batch of the first
// maximum, or INT64_MAX when no chunk holds a finite value.  Each word is
// cleared once read, ready for the next call.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fold_row_chunks(const StepParams& P, int row, int c0, int c1, int lane, float& M,
                                                float& S, long long& key) {
    M = -INFINITY;
    S = 0.f;
    key = 0x7fffffffffffffffLL;
    for (int c = c0 + lane; c < c1; c += 32) {
        unsigned long long* wp = P.part + (long long)row * P.NC + c;
        unsigned long long w = ld_relaxed_gpu_u64(wp);
        if (w == 0ull) w = poll_word(wp, P.err);
        *wp = 0ull;
        float pm, ps;
        int pk;
        unpack_partial(w, pm, ps, pk);
        const long long kc = (long long)(c - c0) * kBatchesPerChunk + min(max(pk, 0), kBatchesPerChunk - 1);
        if (pm > M) key = kc;
        combine(M, S, pm, ps);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, M, off);
        const float so = __shfl_xor_sync(0xffffffffu, S, off);
        const long long ko = __shfl_xor_sync(0xffffffffu, key, off);
        if (mo > M || (mo == M && ko < key)) key = ko;
        combine(M, S, mo, so);
    }
}

// The argmax: the first element equal to M inside the 2048-element batch
// `key` of the row at rp (Vr elements); each lane loads all of its vectors
// at once, then scans them in order.  0xffffffff when there is none (no
// finite maximum: nothing is read).
__device__ __forceinline__ unsigned first_max_in_batch_at(const uint16_t* rp, int Vr, long long key, float M,
                                                          int lane) {
    if (key == 0x7fffffffffffffffLL) return 0xffffffffu;
    const long long start = key * kBatchElems;
    uint4 v[kBatchVecs];
#pragma unroll
    for (int k = 0; k < kBatchVecs; ++k) {
        const long long e = start + (long long)(lane + 32 * k) * 8;
        v[k] = (e < Vr) ? __ldg(reinterpret_cast<const uint4*>(rp + e))
                        : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    }
    unsigned best = 0xffffffffu;
#pragma unroll
    for (int k = kBatchVecs - 1; k >= 0; --k) {
        const long long e = start + (long long)(lane + 32 * k) * 8;
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int h = 7; h >= 0; --h) {
            const float x = (h & 1) ? bf16_hi(w[h >> 1]) : bf16_lo(w[h >> 1]);
            if (e + h < Vr && x == M) best = (unsigned)(e + h);
        }
    }
    return __reduce_min_sync(0xffffffffu, best);
}

// ---------------------------------------------------------------------------
// Row finisher: fold the chunk partials of `row` in a fixed order, write the
// row results, then count the row towards its request.
// ---------------------------------------------------------------------------
__device__ __noinline__ void finish_row(const StepParams& P, const uint16_t* s_gmask, int row, int lrow, int lane) {
    // Every chunk of the row has been counted, but the words holding the
    // partials are written with relaxed stores: a word still reading zero
    // is polled (bounded in time) until its store lands.  Each word is
    // cleared once read, ready for the next call.
    const int NC = P.NC;
    const int b = row / P.L;
    // Claim the row on its request's counter first: the add's round trip
    // overlaps the fold and the argmax re-read.  The request's last claimer
    // finalises it, polling for the words of rows other warps are still
    // finishing.
    int old = 0;
    if (lane == 0 && !P.shard) old = atom_add_relaxed_gpu(P.cnt + P.BL + b, 1);
    // masked rows of this request at entry, from this CTA's scan bitmask
    int mb = 0;
    {
        const int p0 = b * P.L, p1 = p0 + P.L;
        for (int g = (p0 >> 4) + lane; g <= ((p1 - 1) >> 4); g += 32) {
            unsigned bits = s_gmask[g];
            const int lo = max(p0 - (g << 4), 0), hi = min(p1 - (g << 4), 16);
            bits &= ((hi >= 16) ? 0xffffu : ((1u << hi) - 1u)) & ~((1u << lo) - 1u);
            mb += __popc(bits);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) mb += __shfl_xor_sync(0xffffffffu, mb, off);
    }
    float M, S;
    long long key;
    const uint16_t* rp;
    int Vr, v0 = 0;
    if (P.n_shards == 0) {
        fold_row_chunks(P, row, 0, NC, lane, M, S, key);
        rp = P.logits + (long long)lrow * P.ldv;
        Vr = P.V;
    } else {
        // each shard folded as a launch over that shard alone folds it, then
        // the shards merged in order as dllm_step_merge merges their triples:
        // the token comes from the first shard attaining the maximum
        M = -INFINITY;
        S = 0.f;
        key = 0x7fffffffffffffffLL;
        int ks = -1;
        for (int k = 0; k < P.n_shards; ++k) {
            float mk, sk;
            long long kk;
            fold_row_chunks(P, row, P.sh_c0[k], P.sh_c0[k + 1], lane, mk, sk, kk);
            if (mk > M || ks < 0) {
                ks = k;
                key = kk;
            }
            combine(M, S, mk, sk);
        }
        rp = P.sh_logits[ks] + (long long)lrow * P.sh_ldv[ks];
        Vr = P.sh_V[ks];
        v0 = P.sh_v0[ks];
    }
    const unsigned best0 = first_max_in_batch_at(rp, Vr, key, M, lane);
    const unsigned best = (best0 == 0xffffffffu || P.n_shards == 0) ? best0 : best0 + (unsigned)v0;
    const float conf = __fdiv_rn(1.0f, S);
    const float lse = M + logf(S);
    if (P.shard) {   // S2 of a vocabulary shard: the row's triple, nothing else
        if (lane == 0) {
            P.trip_m[row] = M;
            P.trip_s[row] = S;
            P.trip_i[row] = best == 0xffffffffu ? -1 : (int)best + P.v0;
            P.cnt[row] = 0;
        }
        return;
    }
    // publish the row's word (relaxed: the request's finalizer polls)
    if (lane == 0) {
        P.row_tok[row] = (int)best;
        if (P.conf_out) P.conf_out[row] = conf;
        if (P.lse_out) P.lse_out[row] = lse;
        if (P.tok_out) P.tok_out[row] = (int)best;
        P.cnt[row] = 0;
        st_relaxed_gpu_u64(P.row_word + row, pack_row(conf, (int)best));
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == mb - 1) {
        __syncwarp();   // lane 0's word store is ordered before the other lanes' loads
        finalize_request(P, b, true, lane);
    }
}

// ---------------------------------------------------------------------------
// Finish queue: rows this CTA completed, drained in order by the finisher
// warps and, once they are done streaming, by the streaming warps too.  A warp claims
// the next slot, waits for it to be filled, and stops once every streaming
// warp is done and its slot stayed empty.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void drain_queue(const StepParams& P, const uint16_t* s_gmask, int* s_queue, int* s_qhead,
                                            const int* s_ndone, int lane) {
    uint32_t idle = 0;
    uint64_t t0 = globaltimer_ns();
    int h = (lane == 0) ? atomicAdd(s_qhead, 1) : 0;
    h = __shfl_sync(0xffffffffu, h, 0);
    while (h < P.list_cap) {
        int v = (lane == 0) ? ld_acquire_cta_shared(&s_queue[2 * h]) : 0;
        v = __shfl_sync(0xffffffffu, v, 0);
        if (v != 0) {
            __syncwarp();   // lane 0's acquire orders the whole warp's reads
            finish_row(P, s_gmask, v - 1, s_queue[2 * h + 1], lane);
            t0 = globaltimer_ns();   // the limit bounds idle waiting, not work
            h = (lane == 0) ? atomicAdd(s_qhead, 1) : 0;
            h = __shfl_sync(0xffffffffu, h, 0);
            continue;
        }
        int nd = (lane == 0) ? ld_acquire_cta_shared(s_ndone) : 0;
        nd = __shfl_sync(0xffffffffu, nd, 0);
        if (nd == kStreamWarps) {
            // every completed row is queued: slot h is filled now or never
            int v2 = (lane == 0) ? ld_acquire_cta_shared(&s_queue[2 * h]) : 0;
            if (__shfl_sync(0xffffffffu, v2, 0) != 0) continue;
            break;
        }
        __nanosleep(DLLM_STEP_IDLE_NS);
        if ((++idle & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            if (lane == 0) set_error(P.err, DLLM_DEVERR_TIMEOUT);
            break;
        }
    }
}

// ---------------------------------------------------------------------------
// A CTA's pool of n units (chunks u_first .. u_first + n - 1) in groups: up to
// kGroup consecutive chunks of one row, except the last `single` units, which
// go one at a time so that the warps finish together.  Groups are numbered in
// unit order, so a warp takes the next group with one fetch-and-add on a
// counter (a compare-and-swap loop over units costs every warp a round trip
// per lost race, and all of a CTA's warps start their first grab together).
// ---------------------------------------------------------------------------
struct PoolGroups {
    int n, z;       // pool size; units [0, z) go in groups of up to kGroup
    int a0, ga0;    // units in [0, z) of the first row, and their groups
    int f, gpr;     // whole rows after it in [0, z), groups per whole row
    int p, gp;      // units of the last row in [0, z), and their groups
};

__device__ __forceinline__ PoolGroups make_pool_groups(int u_first, int n, int NC, const FastDiv& div_nc,
                                                       int single) {
    PoolGroups q;
    q.n = n;
    q.z = max(0, n - single);
    const int lead = (fast_div(u_first, div_nc) + 1) * NC - u_first;   // units up to the first row's end
    q.a0 = min(q.z, lead);
    q.ga0 = (q.a0 + kGroup - 1) / kGroup;
    q.gpr = (NC + kGroup - 1) / kGroup;
    q.f = (q.z - q.a0) / NC;
    q.p = q.z - q.a0 - q.f * NC;
    q.gp = (q.p + kGroup - 1) / kGroup;
    return q;
}

// Group g of the pool: its first unit (relative to u_first) and size, or -1.
__device__ __forceinline__ int pool_group(const PoolGroups& q, int g, int NC, int& size) {
    if (g < q.ga0) {
        size = min(kGroup, q.a0 - g * kGroup);
        return g * kGroup;
    }
    g -= q.ga0;
    if (g < q.f * q.gpr) {
        const int r = g / q.gpr, j = g - r * q.gpr;
        size = min(kGroup, NC - j * kGroup);
        return q.a0 + r * NC + j * kGroup;
    }
    g -= q.f * q.gpr;
    if (g < q.gp) {
        size = min(kGroup, q.p - g * kGroup);
        return q.a0 + q.f * NC + g * kGroup;
    }
    g -= q.gp;
    if (g < q.n - q.z) {
        size = 1;
        return q.z + g;
    }
    size = 0;
    return -1;
}

// ---------------------------------------------------------------------------
// The step kernel: kStreamWarps streaming warps and kFinishWarps finisher
// warps per CTA.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepParams P) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(kStreamWarps) * kStages * kCopyBytes);
    int* s_list = reinterpret_cast<int*>(bars + kStreamWarps * kStages);
    int* s_queue = s_list + P.list_cap;   // rows this CTA completed: (position + 1, logits row) pairs
    int* s_zero = s_queue + 2 * P.list_cap;   // this CTA's requests without masked rows
    uint16_t* s_gmask = reinterpret_cast<uint16_t*>(s_zero + P.zero_cap);   // masked bits, 16 positions each
    __shared__ int s_wsum[kWarpsTotal];
    __shared__ int s_nzero, s_qtail, s_qhead, s_ndone, s_last, s_next, s_ring_busy;
    // The row finishers, request finalisation and the exit read many launch
    // parameters once each, late in the launch, when the constant cache no
    // longer holds them: they read this copy instead.
    __shared__ __align__(16) StepParams s_P;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, cta = blockIdx.x;
    static_assert(sizeof(StepParams) % 4 == 0, "copied as words");
    for (int i = tid; i < (int)(sizeof(StepParams) / 4); i += kThreads)
        reinterpret_cast<int*>(&s_P)[i] = reinterpret_cast<const int*>(&P)[i];
    const StepParams& FP = s_P;

    if (tid < kStreamWarps * kStages) mbar_init(smem_addr(&bars[tid]), 1);
    if (tid == 0) {
        s_all_scanned = 0;
        s_next = 0;
        s_ring_busy = 0;
        s_nzero = 0;
        s_qtail = 0;
        s_qhead = 0;
        s_ndone = 0;
    }
    for (int i = tid; i < 2 * P.list_cap; i += kThreads) s_queue[i] = 0;
    if (tid < kStreamWarps * kStages) mbar_fence_init();
    // everything above touches shared memory only; the previous kernel's
    // writes (input_ids, logits, state) are read from here on
    pdl_wait();
    pdl_release();

    // ---- S1: masked bits of the entry state, 16 positions per thread ------
    const int BL = P.BL;
    const int ngroups = (BL + 15) >> 4;
    const bool ids_vec = (reinterpret_cast<uintptr_t>(P.ids) & 15u) == 0;
    for (int g = tid; g < ngroups; g += kThreads) {
        const int p0 = g << 4;
        unsigned bits = 0;
        if (ids_vec && p0 + 16 <= BL) {
            const int4* q = reinterpret_cast<const int4*>(P.ids + p0);
            const int4 a0 = q[0], a1 = q[1], a2 = q[2], a3 = q[3];
            const int v[16] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w,
                               a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
#pragma unroll
            for (int i = 0; i < 16; ++i) bits |= (v[i] == P.mask_id ? 1u : 0u) << i;
        } else {
            for (int i = 0; i < 16; ++i)
                if (p0 + i < BL && P.ids[p0 + i] == P.mask_id) bits |= 1u << i;
        }
        s_gmask[g] = (uint16_t)bits;
    }
    __syncthreads();
    // ranks: each thread owns a contiguous run of groups; block-wide scan
    const int gper = (ngroups + kThreads - 1) / kThreads;
    const int g0 = min(ngroups, tid * gper), g1 = min(ngroups, g0 + gper);
    int cnt = 0;
    for (int g = g0; g < g1; ++g) cnt += __popc((unsigned)s_gmask[g]);
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int wbase = 0, M = 0;
#pragma unroll
    for (int w = 0; w < kWarpsTotal; ++w) {
        const int cw = s_wsum[w];
        if (w < warp) wbase += cw;
        M += cw;
    }
    const int before = wbase + incl - cnt;
    const int NC = P.NC;
    const int V = P.V;
    if (P.compact && M > P.logits_rows) {
        // a compact logits array too short for the batch: nothing is read
        if (tid == 0 && cta == 0) set_error(P.err, DLLM_DEVERR_LOGITS_ROWS);
        M = 0;
    }
    const int U = M * NC;   // units fit in 32 bits (checked on the host)
    // The last T = min(ceil(M / kTailDen), kTailRowsMax) masked rows (the
    // tail) are taken one chunk at a time by any warp whose CTA has run out,
    // so that CTAs the memory system serves more slowly do not hold up the
    // end of the step; the rows before them are split evenly over the CTAs.
    // With Ms = M - T, CTA k's share starts at element floor(Ms V k / G) =
    // V a + e with a = floor(Ms k / G) and e = floor(V (Ms k mod G) / G) < V:
    // row a, element e of that row.  Its first unit is the first chunk
    // starting there or later; k = G gives the tail's first unit Ms * NC.
    // Only 32-bit divisions (M G and V G fit in 32 bits, checked on the host).
    const int T = min((M + kTailDen - 1) / kTailDen, kTailRowsMax);
    const int Ms = M - T;
    auto first_unit = [&](int k) -> int {
        const int mk = Ms * k;
        int r = fast_div(mk, P.div_g);
        const int e = fast_div(V * (mk - r * G), P.div_g);
        // the first chunk starting at or after element e of the row (shard
        // by shard when the row is split into vocabulary shards)
        int cc;
        if (P.n_shards == 0) {
            cc = (e + kChunkElems - 1) / kChunkElems;
        } else {
            int k = 0;
            for (int i = 1; i < P.n_shards; ++i)
                if (e >= P.sh_v0[i]) k = i;
            cc = P.sh_c0[k] + (e - P.sh_v0[k] + kChunkElems - 1) / kChunkElems;
        }
        if (cc >= NC) {
            r += 1;
            cc = 0;
        }
        return r * NC + cc;
    };
    const int u0 = first_unit(cta);
    const int u1 = first_unit(cta + 1);
    const int u_tail = Ms * NC;
    const int n_tail = U - u_tail;
    const int r_lo = fast_div(u0, P.div_nc);
    const int r_hi = (u1 > u0) ? fast_div(u1 - 1, P.div_nc) : r_lo - 1;
    const int r_tail = Ms;   // first row of the tail
    const int r_last = (n_tail > 0) ? M - 1 : r_hi;
    const int static_cap = P.static_cap;
    // each set bit's rank is independent of the others: before the group's
    // first rank plus the set bits below it in the group
    int rank0 = before;
    for (int g = g0; g < g1 && rank0 <= r_last; ++g) {
        const unsigned bits = s_gmask[g];
        const int c = __popc(bits);
        if ((rank0 <= r_hi && rank0 + c > r_lo) || rank0 + c > r_tail) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if ((bits >> i) & 1u) {
                    const int rank = rank0 + __popc(bits & ((1u << i) - 1u));
                    if (rank >= r_lo && rank <= r_hi) s_list[rank - r_lo] = (g << 4) + i;
                    if (rank >= r_tail) s_list[static_cap + rank - r_tail] = (g << 4) + i;
                }
            }
        }
        rank0 += c;
    }
    // this CTA's requests (b = cta + G*k) without a masked position
    for (long long k = tid; cta + (long long)G * k < P.B; k += kThreads) {
        const int b = cta + G * (int)k;
        const int p0 = b * P.L, p1 = p0 + P.L;
        bool anym = false;
        for (int g = p0 >> 4; g <= ((p1 - 1) >> 4) && !anym; ++g) {
            unsigned bits = s_gmask[g];
            const int lo = max(p0 - (g << 4), 0), hi = min(p1 - (g << 4), 16);
            bits &= ((hi >= 16) ? 0xffffu : ((1u << hi) - 1u)) & ~((1u << lo) - 1u);
            anym = bits != 0;
        }
        if (!anym) s_zero[atomicAdd(&s_nzero, 1)] = b;
    }
    __syncthreads();

    const int n_units = u1 - u0;   // this CTA's chunks: unit k is chunk u0 + k
    const int u_first = u0;
    // masked position of unit gu's row (units of the tail have their own slots)
    auto row_of = [&](int gu) -> int {
        const int rr = fast_div(gu, P.div_nc);
        return (gu >= u_tail) ? s_list[static_cap + rr - r_tail] : s_list[rr - r_lo];
    };

    if (warp < kStreamWarps) {
        // ---- S2: stream groups of chunks through this warp's ring ----------
        // A group is up to kGroup consecutive chunks of one row, taken from
        // the CTA's pool (PoolGroups); near the end of the pool groups shrink
        // to one chunk so that the warps finish together.  Each chunk keeps its own
        // partial (the reduction order depends only on V); the group's
        // partials are reduced across the warp together and published with
        // one add on the row counter.
        const uint32_t stage0 = smem_addr(stages + size_t(warp) * kStages * kCopyBytes);
        const uint32_t bar0 = smem_addr(&bars[warp * kStages]);
        const uint64_t pol = l2_policy_evict_first();
        const int tail_units = 2 * kStreamWarps;   // single-chunk grabs below this many left
        const PoolGroups pool = make_pool_groups(u_first, n_units, NC, P.div_nc, tail_units);

        // Take the next group: returns its first unit (or -1) and its size.
        // Once the CTA's pool is spent, units come one at a time from the
        // shared tail through tickets on ctl[2].  Lane 0 draws its first
        // ticket while the CTA's pool is nearly spent, hiding that atomic's
        // latency; later tickets are drawn when needed (a ticket held ahead
        // is a chunk of work one warp still owes while others idle).
        int t_ahead = -1;   // lane 0: ticket drawn ahead of use
        auto grab = [&](int& k) -> int {
            int got = -1, kk = 0;
            if (lane == 0) {
                int want;
                const int st = pool_group(pool, atomicAdd(&s_next, 1), NC, want);
                if (st >= 0) {
                    got = u_first + st;
                    kk = want;
                    // the pool is nearly spent: draw the first tail ticket now
                    if (n_tail > 0 && t_ahead < 0 && st + want >= pool.z) t_ahead = atomicAdd(P.ctl + 2, 1);
                }
                if (got < 0 && n_tail > 0) {
                    const int t = (t_ahead >= 0) ? t_ahead : atomicAdd(P.ctl + 2, 1);
                    t_ahead = -1;
                    if (t < n_tail) {
                        got = u_tail + t;
                        kk = 1;
                    }
                }
            }
            k = __shfl_sync(0xffffffffu, kk, 0);
            return __shfl_sync(0xffffffffu, got, 0);
        };

        // producer side: the chunk being issued
        int p_unit = 0, p_left = 0, p_q = 0, p_len = 0;
        const uint16_t* p_src = nullptr;
        bool p_done = false;
        // groups whose copies are issued but not yet folded, oldest first
        int fifo_u[kStages + 1], fifo_k[kStages + 1];
        int nfifo = 0;
        uint32_t issued = 0, consumed = 0;
        bool failed = false;

        auto start_chunk = [&](int gu) {
            const int rr = fast_div(gu, P.div_nc);
            const int c = gu - rr * NC;
            const int lrow = P.compact ? rr : row_of(gu);   // compact logits are indexed by rank
            p_unit = gu;
            p_q = 0;
            const ChunkRef cr = chunk_ref(P, c);
            p_len = cr.len;
            p_src = cr.base + (long long)lrow * cr.ldv + cr.start;
        };
        auto issue = [&]() {
            if (p_done) return;
            if (p_q * kCopyElems >= p_len) {   // current chunk fully issued
                if (p_left > 0) {
                    --p_left;
                    start_chunk(p_unit + 1);
                } else {
                    int k = 0;
                    const int u = grab(k);
                    if (u < 0) {
                        p_done = true;
                        return;
                    }
#pragma unroll
                    for (int i = 0; i <= kStages; ++i)
                        if (i == nfifo) {
                            fifo_u[i] = u;
                            fifo_k[i] = k;
                        }
                    ++nfifo;
                    p_left = k - 1;
                    start_chunk(u);
                }
            }
            const int nel = min(kCopyElems, p_len - p_q * kCopyElems);
            const uint32_t bytes = (uint32_t)((nel * 2 + 15) & ~15);
            const int slot = issued % kStages;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar0 + slot * 8, bytes);
                bulk_g2s(stage0 + slot * kCopyBytes, p_src + (long long)p_q * kCopyElems, bytes,
                         bar0 + slot * 8, pol);
            }
            ++issued;
            ++p_q;
        };
        // Publishing a group: lane 1 writes each chunk's partial word with a
        // relaxed store and adds the group's chunk count to the row counter
        // with a relaxed add (no fence: a release here would wait for this
        // warp's memory traffic).  The add's result is tested one group
        // later; the add that brings the counter to NC queues the row for
        // the finishers, who poll for the words still in flight.
        int pend_old = -1, pend_k = 0, pend_row = 0, pend_lrow = 0;   // add issued, result not yet tested
        auto test_pending = [&]() {
            if (lane == 1 && pend_old >= 0 && pend_old + pend_k == NC) {
                const int q = atomicAdd(&s_qtail, 1);
                s_queue[2 * q + 1] = pend_lrow;
                st_release_cta_shared(&s_queue[2 * q], pend_row + 1);
            }
            pend_old = -1;
        };

#pragma unroll 1
        for (int st = 0; st < kStages; ++st) issue();

#pragma unroll 1
        while (consumed < issued && !failed) {
            const int gu = fifo_u[0], k = fifo_k[0];
#pragma unroll
            for (int i = 0; i < kStages; ++i) {
                fifo_u[i] = fifo_u[i + 1];
                fifo_k[i] = fifo_k[i + 1];
            }
            --nfifo;
            const int c0 = gu - fast_div(gu, P.div_nc) * NC;
            const int row = row_of(gu);
            float gm[kGroup], gs[kGroup];
            int gi[kGroup];
#pragma unroll
            for (int j = 0; j < kGroup; ++j) {
                gm[j] = -INFINITY;
                gs[j] = 0.f;
                gi[j] = kBatchesPerChunk;
            }
#pragma unroll 1
            for (int j = 0; j < k && !failed; ++j) {
                const int clen = chunk_ref(P, c0 + j).len;
                const int ncp = (clen + kCopyElems - 1) / kCopyElems;
                float m = -INFINITY, s = 0.f;
                int kb = kBatchesPerChunk;
#pragma unroll 1
                for (int q = 0; q < ncp; ++q) {
                    const int slot = consumed % kStages;
                    const uint32_t par = (consumed / kStages) & 1u;
                    if (!mbar_wait_bounded(bar0 + slot * 8, par, kWaitLimitNs)) {
                        failed = true;
                        break;
                    }
                    const int nel = min(kCopyElems, clen - q * kCopyElems);
                    const uint4* buf =
                        reinterpret_cast<const uint4*>(stages + (size_t(warp) * kStages + slot) * kCopyBytes);
                    if (nel == kCopyElems) process_copy<true>(buf, lane, q, nel, m, s, kb);
                    else process_copy<false>(buf, lane, q, nel, m, s, kb);
                    __syncwarp();
                    ++consumed;
                    issue();
                }
                // keep the chunk's partial in registers (constant indices only)
#pragma unroll
                for (int jj = 0; jj < kGroup; ++jj) {
                    if (jj == j) {
                        gm[jj] = m;
                        gs[jj] = s;
                        gi[jj] = kb;
                    }
                }
            }
            if (failed) break;
            // the group's warp reductions, interleaved
            float lm[kGroup];
#pragma unroll
            for (int j = 0; j < kGroup; ++j) lm[j] = gm[j];
#pragma unroll
            for (int off = 16; off; off >>= 1) {
#pragma unroll
                for (int j = 0; j < kGroup; ++j) {
                    const float mo = __shfl_xor_sync(0xffffffffu, gm[j], off);
                    const float so = __shfl_xor_sync(0xffffffffu, gs[j], off);
                    combine(gm[j], gs[j], mo, so);
                }
            }
            unsigned first[kGroup];
#pragma unroll
            for (int j = 0; j < kGroup; ++j)
                first[j] = __reduce_min_sync(0xffffffffu, (lm[j] == gm[j]) ? (unsigned)gi[j] : (unsigned)kBatchesPerChunk);
            // publish the group's partials (lane 1: lane 0 owns the bulk copies)
            test_pending();
            if (lane == 1) {
#pragma unroll
                for (int j = 0; j < kGroup; ++j) {
                    if (j < k)
                        st_relaxed_gpu_u64(P.part + (long long)row * NC + c0 + j,
                                           pack_partial(gm[j], gs[j], (int)first[j]));
                }
                pend_old = atom_add_relaxed_gpu(P.cnt + row, k);
                pend_k = k;
                pend_row = row;
                pend_lrow = P.compact ? fast_div(gu, P.div_nc) : row;
            }
        }
        test_pending();
        if (failed) {
            if (lane == 0) set_error(P.err, DLLM_DEVERR_TIMEOUT);
            // let this warp's copies in flight land before shared memory goes away
            while (consumed < issued) {
                const int slot = consumed % kStages;
                if (!mbar_wait_bounded(bar0 + slot * 8, (consumed / kStages) & 1u, 100000000ull)) {
                    if (lane == 0) atomicExch(&s_ring_busy, 1);   // the ring may still be written
                    break;
                }
                ++consumed;
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            atomicAdd(&s_ndone, 1);
        }
        drain_queue(FP, s_gmask, s_queue, &s_qhead, &s_ndone, lane);   // help with the backlog
    } else {
        // ---- finisher warps: scan signal, requests without masked rows, queue
        if (warp == kFirstFinisher && lane == 0) {
            __threadfence();
            atomicAdd(P.ctl, 1);   // this CTA no longer reads input_ids' entry state
        }
        if (!P.shard)
            for (int k = warp - kFirstFinisher; k < s_nzero; k += kFinishWarps)
                finalize_request(FP, s_zero[k], false, lane);
        drain_queue(FP, s_gmask, s_queue, &s_qhead, &s_ndone, lane);
    }

    // ---- exit: the last CTA commits deferred requests and resets ----------
    __syncthreads();
    if (tid == 0) {
        const unsigned old = (unsigned)atom_add_acqrel_gpu(FP.ctl + 1, 1);
        s_last = ((int)(old & 0xffffu) == G - 1) ? 1 + (int)(old >> 16) : 0;   // 1 + deferred commits
    }
    // the fused commit's element map depends on launch parameters only:
    // every CTA builds it in its idle rings while the exit add is in flight
    if (FP.commit && !s_ring_busy)
        compact_map<kThreads>(FP.cp, *reinterpret_cast<CompactScratch<kThreads>*>(smem), tid);
    __syncthreads();
    if (s_last) {
        const int n_def = s_last - 1;
        const int* list = FP.cnt + FP.BL + FP.B;
        for (int i = tid; i < n_def; i += kThreads) {   // finalized before every CTA had scanned
            const int e = __ldcg(list + i);
            const int b = e & 0xffff;
            const bool rst = (e & kDeferReset) != 0;
            for (int j = 0; j < FP.L; ++j) {
                const long long idx = (long long)b * FP.L + j;
                if (rst) FP.ids[idx] = FP.mask_id;
                else if (FP.sel[idx]) FP.ids[idx] = __ldcg(FP.row_tok + idx);
            }
        }
        if (FP.commit) {
            // every request is committed: compact the caller's row arrays by
            // the eviction flags, staged through the (now idle) copy rings
            __syncthreads();
            if (s_ring_busy) {
                if (tid == 0) set_error(FP.err, DLLM_DEVERR_TIMEOUT);
            } else {
                auto& scratch = *reinterpret_cast<CompactScratch<kThreads>*>(smem);
                unsigned char* stage = smem + kCommitScratchBytes;
                compact_rows<kThreads>(FP.cp, scratch, stage, FP.c_evict, FP.B, tid);
            }
        }
        if (tid == 0) {
            FP.ctl[0] = 0;
            FP.ctl[1] = 0;
            FP.ctl[2] = 0;
        }
    }
}

// Standalone features: one warp per request.
template <int NK>
__device__ __forceinline__ void features_one(int b, int L, int mask_id, const int* ids, const float* cs, float* feats,
                                             int lane) {
    float val[NK];
    bool inU[NK];
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        const int j = lane + 32 * k;
        const bool valid = j < L;
        const int id = valid ? ids[(long long)b * L + j] : mask_id;
        inU[k] = valid && id != mask_id;
        val[k] = valid ? cs[(long long)b * L + j] : 0.f;
    }
    warp_features<NK>(val, inU, L, lane, feats + (long long)b * DLLM_NUM_FEATURES);
}

__global__ void __launch_bounds__(256) features_kernel(int B, int L, int mask_id, const int* ids, const float* cs,
                                                      float* feats) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= B) return;
    const int nk = (L + 31) >> 5;
    if (nk <= 1) features_one<1>(b, L, mask_id, ids, cs, feats, lane);
    else if (nk <= 2) features_one<2>(b, L, mask_id, ids, cs, feats, lane);
    else if (nk <= 4) features_one<4>(b, L, mask_id, ids, cs, feats, lane);
    else features_one<32>(b, L, mask_id, ids, cs, feats, lane);
}

// ---------------------------------------------------------------------------
// Merge of vocabulary-shard triples, then S3-S6: one warp per request.
// Shard k's triple of position r is at m/s/idx[k * stride + r]; the shards
// are folded in order with the finisher's combine (so the lowest global
// argmax wins ties when the shards ascend through the vocabulary).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ StepParams P, int n_shards,
                                                    const float* __restrict__ tm, const float* __restrict__ ts,
                                                    const int* __restrict__ ti, long long stride) {
    pdl_wait();      // the triples and the batch state come from earlier kernels
    pdl_release();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= P.B) return;
    bool any = false;
    for (int j = lane; j < P.L; j += 32) {
        const long long r = (long long)b * P.L + j;
        if (P.ids[r] != P.mask_id) continue;
        any = true;
        float M = -INFINITY, S = 0.f;
        int tok = -1;
        for (int k = 0; k < n_shards; ++k) {
            const float mk = tm[k * stride + r];
            if (mk > M || tok < 0) tok = ti[k * stride + r];
            combine(M, S, mk, ts[k * stride + r]);
        }
        const float conf = __fdiv_rn(1.0f, S);
        if (P.conf_out) P.conf_out[r] = conf;
        if (P.lse_out) P.lse_out[r] = M + logf(S);
        if (P.tok_out) P.tok_out[r] = tok;
        P.row_tok[r] = tok;
        st_relaxed_gpu_u64(P.row_word + r, pack_row(conf, tok));
    }
    any = __any_sync(0xffffffffu, any);
    __syncwarp();
    finalize_request(P, b, any, lane, true);
}

// per-device launch state, read without the lock on the launch path:
// atomics publish it (release) and read it (acquire)
std::atomic<int> g_smem_configured[64];

struct LaunchFacts {
    std::atomic<bool> ready{false};
    long long max_dynamic = 0;   // dynamic shared memory available to step_kernel (written before ready)
};
LaunchFacts g_launch_facts[64];
std::mutex g_launch_mu;

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" size_t dllm_step_workspace_size(int32_t B, int32_t L, int32_t V) {
    if (B < 0 || L < 1 || L > DLLM_MAX_L || V < 1) return 0;
    return ws_required(B, L, V);
}

extern "C" int dllm_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (!workspace && bytes) return DLLM_ERR_INVAL;
    if (!bytes) return DLLM_OK;
    DLLM_CUDA_TRY(cudaMemsetAsync(workspace, 0, bytes, as_stream(stream)));
    return DLLM_OK;
}

namespace dllm {
namespace {

struct ShardOut {
    int v0;
    float* m;
    float* s;
    int* idx;
};

// The block commit and compaction fused into a step (dllm_step_commit).
struct CommitSpec {
    const dllm_advance_args* adv;
    const dllm_compact_args* cmp;
};

// Vocabulary shards reduced in one launch (dllm_step_vocab_shards), already
// checked to tile [0, V) in order.
struct ShardTable {
    int n;
    const dllm_vocab_shard* s;
};

// A checked step launch: grid, block, shared memory and parameters.
struct StepLaunch {
    bool empty;   // B == 0: nothing to launch
    int grid;
    size_t smem;
    StepParams P;
};

// Host checks of a step call and its launch parameters; launches nothing
// and writes no device memory.  quota null selects the threshold rule;
// logits_rows >= 0 the compact layout; shard non-null S2 alone over a
// vocabulary shard.
int prepare_step(const dllm_step_args* a, const int32_t* quota, long long logits_rows, const ShardOut* shard,
                 StepLaunch* out, const CommitSpec* commit = nullptr, const ShardTable* vs = nullptr) {
    out->empty = true;
    if (!a) return DLLM_ERR_INVAL;
    if (a->B < 0 || a->L < 1 || a->L > DLLM_MAX_L || a->V < 1 || (!vs && a->ldv < a->V)) return DLLM_ERR_INVAL;
    if (a->B == 0) return DLLM_OK;
    if ((long long)a->B * a->L > 0x7fffffffLL || a->B >= (1 << 16)) return DLLM_ERR_UNSUPPORTED;
    if ((!vs && !a->logits) || !a->input_ids) return DLLM_ERR_INVAL;
    if (!shard && ((!quota && !a->thr) || !a->conf_state || !a->done || !a->accept_len || !a->n_new))
        return DLLM_ERR_INVAL;
    if (shard && (!shard->m || !shard->s || !shard->idx || shard->v0 < 0)) return DLLM_ERR_INVAL;
    if (!vs && ((a->ldv % 8) != 0 || (reinterpret_cast<uintptr_t>(a->logits) & 15u) != 0)) return DLLM_ERR_ALIGN;
    if (!a->workspace || (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0) return DLLM_ERR_WORKSPACE;
    // chunks per row: the row's, or each shard's in turn
    long long nc_ll = (a->V + kChunkElems - 1) / kChunkElems;
    if (vs) {
        nc_ll = 0;
        for (int k = 0; k < vs->n; ++k) nc_ll += (vs->s[k].V + kChunkElems - 1) / kChunkElems;
    }
    WsLayout w;
    if (!ws_layout_nc(a->B, a->L, nc_ll, a->workspace_bytes, &w)) return DLLM_ERR_WORKSPACE;

    int dev = 0;
    DLLM_CUDA_TRY(cudaGetDevice(&dev));
    const int G = sm_count();
    if (G <= 0) return DLLM_ERR_CUDA;
    if (G >= (1 << 15)) return DLLM_ERR_UNSUPPORTED;   // the exit counter's low half counts CTAs
    const int BL = a->B * a->L;
    if ((long long)BL * nc_ll > 0x7fffffffLL) return DLLM_ERR_UNSUPPORTED;
    const int NC = (int)nc_ll;
    if ((long long)BL * NC > 0x7fffffffLL || (long long)BL * G > 0x7fffffffLL || (long long)a->V * G > 0x7fffffffLL)
        return DLLM_ERR_UNSUPPORTED;
    // rows one CTA touches: its static share (< BL / G + 3 rows) plus the
    // tail (at most min(ceil(BL / kTailDen), kTailRowsMax) rows)
    const int static_cap = BL / G + 3;
    const int list_cap = static_cap + min((BL + kTailDen - 1) / kTailDen, kTailRowsMax);
    const int zero_cap = a->B / G + 1;
    const size_t smem = size_t(kStreamWarps) * kStages * kCopyBytes + size_t(kStreamWarps) * kStages * 8 +
                        size_t(3 * list_cap + zero_cap) * 4 + size_t((BL + 15) / 16) * 2;
    // per-device launch facts, queried once
    if (dev < 0 || dev >= 64) return DLLM_ERR_UNSUPPORTED;
    LaunchFacts& lf = g_launch_facts[dev];
    if (!lf.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_launch_mu);
        if (!lf.ready.load(std::memory_order_relaxed)) {
            int max_optin = 0;
            DLLM_CUDA_TRY(cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
            cudaFuncAttributes fa;
            DLLM_CUDA_TRY(cudaFuncGetAttributes(&fa, step_kernel));
            lf.max_dynamic = max_optin - (long long)fa.sharedSizeBytes;
            lf.ready.store(true, std::memory_order_release);
        }
    }
    if ((long long)smem > lf.max_dynamic) return DLLM_ERR_UNSUPPORTED;
    if (g_smem_configured[dev].load(std::memory_order_acquire) < (int)smem) {
        std::lock_guard<std::mutex> lock(g_launch_mu);
        if (g_smem_configured[dev].load(std::memory_order_relaxed) < (int)smem) {
            DLLM_CUDA_TRY(cudaFuncSetAttribute(step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            g_smem_configured[dev].store((int)smem, std::memory_order_release);
        }
    }

    unsigned char* ws = static_cast<unsigned char*>(a->workspace);
    unsigned char* data = ws + ((a->workspace_bytes - w.data_bytes) & ~size_t(255));
    StepParams& P = out->P;
    memset(&P, 0, sizeof(P));
    if (commit) {
        const dllm_advance_args* v = commit->adv;
        P.commit = 1;
        P.c_rid = v->rid;
        P.c_K = v->K;
        P.c_b = v->b;
        P.c_gen = v->gen_tokens;
        P.c_ld_gen = v->ld_gen;
        P.c_evict = v->evict;
        const int prc = make_compact_plan(commit->cmp, kThreads, kCommitStageBytes, &P.cp);
        if (prc != DLLM_OK) return prc;
    }
    if (vs) {
        P.n_shards = vs->n;
        int c0 = 0;
        for (int k = 0; k < vs->n; ++k) {
            P.sh_logits[k] = vs->s[k].logits;
            P.sh_ldv[k] = vs->s[k].ldv;
            P.sh_v0[k] = vs->s[k].v0;
            P.sh_V[k] = vs->s[k].V;
            P.sh_c0[k] = c0;
            c0 += (vs->s[k].V + kChunkElems - 1) / kChunkElems;
        }
        for (int k = vs->n; k <= DLLM_MAX_VOCAB_SHARDS; ++k) P.sh_c0[k] = c0;
    }
    P.B = a->B; P.L = a->L; P.V = a->V; P.NC = NC; P.BL = BL; P.mask_id = a->mask_id;
    P.list_cap = list_cap; P.static_cap = static_cap; P.zero_cap = zero_cap; P.ldv = a->ldv;
    P.div_nc = make_fastdiv((uint32_t)NC);
    P.compact = logits_rows >= 0 ? 1 : 0;
    P.logits_rows = logits_rows;
    P.shard = shard ? 1 : 0;
    P.v0 = shard ? shard->v0 : 0;
    P.trip_m = shard ? shard->m : nullptr;
    P.trip_s = shard ? shard->s : nullptr;
    P.trip_i = shard ? shard->idx : nullptr;
    P.div_g = make_fastdiv((uint32_t)G);
    P.logits = a->logits; P.ids = a->input_ids; P.thr = a->thr; P.quota = quota; P.cs = a->conf_state;
    P.done = a->done; P.accept = a->accept_len; P.n_new = a->n_new; P.feats = a->feats;
    P.conf_out = a->conf_out; P.lse_out = a->lse_out; P.tok_out = a->tok_out;
    P.ctl = reinterpret_cast<int*>(ws);
    P.cnt = reinterpret_cast<int*>(ws + 64);
    P.part = reinterpret_cast<unsigned long long*>(ws + w.off_part);
    P.row_word = reinterpret_cast<unsigned long long*>(ws + w.off_row);
    P.row_tok = reinterpret_cast<int*>(data + w.off_tok);
    P.sel = data + w.off_sel;
    P.err = error_word_ptr();
    if (!P.err) return DLLM_ERR_CUDA;
    out->grid = G;
    out->smem = smem;
    out->empty = false;
    return DLLM_OK;
}

int launch_prepared(const StepLaunch& sl, void* stream) {
    if (sl.empty) return DLLM_OK;
    DLLM_CUDA_TRY(launch_dependent(step_kernel, dim3(sl.grid), dim3(kThreads), sl.smem, as_stream(stream), sl.P));
    return DLLM_OK;
}

int launch_step(const dllm_step_args* a, const int32_t* quota, long long logits_rows, const ShardOut* shard,
                void* stream, const CommitSpec* commit = nullptr, const ShardTable* vs = nullptr) {
    StepLaunch sl;
    const int rc = prepare_step(a, quota, logits_rows, shard, &sl, commit, vs);
    if (rc != DLLM_OK) return rc;
    return launch_prepared(sl, stream);
}

// The fused commit's arguments against the step's: the same rows, block
// length, mask id, input_ids and conf_state, and the step's done flags as
// the advance flags.
int check_commit(const dllm_step_args* a, const dllm_advance_args* adv, const dllm_compact_args* cmp) {
    if (!a || !adv || !cmp) return DLLM_ERR_INVAL;
    if (adv->A != a->B || cmp->A != a->B || adv->L != a->L || adv->mask_id != a->mask_id) return DLLM_ERR_INVAL;
    if (adv->input_ids != a->input_ids || adv->conf_state != a->conf_state) return DLLM_ERR_INVAL;
    if (adv->advance && adv->advance != a->done) return DLLM_ERR_INVAL;   // the step's done flags advance
    if (a->B > 0 && (!adv->rid || !adv->K || !adv->b || !adv->gen_tokens || !adv->evict || adv->ld_gen < 0))
        return DLLM_ERR_INVAL;
    return DLLM_OK;
}

// A shard table: 1..DLLM_MAX_VOCAB_SHARDS shards tiling [0, V) in order,
// each row at least its shard wide, 16-byte rows.
int check_shards(const dllm_step_args* a, int32_t n_shards, const dllm_vocab_shard* shards) {
    if (!a || !shards || n_shards < 1 || n_shards > DLLM_MAX_VOCAB_SHARDS) return DLLM_ERR_INVAL;
    long long next = 0;
    for (int k = 0; k < n_shards; ++k) {
        const dllm_vocab_shard& sh = shards[k];
        if (!sh.logits || sh.V < 1 || sh.v0 != next || sh.ldv < sh.V) return DLLM_ERR_INVAL;
        next += sh.V;
    }
    if (next != a->V) return DLLM_ERR_INVAL;
    for (int k = 0; k < n_shards; ++k)
        if (shards[k].ldv % 8 != 0 || (reinterpret_cast<uintptr_t>(shards[k].logits) & 15u) != 0) return DLLM_ERR_ALIGN;
    return DLLM_OK;
}

}  // namespace
}  // namespace dllm

extern "C" int dllm_step(const dllm_step_args* a, void* stream) { return launch_step(a, nullptr, -1, nullptr, stream); }

extern "C" int dllm_step_quota(const dllm_step_args* a, const int32_t* quota, void* stream) {
    if (!quota) return DLLM_ERR_INVAL;
    return launch_step(a, quota, -1, nullptr, stream);
}

extern "C" int dllm_step_compact(const dllm_step_args* a, int64_t logits_rows, const int32_t* quota, void* stream) {
    if (logits_rows < 0) return DLLM_ERR_INVAL;
    return launch_step(a, quota, logits_rows, nullptr, stream);
}

extern "C" int dllm_step_commit(const dllm_step_args* a, const int32_t* quota, int64_t logits_rows,
                                const dllm_advance_args* adv, const dllm_compact_args* cmp, void* stream) {
    const int rc = check_commit(a, adv, cmp);
    if (rc != DLLM_OK) return rc;
    const CommitSpec commit{adv, cmp};
    return launch_step(a, quota, logits_rows < 0 ? -1 : logits_rows, nullptr, stream, &commit);
}

extern "C" int dllm_step_vocab_shards(const dllm_step_args* a, int32_t n_shards, const dllm_vocab_shard* shards,
                                      const int32_t* quota, void* stream) {
    const int rc = check_shards(a, n_shards, shards);
    if (rc != DLLM_OK) return rc;
    const ShardTable vs{n_shards, shards};
    return launch_step(a, quota, -1, nullptr, stream, nullptr, &vs);
}

extern "C" int dllm_step_vocab_shards_commit(const dllm_step_args* a, int32_t n_shards,
                                             const dllm_vocab_shard* shards, const int32_t* quota,
                                             const dllm_advance_args* adv, const dllm_compact_args* cmp,
                                             void* stream) {
    int rc = check_shards(a, n_shards, shards);
    if (rc != DLLM_OK) return rc;
    rc = check_commit(a, adv, cmp);
    if (rc != DLLM_OK) return rc;
    const ShardTable vs{n_shards, shards};
    const CommitSpec commit{adv, cmp};
    return launch_step(a, quota, -1, nullptr, stream, &commit, &vs);
}

extern "C" int dllm_step_shard(const dllm_step_args* a, int32_t v0, float* m, float* s, int32_t* idx, void* stream) {
    ShardOut sh{v0, m, s, idx};
    return launch_step(a, nullptr, -1, &sh, stream);
}

extern "C" int dllm_step_merge(const dllm_step_args* a, int32_t n_shards, const float* m, const float* s,
                               const int32_t* idx, int64_t shard_stride, const int32_t* quota, void* stream) {
    if (!a || a->B < 0 || a->L < 1 || a->L > DLLM_MAX_L || a->V < 1) return DLLM_ERR_INVAL;
    if (a->B == 0) return DLLM_OK;
    if ((long long)a->B * a->L > 0x7fffffffLL || a->B >= (1 << 16)) return DLLM_ERR_UNSUPPORTED;
    if (n_shards < 1 || !m || !s || !idx || shard_stride < (int64_t)a->B * a->L) return DLLM_ERR_INVAL;
    if (!a->input_ids || (!quota && !a->thr) || !a->conf_state || !a->done || !a->accept_len || !a->n_new)
        return DLLM_ERR_INVAL;
    if (!a->workspace || (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0) return DLLM_ERR_WORKSPACE;
    WsLayout w;   // only the zero-at-rest row words and the data end are used: any V lays them out
    if (!ws_layout(a->B, a->L, 1, a->workspace_bytes, &w)) return DLLM_ERR_WORKSPACE;
    unsigned char* ws = static_cast<unsigned char*>(a->workspace);
    unsigned char* data = ws + ((a->workspace_bytes - w.data_bytes) & ~size_t(255));
    StepParams P;
    memset(&P, 0, sizeof(P));
    P.B = a->B; P.L = a->L; P.V = a->V; P.BL = a->B * a->L; P.mask_id = a->mask_id;
    P.ids = a->input_ids; P.thr = a->thr; P.quota = quota; P.cs = a->conf_state;
    P.done = a->done; P.accept = a->accept_len; P.n_new = a->n_new; P.feats = a->feats;
    P.conf_out = a->conf_out; P.lse_out = a->lse_out; P.tok_out = a->tok_out;
    P.ctl = reinterpret_cast<int*>(ws);
    P.cnt = reinterpret_cast<int*>(ws + 64);
    P.row_word = reinterpret_cast<unsigned long long*>(ws + w.off_row);
    P.row_tok = reinterpret_cast<int*>(data + w.off_tok);
    P.sel = data + w.off_sel;
    P.err = error_word_ptr();
    if (!P.err) return DLLM_ERR_CUDA;
    const int wpb = 8;
    DLLM_CUDA_TRY(launch_dependent(merge_kernel, dim3((a->B + wpb - 1) / wpb), dim3(wpb * 32), 0, as_stream(stream), P,
                                   n_shards, m, s, idx, (long long)shard_stride));
    return DLLM_OK;
}

extern "C" int32_t dllm_transfer_quota(int32_t L, int32_t S, int32_t s) {
    if (L < 1 || S < 1 || s < 0) return -1;
    if (s >= S) return L;
    return L / S + (s < L % S ? 1 : 0);
}

extern "C" int dllm_features(int32_t B, int32_t L, int32_t mask_id, const int32_t* input_ids,
                             const float* conf_state, float* feats, void* stream) {
    if (B < 0 || L < 1 || L > DLLM_MAX_L) return DLLM_ERR_INVAL;
    if (B == 0) return DLLM_OK;
    if (!input_ids || !conf_state || !feats) return DLLM_ERR_INVAL;
    const int wpb = 8;
    features_kernel<<<(B + wpb - 1) / wpb, wpb * 32, 0, as_stream(stream)>>>(B, L, mask_id, input_ids, conf_state,
                                                                          feats);
    DLLM_CUDA_TRY(cudaGetLastError());
    return DLLM_OK;
}

// ---------------------------------------------------------------------------
// dllm_step_noalloc: dllm_step with a built-in scratch buffer.
//
// Some callers cannot allocate device memory for the step's workspace: a
// serving engine that has already handed every byte of HBM to its own pool,
// a plain C host with no allocator of its own, or a latency-critical loop
// where a cudaMalloc (which may synchronise the device) is not allowed.
// For them the workspace lives in this file-scope array instead.  Every GPU
// that loads the library holds the array until the process exits.
// ---------------------------------------------------------------------------
namespace dllm {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;   // 16 MiB per device

static __device__ __align__(256) unsigned char g_step_scratch[kNoallocScratchBytes];

void* g_scratch_dev_ptr[64];
std::mutex g_scratch_mu;

// Device address of this device's scratch array; looked up once per device
// with that device current.  nullptr if the lookup fails.
void* scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_dev_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
        if (e != cudaSuccess) {
            note_cuda_error(e);
            return nullptr;
        }
        g_scratch_dev_ptr[dev] = p;
    }
    return g_scratch_dev_ptr[dev];
}

}  // namespace
}  // namespace dllm

extern "C" size_t dllm_step_noalloc_capacity(void) { return dllm::kNoallocScratchBytes; }

extern "C" int dllm_step_noalloc(const dllm_step_args* a, void* stream) {
    if (!a) return DLLM_ERR_INVAL;
    if (a->B < 0 || a->L < 1 || a->L > DLLM_MAX_L || a->V < 1) return DLLM_ERR_INVAL;
    if (a->B == 0) return DLLM_OK;
    dllm::WsLayout w;
    if (!dllm::ws_layout(a->B, a->L, a->V, dllm::kNoallocScratchBytes, &w)) return DLLM_ERR_SCRATCH_LIMIT;
    void* scratch = dllm::scratch_ptr();
    if (!scratch) return DLLM_ERR_CUDA;
    dllm_step_args b = *a;
    b.workspace = scratch;
    b.workspace_bytes = dllm::kNoallocScratchBytes;
    // Every check of dllm_step runs before anything touches the shared
    // array, so a rejected call leaves it (and everything else) unchanged.
    dllm::StepLaunch sl;
    const int rc = dllm::prepare_step(&b, nullptr, -1, nullptr, &sl);
    if (rc != DLLM_OK) return rc;
    // The array keeps whatever the previous call left; the step needs its
    // counter region at zero, so clear exactly that part first.
    DLLM_CUDA_TRY(cudaMemsetAsync(scratch, 0, w.counters_bytes, dllm::as_stream(stream)));
    return dllm::launch_prepared(sl, stream);
}
