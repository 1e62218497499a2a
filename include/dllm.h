/*
 * dllm.h -- C ABI of libdllm.so: the data-parallel hot path of block-wise
 * diffusion-LLM serving on one GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *   FDFO page      "FDFO: 让 dLLM 推理从「整批等最慢」变成「谁先完成谁先走」"
 *                  (write-up of SGLang PRs #27551 / #27877)
 *   BlockServe     "BlockServe: 块粒度连续批处理实现高吞吐扩散大语言模型服务"
 *   DiLaServe      "DiLaServe: High SLO Attainment Serving for Diffusion
 *                  Language Models" (paper review)
 *
 * Conventions shared by every entry point
 *   - Every function returns int: DLLM_OK (0) or a negative DLLM_ERR_* code.
 *     Nothing is thrown across the ABI.  dllm_strerror() names a code.
 *   - "device" pointers are caller-owned CUDA device memory on the current
 *     device; "host" pointers are ordinary host memory.  The library never
 *     allocates or frees device memory, and no entry point keeps a pointer
 *     after returning -- except the native loop object (dllm_loop_create:
 *     host memory and a small pinned staging block of its own, and the
 *     caller's workspace, all held until dllm_loop_destroy).
 *   - Device entry points are asynchronous on `stream` (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).  Only
 *     dllm_get_device_error() synchronises.
 *   - Arguments are validated on the host before any launch; a rejected call
 *     launches nothing and changes nothing.
 *   - Conditions only the device can see (an inconsistent row width in
 *     dllm_pack, an expired wait) are recorded in a per-device error word,
 *     read and cleared by dllm_get_device_error().  Kernels never trap.
 *   - Integer widths are fixed (int32_t / int64_t); bf16 data is passed as
 *     raw 16-bit patterns (uint16_t).
 */
#ifndef DLLM_H
#define DLLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DLLM_ABI_VERSION 2

#define DLLM_OK 0
#define DLLM_ERR_INVAL (-1)       /* a size, pointer or value is out of range */
#define DLLM_ERR_ALIGN (-2)       /* a pointer or stride breaks an alignment rule */
#define DLLM_ERR_CUDA (-3)        /* a CUDA runtime call failed */
#define DLLM_ERR_DEVICE (-4)      /* the device error word was set (see below) */
#define DLLM_ERR_WORKSPACE (-5)   /* workspace missing or too small */
#define DLLM_ERR_UNSUPPORTED (-6) /* shape beyond this build's limits */
#define DLLM_ERR_SCRATCH_LIMIT (-7) /* shape needs more than dllm_step_noalloc's built-in scratch */

/* Device error word values (read with dllm_get_device_error). */
#define DLLM_DEVERR_NONE 0
#define DLLM_DEVERR_TIMEOUT 1     /* a bounded wait (bulk copy, partial word) expired */
#define DLLM_DEVERR_ROW_WIDTH 2   /* dllm_pack: p + (b + 1) * L > W for a row */
#define DLLM_DEVERR_BLOCK_INDEX 3 /* dllm_advance: block index outside [0, K) or output row too short */
#define DLLM_DEVERR_LOGITS_ROWS 4 /* dllm_step_compact: more masked positions than logits rows */

#define DLLM_MAX_L 1024
#define DLLM_NUM_FEATURES 6
#define DLLM_COMPACT_MAX_ARRAYS 16

/* Describe a status code (static string; never NULL). */
const char* dllm_strerror(int code);

/* ABI version of the loaded library (DLLM_ABI_VERSION). */
int dllm_abi_version(void);

/* The cudaError_t of the last CUDA runtime call that failed inside this
 * library on the calling thread (0 if none), and its name in *name when
 * name is not NULL.  Explains a DLLM_ERR_CUDA return. */
int dllm_last_cuda_error(const char** name);

/* sizeof() of the argument structs below, for binding self-checks:
 * which = 0 dllm_step_args, 1 dllm_pack_args, 2 dllm_compact_args,
 * 3 dllm_advance_args, 4 dllm_refill_args, 5 dllm_loop_config,
 * 6 dllm_loop_info_t, 7 dllm_vocab_shard.  Returns 0 for an unknown `which`. */
size_t dllm_struct_size(int which);

/* Fault injection for tests of the status plumbing (host only; nothing
 * reaches the GPU).  The `countdown`-th CUDA runtime call that this library
 * makes next on the calling thread is not made: it reports `cuda_error` (a
 * cudaError_t value) instead, so the entry point that made it returns
 * DLLM_ERR_CUDA and dllm_last_cuda_error() names `cuda_error`.  Calls
 * before it run normally; countdown 0 disarms.  DLLM_ERR_INVAL for a
 * negative countdown or a zero cuda_error with a countdown. */
int dllm_inject_cuda_error(int32_t cuda_error, int32_t countdown);

/* Synchronise `stream`, then return in *code the first device error
 * recorded on the current device since the last call (DLLM_DEVERR_*), and
 * clear it.  Returns DLLM_ERR_CUDA if the synchronisation fails. */
int dllm_get_device_error(void* stream, int32_t* code);

/* ======================================================================
 * dllm_step -- one denoise step over a mixed-state batch (S1-S6).
 *
 * FDFO page, section "工程设计一": step(forward_batch, full_logits, states)
 * -> done_flags reads the current logits, updates forward_batch.input_ids
 * by the algorithm's rule and reports, per block, whether it is complete.
 * The rule is LowConfidence (same section; DiLaServe review, section 3.1):
 * for every masked position take the softmax probability of the argmax
 * token as its confidence; unmask positions whose confidence exceeds the
 * request's threshold; if none does, unmask the single most confident one.
 *
 * Per request b (row block of L positions) and masked position j
 * (input_ids[b][j] == mask_id at entry), over x = logits row b*L + j:
 *   m = max_v x_v; tok = lowest v with x_v == m;
 *   s = sum_v exp(x_v - m); conf = 1 / s; lse = m + ln(s).
 * Selection: sel = { masked j : conf_j > thr[b] } (strict, float32); if sel
 *   is empty and some position is masked, sel = { the masked j of largest
 *   conf, lowest j on ties }.
 * Update: input_ids[b][j] = tok_j and conf_state[b][j] = conf_j for j in sel.
 * Outputs (FDFO page, section "工程设计二": accept_length is 0 while the
 * block continues and block_size once it can be committed):
 *   n_new[b]      = |sel|
 *   done[b]       = 1 iff no position of block b holds mask_id afterwards
 *   accept_len[b] = done[b] ? L : 0
 *   feats[b][0..5] (DiLaServe review, section 4.2 item ③) over the block's
 *     positions not holding mask_id afterwards, values conf_state[b][j]:
 *     min, q25, median, mean, q75 (linear interpolation at rank q*(n-1) of
 *     the ascending values) and n / L; NaN x5 and 0 when n == 0.
 *   conf_out / lse_out / tok_out (optional): per position, the row results
 *     for positions masked at entry, NaN / NaN / -1 elsewhere.
 *
 * Only rows of positions masked at entry are read; other logits rows may
 * hold anything.  Rows must hold at least one finite value.  The reduction
 * order of every row depends only on V, so a request's results are
 * bit-identical whatever else is in the batch.
 * ====================================================================== */
typedef struct dllm_step_args {
    int32_t B;                  /* requests (>= 0) */
    int32_t L;                  /* block length, 1..DLLM_MAX_L */
    int32_t V;                  /* vocabulary size (>= 1) */
    int32_t mask_id;            /* token id marking a masked position */
    int64_t ldv;                /* logits row stride in elements: >= V, multiple of 8 */
    const uint16_t* logits;     /* device bf16 [B*L][ldv]; row b*L+j = position j of request b;
                                   16-byte aligned; all B*L*ldv elements addressable */
    int32_t* input_ids;         /* device [B][L], in/out (the block's tokens) */
    const float* thr;           /* device [B] per-request threshold */
    float* conf_state;          /* device [B][L], in/out: confidence recorded at unmask time
                                   (the per-request algorithm state carried between rounds);
                                   finite wherever input_ids != mask_id */
    uint8_t* done;              /* device [B] out */
    int32_t* accept_len;        /* device [B] out */
    int32_t* n_new;             /* device [B] out */
    float* feats;               /* device [B][6] out, or NULL */
    float* conf_out;            /* device [B][L] out, or NULL */
    float* lse_out;             /* device [B][L] out, or NULL */
    int32_t* tok_out;           /* device [B][L] out, or NULL */
    void* workspace;            /* device, >= dllm_step_workspace_size() bytes, 256-byte aligned,
                                   zero-filled before first use (dllm_workspace_init); every
                                   completed call leaves it ready for the next */
    size_t workspace_bytes;
} dllm_step_args;

/* Workspace bytes dllm_step needs for this shape (0 if the shape is invalid).
 * A workspace sized for (B, L, V) also serves every call with B' <= B,
 * B'*L' <= B*L and B'*L'*ceil(V'/8192) <= B*L*ceil(V/8192): its first
 * quarter holds the words that must be zero between calls (counters and
 * the packed chunk partials, which each call clears as it reads them) and
 * the rest the per-call data, so no call's data lands on another's
 * zero-at-rest words.  Calls sharing a workspace must be ordered on one
 * stream.  After a device error (DLLM_DEVERR_TIMEOUT) re-initialise it. */
size_t dllm_step_workspace_size(int32_t B, int32_t L, int32_t V);

/* cudaMemsetAsync(workspace, 0, bytes) on `stream`. */
int dllm_workspace_init(void* workspace, size_t bytes, void* stream);

/* Run S1-S6.  Errors: DLLM_ERR_INVAL (shape, NULL required pointer),
 * DLLM_ERR_ALIGN (logits not 16-byte aligned, ldv % 8 != 0),
 * DLLM_ERR_WORKSPACE, DLLM_ERR_CUDA, DLLM_ERR_UNSUPPORTED (B >= 65536,
 * B * L * number of SMs * 8 or V * number of SMs * 8 at or above 2^31, or
 * the shared memory the shape needs above the device's limit).  A NaN
 * threshold never passes.  input_ids and conf_state may not alias any
 * output. */
int dllm_step(const dllm_step_args* args, void* stream);

/* S1-S6 with the fixed-steps rule in place of the threshold rule (BlockServe
 * page, section II-E: each block's masked tokens are transferred over S
 * denoising steps by a per-step quota).  Request b unmasks exactly quota[b]
 * of its masked positions -- the most confident ones, ties to the lower
 * position -- or all of them when fewer are masked; quota[b] <= 0 unmasks
 * nothing.  quota: device int32 [B].  Everything else is dllm_step's (S1, S2,
 * S4-S6, outputs, workspace rules); args->thr is not read and may be NULL.
 * Errors as dllm_step, plus DLLM_ERR_INVAL for a NULL quota. */
int dllm_step_quota(const dllm_step_args* args, const int32_t* quota, void* stream);

/* S1-S6 reading compact logits: args->logits holds logits_rows rows of the
 * row stride args->ldv, and row k is the logits of the k-th masked position
 * of the batch at entry, in position order (b * L + j ascending) -- the rows
 * dllm_step reads, and only those (a model may compute its LM head for the
 * masked positions alone; a host copies M rows instead of B * L).  quota
 * NULL selects the threshold rule, else the fixed-steps rule as
 * dllm_step_quota.  Everything else, including the results, is as
 * dllm_step.  If the batch has more masked positions than logits_rows, no
 * logits are read, the device error word gets DLLM_DEVERR_LOGITS_ROWS and
 * the outputs of requests with masked positions are unspecified (the
 * workspace stays valid).  DLLM_ERR_INVAL for logits_rows < 0. */
int dllm_step_compact(const dllm_step_args* args, int64_t logits_rows, const int32_t* quota, void* stream);

/* S1-S2 over one vocabulary shard (a vocabulary-parallel LM head -- the
 * tensor parallelism of the DiLaServe review, section 2.2.2 -- or an LM head
 * computed in vocabulary chunks).  args->logits points at the shard's first
 * column, global token v0 (v0 % 8 == 0 keeps the rows 16-byte aligned),
 * args->V is the shard's width and args->ldv the full row stride.  For every
 * masked position r (input_ids[r] == mask_id) it writes the shard's triple
 * m[r] = max, s[r] = sum of exp(x - m) over the shard, idx[r] = the lowest
 * global index attaining m; nothing else (input_ids unchanged; thr,
 * conf_state and the outputs are not read or written).  m, s, idx: device
 * [B * L].  The workspace rules are dllm_step's (sized for the shard's V). */
int dllm_step_shard(const dllm_step_args* args, int32_t v0, float* m, float* s, int32_t* idx, void* stream);

/* S3-S6 from the triples of n_shards vocabulary shards: shard k's triple of
 * position r at m / s / idx[k * shard_stride + r] (device), shards in
 * ascending vocabulary order.  They are folded in that order as the step's
 * finisher folds chunk partials (M = max, S = sum of s_k exp(m_k - M), the
 * first shard attaining M gives the token: the lowest global index), then
 * selection, update, done and features exactly as dllm_step (quota NULL:
 * threshold rule; else the fixed-steps rule).  args->logits is not read; the
 * workspace must be sized for (B, L, any V >= 1).  Errors as dllm_step, plus
 * DLLM_ERR_INVAL for n_shards < 1, shard_stride < B * L or NULL triples. */
int dllm_step_merge(const dllm_step_args* args, int32_t n_shards, const float* m, const float* s,
                    const int32_t* idx, int64_t shard_stride, const int32_t* quota, void* stream);

/* The step over logits held as vocabulary shards, all on this device, in
 * one launch: what dllm_step_shard on every shard followed by
 * dllm_step_merge computes, bit for bit, without the triples' round trip or
 * the per-launch start-up and tail paid once per shard (an LM head computed
 * in vocabulary chunks into separate buffers, or the shards of a
 * vocabulary-parallel head gathered on one GPU).
 *   - shards[k]: logits (device bf16 [B*L][ldv], 16-byte aligned, ldv a
 *     multiple of 8 and >= V) holding global tokens [v0, v0 + V); shard 0
 *     starts at v0 = 0, each next one where the previous ends, and their
 *     widths add up to args->V.  1 <= n_shards <= DLLM_MAX_VOCAB_SHARDS.
 *   - args as for dllm_step; args->logits and args->ldv are not read.  quota
 *     NULL: the threshold rule, else the fixed-steps rule.
 *   - Each shard is reduced in its own chunks (a shard's reduction order
 *     depends only on its width), so the workspace must hold
 *     dllm_step_workspace_size(B, L, V + 8192 * (n_shards - 1)) bytes.
 *   - DLLM_ERR_INVAL for a shard list that does not tile [0, V) in order or
 *     a NULL shard, DLLM_ERR_ALIGN as dllm_step per shard, and every error
 *     of dllm_step. */
#define DLLM_MAX_VOCAB_SHARDS 8
typedef struct dllm_vocab_shard {
    const uint16_t* logits;   /* device [B*L][ldv] */
    int64_t ldv;              /* row stride in elements */
    int32_t v0;               /* first global token of the shard */
    int32_t V;                /* tokens in the shard (>= 1) */
} dllm_vocab_shard;

int dllm_step_vocab_shards(const dllm_step_args* args, int32_t n_shards, const dllm_vocab_shard* shards,
                           const int32_t* quota, void* stream);

/* Host.  The fixed-steps quota of step s (0-based) of a block (BlockServe
 * page, section II-E): L spread evenly over S steps, floor(L / S) per step
 * plus one for each of the first L mod S steps; a step past the schedule
 * (s >= S) returns L (transfer everything left).  -1 if L < 1, S < 1 or
 * s < 0. */
int32_t dllm_transfer_quota(int32_t L, int32_t S, int32_t s);

/* dllm_step without a caller workspace (the pages have no counterpart; this
 * is a deployment convenience).  It runs exactly dllm_step, but its scratch
 * is a fixed buffer of dllm_step_noalloc_capacity() bytes (16 MiB) that the
 * library holds on every device it is loaded on, until the process exits.
 * It is meant for callers that cannot allocate device memory: an engine
 * whose memory pool already owns all of HBM, a plain C host without an
 * allocator, or a loop where an allocation (which may synchronise the
 * device) is not allowed.  args->workspace and args->workspace_bytes are
 * ignored; everything else is as for dllm_step.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Each call clears the buffer's counter region (an asynchronous memset
 *     on `stream`) and then launches the step; nothing is allocated or
 *     freed, by this library or any library it calls.
 *   - All calls on a device share the one buffer, which keeps the previous
 *     call's contents: calls whose execution can overlap on the GPU (other
 *     streams, other host threads without ordering) race and corrupt each
 *     other.  Order them on one stream.
 *   - Shapes whose workspace exceeds the buffer (dllm_step_workspace_size
 *     layout; for V near 150k, B * L * ceil(V / 8192) above about 480k) return
 *     DLLM_ERR_SCRATCH_LIMIT and launch nothing.
 *   - Every argument check of dllm_step runs before the memset: a call that
 *     returns an error has queued nothing and left the buffer as it was. */
int dllm_step_noalloc(const dllm_step_args* args, void* stream);

/* Bytes of dllm_step_noalloc's built-in scratch buffer per device. */
size_t dllm_step_noalloc_capacity(void);

/* S6 alone: feats[b][0..5] from input_ids / conf_state as defined above
 * (DiLaServe review, section 4.2 item ③).  All pointers device. */
int dllm_features(int32_t B, int32_t L, int32_t mask_id, const int32_t* input_ids,
                  const float* conf_state, float* feats, void* stream);

/* ======================================================================
 * Confidence-threshold control (host functions; DiLaServe review, section
 * 3.2, "Confidence Threshold Controller").  Thresholds are indexed by their
 * position in an ascending candidate list (e.g. {0.5, 0.6, 0.7, 0.8, 0.9},
 * section 4.1).  All arrays are host memory, row-major [R][T].
 * ====================================================================== */

/* A stand-in for the review's step predictor (item ③: a gradient-boosted
 * model over 11 features, trained offline -- not built here).  For request
 * i at candidate threshold cand[k]: P = P(confidence > cand[k]) read off
 * the block features feats[i][0..5] (dllm_step's output: min, q25, median,
 * avg, q75, unmasked fraction) as the piecewise-linear distribution through
 * (min, 0), (q25, .25), (median, .5), (q75, .75), (1, 1), or 1 - cand[k]
 * when no position is unmasked yet (NaN features); a step then unmasks
 * max(1, floor(P m)) of the m positions still masked.  steps_out[i][k] =
 * steps to clear masked[i] positions + blocks_left[i] * steps to clear L.
 * Double precision, no contraction.  DLLM_ERR_INVAL for R < 0, T < 1,
 * L < 1, masked[i] outside [0, L], blocks_left[i] < 0 or a NULL array. */
int dllm_predict_steps_stub(int32_t R, int32_t T, const double* cand, int32_t L, const float* feats,
                            const int32_t* masked, const int32_t* blocks_left, double* steps_out);

/* Algorithm 2 (item ②, adaptive load control).  load[i][k]: request i's
 * load at threshold k (total tokens x predicted remaining steps); requests
 * in arrival order; capacity = tokens per second x SLO.  For each request in
 * turn, thresholds are tried from the highest down; threshold k is dropped
 * while committed + load[i][k] + rest[i] > capacity (rest[i] = the later
 * requests at their lowest threshold, summed from the back: rest[R-1] = 0,
 * rest[i] = load[i+1][0] + rest[i+1]), and the
 * first that fits becomes max_allowed[i] (the lowest is kept if none fits);
 * committed then adds load[i][max_allowed[i]].  Every threshold at or below
 * max_allowed[i] stays allowed. */
int dllm_load_control(int32_t R, int32_t T, const double* load, double capacity, int32_t* max_allowed);

/* Algorithm 1 (item ①, SLO-aware threshold choice).  choice[i] = the
 * highest k <= max_allowed[i] (T - 1 when max_allowed is NULL) with
 * rem_steps[i][k] * step_latency[i] <= slo_left[i], else 0 (the fastest).
 * DLLM_ERR_INVAL for a max_allowed entry outside [0, T). */
int dllm_slo_thresholds(int32_t R, int32_t T, const double* rem_steps, const double* step_latency,
                        const double* slo_left, const int32_t* max_allowed, int32_t* choice);

/* One decision of the whole controller for R active requests (items ③, ②
 * and ① in that order), all host arithmetic in double precision:
 *   steps_out[i][k]  = dllm_predict_steps_stub(cand, L, feats, masked,
 *                      blocks_left) (remaining steps at threshold k);
 *   load[i][k]       = steps_out[i][k] * total_tokens[i] (prompt + output
 *                      tokens; item ②);
 *   max_allowed[i]   = dllm_load_control over that load with capacity =
 *                      tokens_per_s * slo_s;
 *   choice[i]        = dllm_slo_thresholds with step latency step_latency_s
 *                      (the latency of one step at the current batch size,
 *                      from the instance's one-off profile) and
 *                      slo_left[i] = slo_s - elapsed_s[i] (the SLO budget
 *                      left since request i arrived).
 * Outputs: steps_out [R][T], max_allowed [R], choice [R] (host).  Inputs
 * as for dllm_predict_steps_stub, plus total_tokens [R] (>= 0) and
 * elapsed_s [R] (host).  DLLM_ERR_INVAL for a NULL array, a negative token
 * count or any input dllm_predict_steps_stub rejects. */
int dllm_threshold_control(int32_t R, int32_t T, const double* cand, int32_t L, const float* feats,
                           const int32_t* masked, const int32_t* blocks_left, const int64_t* total_tokens,
                           const double* elapsed_s, double slo_s, double tokens_per_s, double step_latency_s,
                           double* steps_out, int32_t* max_allowed, int32_t* choice);

/* ======================================================================
 * Bounding-box planning and admission (host functions).
 *
 * BlockServe page, section II-D, eq. (1):
 *   Cost(A) = |A| * max_{i in A} (p_i + (b_i + 1) * L).
 * ====================================================================== */

/* Host.  W = max_i (p[i] + (b[i] + 1) * L) (0 when A == 0) and
 * cost = A * W.  p, b: host [A], p >= 0, b >= 0.  W and cost may be NULL. */
int dllm_pack_plan(int32_t A, const int32_t* p, const int32_t* b, int32_t L,
                   int32_t* W, int64_t* cost);

/* Host.  Length-aware greedy ("sand-fill") admission, BlockServe page,
 * section II-D and Algorithm 1 (section II-C):
 *   repeat: let W_cur be the active box width; among the remaining pending
 *   requests whose starting width p + L fits within W_cur, take the longest
 *   prompt (earliest in the queue on ties); if none fits, take the head of
 *   the queue; admit it iff Cost(A plus it, at b = 0) <= budget, else stop.
 * pending_p: host [n_pending], sorted ascending (the queue order).
 * active_p, active_b: host [A] of the active set (may be NULL when A == 0).
 * admit_idx: host [n_pending] out, indices into pending_p in admission
 * order; *n_admit receives their count. */
int dllm_admit(int32_t n_pending, const int32_t* pending_p, int32_t A,
               const int32_t* active_p, const int32_t* active_b, int32_t L,
               int64_t budget, int32_t* admit_idx, int32_t* n_admit);

/* ======================================================================
 * dllm_pack -- materialise the box (S7), BlockServe page, section II-E
 * ("逻辑位置对齐" and "向量化混合调度执行").
 *
 * Row i (request rid[i], prompt length p[i], block index b[i]):
 *   width_i = p[i] + (b[i] + 1) * L;  pad_i = W - width_i
 *   ids[i]  = [pad_id x pad_i, prompt tokens, gen_tokens[rid][0 : b*L],
 *              block_ids[i][0 : L]]
 *   attn[i][c] = c >= pad_i;  pos[i][c] = max(c - pad_i, 0)
 *     (the cumulative index over the attention mask, first real token at 0)
 *   blk_start[i] = p[i] + b[i] * L, the logical position of the active
 *     block, which always occupies box columns [W - L, W) (the gather /
 *     scatter region of every row).
 * A row with width_i > W, or one that needs prompt_tokens or gen_tokens
 * while that pointer is NULL, is skipped and sets DLLM_DEVERR_ROW_WIDTH.
 * (prompt_tokens may be NULL when every p is 0, gen_tokens when every b is 0.)
 * ====================================================================== */
typedef struct dllm_pack_args {
    int32_t A;                    /* rows */
    int32_t L;                    /* block length */
    int32_t W;                    /* box width (dllm_pack_plan) */
    int32_t pad_id;
    const int32_t* p;             /* device [A] prompt length per row */
    const int32_t* b;             /* device [A] block index per row */
    const int32_t* rid;           /* device [A] request id per row */
    const int64_t* prompt_off;    /* device [R + 1]: prompt of request r is
                                     prompt_tokens[prompt_off[r] : prompt_off[r] + p] */
    const int32_t* prompt_tokens; /* device */
    const int32_t* gen_tokens;    /* device [R][ld_gen]: committed blocks of request r */
    int64_t ld_gen;
    const int32_t* block_ids;     /* device [A][L]: current block of each row */
    int32_t* ids;                 /* device [A][W] out */
    uint8_t* attn;                /* device [A][W] out, or NULL */
    int32_t* pos;                 /* device [A][W] out, or NULL */
    int32_t* pad;                 /* device [A] out, or NULL */
    int32_t* blk_start;           /* device [A] out, or NULL */
} dllm_pack_args;

int dllm_pack(const dllm_pack_args* args, void* stream);

/* The in-place re-loop's box update (FDFO page, section "工程设计四",
 * #27877: when no block completed in a round, the next forward and step run
 * on the same batch without a return to the scheduler).  With no block
 * committed, no row was admitted or evicted and every width is unchanged, so
 * the box differs from the last dllm_pack only in the active blocks: this
 * rewrites ids[i][W - L + j] = block_ids[i][j] for i < A, j < L and leaves
 * every other column and attn / pos / pad / blk_start as they are.  Reads
 * args->A, L, W, block_ids and ids only.  Errors: DLLM_ERR_INVAL (A < 0,
 * L < 1, W < L with A > 0, NULL block_ids or ids). */
int dllm_pack_block(const dllm_pack_args* args, void* stream);

/* ======================================================================
 * dllm_advance -- commit finished blocks (BlockServe Algorithm 1: update
 * r_i's outputs with its block, b_i <- b_i + 1, evict when b_i >= K_i;
 * FDFO page, section "FDFO 的核心思想": a request whose block is done
 * commits at once).
 *
 * For every row i with advance[i] != 0:
 *   gen_tokens[rid[i]][b[i]*L : (b[i]+1)*L] = input_ids[i][0 : L];
 *   b[i] += 1;  evict[i] = (b[i] >= K[i]);
 *   if not evicted: input_ids[i][:] = mask_id, conf_state[i][:] = NaN
 *   (every block starts fully masked, BlockServe section II-E).
 * Rows with advance[i] == 0 get evict[i] = 0 and are untouched.
 * ====================================================================== */
typedef struct dllm_advance_args {
    int32_t A;
    int32_t L;
    int32_t mask_id;
    int32_t pad0;
    const uint8_t* advance;   /* device [A] */
    const int32_t* rid;       /* device [A] */
    const int32_t* K;         /* device [A] blocks to generate */
    int32_t* b;               /* device [A] in/out */
    int32_t* input_ids;       /* device [A][L] in/out */
    float* conf_state;        /* device [A][L] in/out */
    int32_t* gen_tokens;      /* device [R][ld_gen] out (rows of advanced requests) */
    int64_t ld_gen;           /* >= K * L for every request */
    uint8_t* evict;           /* device [A] out */
} dllm_advance_args;

int dllm_advance(const dllm_advance_args* args, void* stream);

/* ======================================================================
 * dllm_compact -- stable compaction for FDFO eviction (S9).
 *
 * keep[i] = !evict[i];  new_index[i] = number of kept rows before i (or -1
 * when evicted);  src_row[k] = the k-th kept row;  *A_out = kept rows.
 * Every listed row-major array is compacted in place: row k becomes old row
 * src_row[k] for k < A_out (rows >= A_out are left unspecified).  Survivors
 * keep their order; refills are appended after them by the caller.
 * ====================================================================== */
typedef struct dllm_compact_args {
    int32_t A;                                   /* rows */
    int32_t n_arrays;                            /* 0..DLLM_COMPACT_MAX_ARRAYS */
    const uint8_t* evict;                        /* device [A] */
    int32_t* new_index;                          /* device [A] out, or NULL */
    int32_t* src_row;                            /* device [A] out (first A_out valid), or NULL */
    int32_t* A_out;                              /* device [1] out */
    void* arrays[DLLM_COMPACT_MAX_ARRAYS];       /* device, A rows each */
    int64_t row_bytes[DLLM_COMPACT_MAX_ARRAYS];  /* bytes per row (> 0) */
    void* workspace;                             /* device, dllm_compact_workspace_size() bytes */
    size_t workspace_bytes;
} dllm_compact_args;

/* dllm_advance followed by dllm_compact on the evict flags it computes, in
 * one launch (one CTA): the batch-management tail of a serving-loop
 * iteration (BlockServe Algorithm 1: commit, b += 1, evict; FDFO page,
 * section "FDFO 的核心思想": done requests leave at once).  Results equal
 * dllm_advance(adv) then dllm_compact(cmp) with cmp->evict = adv->evict
 * (cmp->evict is not read).  When the rows of all the arrays exceed one
 * 96 KiB staging chunk and cmp supplies a workspace of at least
 * dllm_compact_workspace_size bytes, the call runs exactly those two
 * (several CTAs each); otherwise one CTA does both and the workspace is
 * not read.  The compacted arrays may
 * include adv's b / input_ids / conf_state (they are compacted after the
 * commit).  Errors as the two calls, plus DLLM_ERR_INVAL when cmp->A !=
 * adv->A and DLLM_ERR_UNSUPPORTED when a row of all the arrays holds more
 * than 2048 elements of one size: each array's row moves in 16-byte
 * elements when its row size and address are multiples of 16, else 4-byte
 * elements when they are multiples of 4, else bytes. */
int dllm_advance_compact(const dllm_advance_args* adv, const dllm_compact_args* cmp, void* stream);

/* One FDFO iteration's step and batch tail in one launch: dllm_step (or
 * dllm_step_quota when quota is not NULL; with logits_rows >= 0 the logits
 * hold the masked positions' rows only, as for dllm_step_compact, and a
 * negative logits_rows means the full [B*L][ldv] array) followed by
 * dllm_advance with the
 * step's done flags as the advance flags and dllm_compact by the eviction
 * flags it sets -- the same results as dllm_step then dllm_advance_compact
 * (FDFO page, section "FDFO 的核心思想": a request whose block is done
 * commits it at once and starts its next block or leaves; BlockServe page,
 * Algorithm 1).  Each request's finaliser commits its own block as soon as
 * the step has decided it; the grid's last CTA then compacts the listed
 * row arrays, staged through the step's shared memory.
 *   - step: as dllm_step.  adv: adv->A == step->B, adv->L == step->L,
 *     adv->mask_id == step->mask_id, adv->input_ids == step->input_ids,
 *     adv->conf_state == step->conf_state, adv->advance NULL or
 *     step->done; rid, K, b, gen_tokens, ld_gen and evict as for
 *     dllm_advance.  cmp: cmp->A == step->B; arrays, row_bytes, new_index,
 *     src_row and A_out as for dllm_compact (cmp->evict and the workspace
 *     are not read); the arrays may include b, input_ids and conf_state.
 *   - DLLM_ERR_INVAL when the pairs above differ, and every error of
 *     dllm_step, dllm_advance and dllm_compact; DLLM_ERR_UNSUPPORTED when
 *     a row of all the arrays holds more than 2048 elements of one size (as
 *     for dllm_advance_compact).
 *   - Any number of rows: the last CTA compacts them in chunks of at most
 *     480 rows, staged through about 140 KiB of shared memory.  A block
 *     index outside [0, K) sets DLLM_DEVERR_BLOCK_INDEX and that row is not
 *     advanced. */
int dllm_step_commit(const dllm_step_args* step, const int32_t* quota, int64_t logits_rows,
                     const dllm_advance_args* adv, const dllm_compact_args* cmp, void* stream);

/* dllm_step_vocab_shards followed by the batch tail of dllm_step_commit, in
 * one launch: the step over logits held as vocabulary shards on this device,
 * then each finished request's block commit and the compaction of the
 * listed row arrays (FDFO page, section "FDFO 的核心思想"; BlockServe page,
 * Algorithm 1).  The results equal dllm_step_vocab_shards then
 * dllm_advance_compact with the step's done flags as the advance flags.
 *   - step, n_shards, shards, quota: as dllm_step_vocab_shards (the
 *     workspace holds dllm_step_workspace_size(B, L, V + 8192 *
 *     (n_shards - 1)) bytes; step->logits and step->ldv are not read).
 *   - adv, cmp: as dllm_step_commit.
 *   - Errors: those of dllm_step_vocab_shards, then those of
 *     dllm_step_commit. */
int dllm_step_vocab_shards_commit(const dllm_step_args* step, int32_t n_shards, const dllm_vocab_shard* shards,
                                  const int32_t* quota, const dllm_advance_args* adv, const dllm_compact_args* cmp,
                                  void* stream);

/* Workspace bytes for dllm_compact over these arrays (0 if invalid). */
size_t dllm_compact_workspace_size(int32_t A, int32_t n_arrays, const int64_t* row_bytes);

int dllm_compact(const dllm_compact_args* args, void* stream);

/* ======================================================================
 * dllm_refill -- append admitted requests (S9 refill).
 *
 * BlockServe page, section II-D (refill from the pending queue) and
 * section II-E (every block starts fully masked); survivors keep their rows
 * and admitted requests are appended after them, in admission order.
 * Rows [A0, A0 + n) of the row arrays receive request new_rid[r] with prompt
 * length new_p[r], new_K[r] blocks to generate and threshold new_thr[r];
 * their block index becomes 0, input_ids becomes mask_id and conf_state NaN.
 * ====================================================================== */
typedef struct dllm_refill_args {
    int32_t A0;               /* first appended row */
    int32_t n;                /* rows appended */
    int32_t L;
    int32_t mask_id;
    const int32_t* new_rid;   /* device [n] */
    const int32_t* new_p;     /* device [n] */
    const int32_t* new_K;     /* device [n] */
    const float* new_thr;     /* device [n] */
    int32_t* rid;             /* device row arrays, >= A0 + n rows */
    int32_t* p;
    int32_t* b;
    int32_t* K;
    float* thr;
    int32_t* input_ids;       /* device [rows][L] */
    float* conf_state;        /* device [rows][L] */
} dllm_refill_args;

int dllm_refill(const dllm_refill_args* args, void* stream);

/* ======================================================================
 * The serving loop, native (BlockServe Algorithm 1, section II-C, in the
 * FDFO or sync mode of the FDFO page, sections "FDFO 的核心思想" and
 * "工程设计一"; the in-place re-loop of its section "工程设计四"; optionally
 * the fixed-steps rule of BlockServe section II-E).
 *
 * One iteration is two calls around the caller's model forward:
 *   dllm_loop_begin: sand-fill admission (dllm_admit) and refill
 *     (dllm_refill) of the pending queue, then the box of eq. (1)
 *     (dllm_pack; dllm_pack_block after a step that committed nothing, when
 *     re-loop is on -- admission is skipped then: it would admit nothing);
 *   dllm_loop_end: the step over the caller's logits ([A * L][ldv], row
 *     i * L + j = position j of active row i), the block commit and
 *     compaction in one launch (dllm_advance_compact) and the readback of
 *     the done flags (it synchronises the stream).  FDFO: the commit
 *     follows the step on the stream before the readback (done rows
 *     advance; with no row done it leaves the batch unchanged).  Sync: it
 *     is launched after the readback, and only when every block is done.
 * Device memory: everything lives in the caller's workspace
 * (dllm_loop_workspace_size bytes, 256-byte aligned); the loop object
 * itself is host memory, with a small pinned block (about 21 bytes per
 * row of capacity) for the per-iteration copies, all freed by
 * dllm_loop_destroy.  The pending queue is every request, sorted by prompt
 * length (ties by request id).
 * ====================================================================== */
typedef struct dllm_loop dllm_loop;

typedef struct dllm_loop_config {
    int32_t R;          /* requests */
    int32_t L;          /* block length, 1..DLLM_MAX_L */
    int32_t V;          /* vocabulary size */
    int32_t mask_id;
    int32_t pad_id;
    int32_t mode;       /* 0 FDFO, 1 sync */
    int32_t reloop;     /* 1: in-place re-loop */
    int32_t S;          /* 0: threshold rule (per-request thresholds); > 0: fixed-steps rule, S steps per block */
    int32_t capacity;   /* most active rows at once (admission beyond it returns DLLM_ERR_UNSUPPORTED) */
    int32_t pad0;
    int64_t budget;     /* token budget of eq. (1) */
} dllm_loop_config;

typedef struct dllm_loop_info_t {
    int32_t A;              /* active rows */
    int32_t W;              /* box width */
    int64_t cost;           /* eq. (1) of the active set */
    int32_t iteration;      /* completed iterations */
    int32_t reloops;        /* iterations that ran in place */
    int32_t pending;        /* requests not yet admitted */
    int32_t admitted_last;  /* requests the last dllm_loop_begin admitted */
    int32_t finished;       /* nothing pending and nothing active */
    int32_t in_place;       /* the next iteration re-loops */
    int64_t ld_gen;         /* row stride of gen_tokens */
    int32_t* block_ids;     /* device [A][L] current blocks */
    float* conf_state;      /* device [A][L] */
    int32_t* box_ids;       /* device [A][W] */
    uint8_t* box_attn;      /* device [A][W] */
    int32_t* box_pos;       /* device [A][W] */
    int32_t* box_pad;       /* device [A] */
    int32_t* box_blk_start; /* device [A] */
    int32_t* gen_tokens;    /* device [R][ld_gen]: committed blocks per request */
    uint8_t* done;          /* device [A], last step's (pre-compaction rows) */
    int32_t* n_new;
    int32_t* accept_len;
    float* feats;           /* device [A][6] */
} dllm_loop_info_t;

/* Workspace bytes for the loop (0 if the configuration is invalid).  p, K:
 * host [R] prompt lengths (>= 0) and blocks to generate (>= 1). */
size_t dllm_loop_workspace_size(const dllm_loop_config* cfg, const int32_t* p, const int32_t* K);

/* Create a loop.  thr: host [R] thresholds (threshold rule); prompt_off:
 * device [R + 1] offsets into prompt_tokens (device; may be NULL when every
 * p is 0).  The workspace's step counters are cleared on `stream`.  Errors:
 * DLLM_ERR_INVAL, DLLM_ERR_WORKSPACE, DLLM_ERR_CUDA. */
int dllm_loop_create(const dllm_loop_config* cfg, const int32_t* p, const int32_t* K, const float* thr,
                     const int64_t* prompt_off, const int32_t* prompt_tokens, void* workspace,
                     size_t workspace_bytes, void* stream, dllm_loop** out);

/* Frees the loop object and its pinned staging (after any upload from it
 * has finished).  The workspace stays the caller's: do not free it while
 * the loop's kernels may still run on the stream. */
void dllm_loop_destroy(dllm_loop* loop);

int dllm_loop_begin(dllm_loop* loop, void* stream);
int dllm_loop_end(dllm_loop* loop, const uint16_t* logits, int64_t ldv, void* stream);

/* State after the last call, with device pointers into the workspace. */
int dllm_loop_info(const dllm_loop* loop, dllm_loop_info_t* out);

/* Host copies of the active rows' request ids, block indices and steps taken
 * in the current block (A entries each; any pointer may be NULL). */
int dllm_loop_rows(const dllm_loop* loop, int32_t* rid, int32_t* b, int32_t* s);

/* Per-request threshold control inside the native loop (DiLaServe review,
 * section 3.2): before every step, dllm_threshold_control picks each active
 * row's threshold from `candidates` and dllm_loop_end uploads them, in place
 * of the requests' fixed thresholds; after the step the rows' block features
 * are read back with the done flags.  The controller's inputs are kept as
 * the Python loop keeps them:
 *   - features: the row's last step's (all NaN for a row admitted since, or
 *     whose block advanced: nothing unmasked yet); masked positions
 *     L - rint(f[5] * L) in float32, L when f[0] is NaN;
 *   - blocks left K - b - 1; total tokens p + K * L;
 *   - time since admission on a modelled clock that advances, after every
 *     step over A rows, by the step latency latency_s + latency_per_row_s * A
 *     (the review's one-off latency profile, as an affine fit), which is
 *     also the latency the controller is given.
 * control: T >= 1 ascending candidates (host, copied), slo_s > 0,
 * tokens_per_s >= 0, both latency terms >= 0; NULL turns the control off
 * (fixed thresholds again).  Rows stepped before the call count as having
 * no features.  Host only; DLLM_ERR_INVAL for a NULL loop or invalid
 * control.  The fixed-steps rule (config S > 0) ignores thresholds. */
typedef struct dllm_loop_control {
    int32_t T;                  /* candidate thresholds */
    const double* candidates;   /* host [T], ascending */
    double slo_s;               /* every request's latency SLO, seconds */
    double tokens_per_s;        /* the instance's rate: capacity = tokens_per_s * slo_s */
    double latency_s;           /* step latency at A rows: latency_s + latency_per_row_s * A */
    double latency_per_row_s;
} dllm_loop_control;

int dllm_loop_set_control(dllm_loop* loop, const dllm_loop_control* control);

/* The thresholds the last dllm_loop_end gave the rows it stepped, in their
 * order at that step (before the commit compacted them): *n entries into
 * thr (host, room for the loop's capacity).  Without control they are the
 * requests' own thresholds. */
int dllm_loop_thresholds(const dllm_loop* loop, float* thr, int32_t* n);

#ifdef __cplusplus
}
#endif

#endif /* DLLM_H */
