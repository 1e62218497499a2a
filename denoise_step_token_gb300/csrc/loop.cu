// The serving loop as native host code: BlockServe Algorithm 1 (section
// II-C: admit under the token budget of eq. (1), run one step, commit
// finished blocks, evict requests whose blocks are all done) in FDFO or sync
// mode (FDFO page, sections "FDFO 的核心思想" and "工程设计一"), with the
// in-place re-loop of the FDFO page, section "工程设计四", and optionally
// the fixed-steps rule of BlockServe section II-E.
//
// One iteration is two calls around the caller's model forward:
//   dllm_loop_begin: admission (host) and refill, then the box of eq. (1)
//     (dllm_pack, or dllm_pack_block when the last step committed nothing);
//   dllm_loop_end: the step over the caller's logits and the done-flag
//     readback (the one host round trip), then the host mirrors.  In FDFO
//     mode the block commit and compaction run in the step's own launch
//     (dllm_step_commit), before the readback: they use the done flags on
//     the device and leave the batch as it is when no block finished.  In
//     sync mode the host decides after the readback (a commit needs every
//     block done) and launches the commit.  With threshold control
//     (dllm_loop_set_control; DiLaServe review, section 3.2) the step's
//     thresholds are chosen on the host just before it and uploaded, and
//     the block features come back with the done flags.
// The host keeps only what admission needs (prompt lengths, block indices,
// steps in the current block) and a small pinned staging block for the
// per-iteration copies; every array the kernels read lives in the caller's
// device workspace.

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <limits>
#include <vector>

#include "common.cuh"

struct dllm_loop {
    dllm_loop_config c;
    int32_t Kmax = 0, Wmax = 0;
    std::vector<int32_t> p_all, K_all;
    std::vector<float> thr_all;
    std::vector<int32_t> pending;     // request ids, queue order
    std::vector<int32_t> pending_p;   // their prompt lengths
    std::vector<int32_t> rid_h, b_h, s_h, p_act;
    std::vector<uint8_t> wait_h;
    std::vector<int32_t> admit_idx;
    // pinned host staging: done flags (readback), quotas and the refill
    // rows (uploads); `staged` orders a rewrite after the last upload
    void* pinned = nullptr;
    uint8_t* done_h = nullptr;
    int32_t* quota_h = nullptr;
    int32_t* stage_h = nullptr;   // [4][n]: rid, p, K, thr bits of the admitted requests
    float* thr_p = nullptr;       // thresholds of the next step (upload)
    float* feat_p = nullptr;      // [A][6] block features of the last step (readback)
    cudaEvent_t staged = nullptr;
    bool staged_pending = false;
    // threshold control (DiLaServe review, section 3.2): the controller's
    // host inputs per active row, the modelled clock and scratch
    bool ctl_on = false;
    std::vector<double> ctl_cand;
    double ctl_slo = 0, ctl_tps = 0, ctl_lat0 = 0, ctl_lat1 = 0;
    double now = 0;                   // modelled clock, seconds
    std::vector<double> admit_h;      // admission time per active row
    std::vector<float> feat_h;        // [A][6] last step's features per active row
    std::vector<float> thr_used;      // thresholds of the rows the last step ran on
    std::vector<int32_t> c_masked, c_left, c_cap, c_choice;
    std::vector<int64_t> c_total;
    std::vector<double> c_elapsed, c_steps;
    int32_t A = 0, W = 0, admitted_last = 0, iteration = 0, reloops = 0;
    int64_t cost = 0;
    bool in_place = false, have_box = false;
    const int64_t* prompt_off = nullptr;
    const int32_t* prompt_tokens = nullptr;
    // device arrays, carved from the caller's workspace
    int32_t *rid = nullptr, *p = nullptr, *b = nullptr, *K = nullptr, *ids = nullptr, *gen = nullptr;
    float *thr = nullptr, *cs = nullptr, *feats = nullptr;
    int32_t *box_ids = nullptr, *box_pos = nullptr, *box_pad = nullptr, *box_blk = nullptr;
    uint8_t *box_attn = nullptr, *done = nullptr, *evict = nullptr;
    int32_t *accept = nullptr, *n_new = nullptr, *new_index = nullptr, *src_row = nullptr, *A_out = nullptr;
    int32_t *quota = nullptr, *stage_d = nullptr;
    void* step_ws = nullptr;
    size_t step_ws_bytes = 0;
    void* compact_ws = nullptr;
    size_t compact_ws_bytes = 0;

    ~dllm_loop() {
        // an upload from the staging may still be in flight (a begin with
        // no end after it): let it finish before the memory goes
        if (staged && staged_pending) cudaEventSynchronize(staged);
        if (staged) cudaEventDestroy(staged);
        if (pinned) cudaFreeHost(pinned);
    }
};

namespace {
// the batch arrays compacted after each commit: rid, p, b, K, thr, ids, cs
inline void compact_row_bytes(int32_t L, int64_t* rb) {
    for (int k = 0; k < 5; ++k) rb[k] = 4;
    rb[5] = rb[6] = (int64_t)L * 4;
}
}  // namespace

namespace {

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Wait until the last upload from the pinned staging has been read, so the
// staging can be rewritten (a no-op in the usual order: every dllm_loop_end
// synchronises the stream).
int staging_free(dllm_loop* lp) {
    if (lp->staged_pending) {
        if (cudaEventSynchronize(lp->staged) != cudaSuccess) return DLLM_ERR_CUDA;
        lp->staged_pending = false;
    }
    return DLLM_OK;
}

int staging_used(dllm_loop* lp, cudaStream_t s) {
    if (cudaEventRecord(lp->staged, s) != cudaSuccess) return DLLM_ERR_CUDA;
    lp->staged_pending = true;
    return DLLM_OK;
}

// Arguments of the block commit and compaction of the A active rows: rows
// whose device done flag is set advance (a fresh block, or eviction after
// their last block); the survivors are compacted in order.
void commit_args(dllm_loop* lp, int32_t A, dllm_advance_args& aa, dllm_compact_args& ca) {
    const dllm_loop_config& c = lp->c;
    memset(&aa, 0, sizeof(aa));
    aa.A = A; aa.L = c.L; aa.mask_id = c.mask_id; aa.advance = lp->done; aa.rid = lp->rid; aa.K = lp->K; aa.b = lp->b;
    aa.input_ids = lp->ids; aa.conf_state = lp->cs; aa.gen_tokens = lp->gen; aa.ld_gen = (int64_t)lp->Kmax * c.L;
    aa.evict = lp->evict;
    memset(&ca, 0, sizeof(ca));
    ca.A = A; ca.n_arrays = 7; ca.evict = lp->evict; ca.new_index = lp->new_index; ca.src_row = lp->src_row;
    ca.A_out = lp->A_out;
    void* arrays[7] = {lp->rid, lp->p, lp->b, lp->K, lp->thr, lp->ids, lp->cs};
    int64_t rb[7];
    compact_row_bytes(c.L, rb);
    for (int k = 0; k < 7; ++k) {
        ca.arrays[k] = arrays[k];
        ca.row_bytes[k] = rb[k];
    }
    ca.workspace = lp->compact_ws;
    ca.workspace_bytes = lp->compact_ws_bytes;
}

// The commit and compaction as their own launch (sync mode).
int launch_commit(dllm_loop* lp, int32_t A, void* stream) {
    dllm_advance_args aa;
    dllm_compact_args ca;
    commit_args(lp, A, aa, ca);
    return dllm_advance_compact(&aa, &ca, stream);
}

// Carve the loop's device arrays from `base` (or only size them when base is
// null); returns the bytes used.
size_t carve(dllm_loop* lp, unsigned char* base) {
    const dllm_loop_config& c = lp->c;
    const size_t cap = (size_t)c.capacity, L = (size_t)c.L;
    size_t off = 0;
    auto take = [&](size_t bytes) -> unsigned char* {
        unsigned char* q = base ? base + off : nullptr;
        off = al256(off + bytes);
        return q;
    };
    lp->step_ws_bytes = dllm_step_workspace_size(c.capacity, c.L, c.V);
    lp->step_ws = take(lp->step_ws_bytes);   // first: must start zeroed
    lp->rid = (int32_t*)take(cap * 4);
    lp->p = (int32_t*)take(cap * 4);
    lp->b = (int32_t*)take(cap * 4);
    lp->K = (int32_t*)take(cap * 4);
    lp->thr = (float*)take(cap * 4);
    lp->ids = (int32_t*)take(cap * L * 4);
    lp->cs = (float*)take(cap * L * 4);
    lp->gen = (int32_t*)take((size_t)c.R * (size_t)lp->Kmax * L * 4);
    lp->box_ids = (int32_t*)take(cap * (size_t)lp->Wmax * 4);
    lp->box_attn = (uint8_t*)take(cap * (size_t)lp->Wmax);
    lp->box_pos = (int32_t*)take(cap * (size_t)lp->Wmax * 4);
    lp->box_pad = (int32_t*)take(cap * 4);
    lp->box_blk = (int32_t*)take(cap * 4);
    lp->done = (uint8_t*)take(cap);
    lp->evict = (uint8_t*)take(cap);
    lp->accept = (int32_t*)take(cap * 4);
    lp->n_new = (int32_t*)take(cap * 4);
    lp->feats = (float*)take(cap * DLLM_NUM_FEATURES * 4);
    lp->new_index = (int32_t*)take(cap * 4);
    lp->src_row = (int32_t*)take(cap * 4);
    lp->A_out = (int32_t*)take(4);
    lp->quota = (int32_t*)take(cap * 4);
    lp->stage_d = (int32_t*)take(cap * 16);
    int64_t rb[7];
    compact_row_bytes(c.L, rb);
    lp->compact_ws_bytes = dllm_compact_workspace_size(c.capacity, 7, rb);
    lp->compact_ws = take(lp->compact_ws_bytes);
    return off;
}

bool config_ok(const dllm_loop_config* c) {
    return c && c->R >= 0 && c->L >= 1 && c->L <= DLLM_MAX_L && c->V >= 1 && c->capacity >= 1 &&
           (c->mode == 0 || c->mode == 1) && c->S >= 0 && c->budget >= 0;
}

bool shapes(const dllm_loop_config* c, const int32_t* p, const int32_t* K, int32_t* Kmax, int32_t* Wmax) {
    long long km = 1, wm = c->L;
    for (int32_t r = 0; r < c->R; ++r) {
        if (p[r] < 0 || K[r] < 1) return false;
        km = std::max<long long>(km, K[r]);
        wm = std::max<long long>(wm, (long long)p[r] + (long long)K[r] * c->L);
    }
    if (wm > 0x7fffffffLL || km * c->L > 0x7fffffffLL) return false;
    *Kmax = (int32_t)km;
    *Wmax = (int32_t)wm;
    return true;
}

// The controller's thresholds for the A active rows into thr_used.
int choose_thresholds(dllm_loop* lp, int32_t A) {
    const int32_t L = lp->c.L, T = (int32_t)lp->ctl_cand.size();
    lp->c_masked.resize(A);
    lp->c_left.resize(A);
    lp->c_total.resize(A);
    lp->c_elapsed.resize(A);
    lp->c_cap.resize(A);
    lp->c_choice.resize(A);
    lp->c_steps.resize((size_t)A * T);
    for (int32_t i = 0; i < A; ++i) {
        const float* f = &lp->feat_h[(size_t)i * DLLM_NUM_FEATURES];
        const float frac = isnan(f[0]) ? 0.0f : f[5];
        lp->c_masked[i] = L - (int32_t)rintf(frac * (float)L);
        const int32_t r = lp->rid_h[i];
        lp->c_left[i] = lp->K_all[r] - lp->b_h[i] - 1;
        lp->c_total[i] = (int64_t)lp->p_all[r] + (int64_t)lp->K_all[r] * L;
        lp->c_elapsed[i] = lp->now - lp->admit_h[i];
    }
    const double lat = lp->ctl_lat0 + lp->ctl_lat1 * A;
    const int rc = dllm_threshold_control(A, T, lp->ctl_cand.data(), L, lp->feat_h.data(), lp->c_masked.data(),
                                          lp->c_left.data(), lp->c_total.data(), lp->c_elapsed.data(), lp->ctl_slo,
                                          lp->ctl_tps, lat, lp->c_steps.data(), lp->c_cap.data(), lp->c_choice.data());
    if (rc != DLLM_OK) return rc;
    for (int32_t i = 0; i < A; ++i) lp->thr_used[i] = (float)lp->ctl_cand[lp->c_choice[i]];
    return DLLM_OK;
}

}  // namespace

extern "C" size_t dllm_loop_workspace_size(const dllm_loop_config* c, const int32_t* p, const int32_t* K) {
    if (!config_ok(c) || (c->R > 0 && (!p || !K))) return 0;
    dllm_loop tmp;
    tmp.c = *c;
    if (!shapes(c, p, K, &tmp.Kmax, &tmp.Wmax)) return 0;
    return carve(&tmp, nullptr);
}

extern "C" int dllm_loop_create(const dllm_loop_config* c, const int32_t* p, const int32_t* K, const float* thr,
                                const int64_t* prompt_off, const int32_t* prompt_tokens, void* workspace,
                                size_t workspace_bytes, void* stream, dllm_loop** out) {
    if (!out) return DLLM_ERR_INVAL;
    *out = nullptr;
    if (!config_ok(c) || (c->R > 0 && (!p || !K || !thr || !prompt_off))) return DLLM_ERR_INVAL;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DLLM_ERR_WORKSPACE;
    dllm_loop* lp = new dllm_loop();
    lp->c = *c;
    if (!shapes(c, p, K, &lp->Kmax, &lp->Wmax)) {
        delete lp;
        return DLLM_ERR_INVAL;
    }
    if (carve(lp, static_cast<unsigned char*>(workspace)) > workspace_bytes) {
        delete lp;
        return DLLM_ERR_WORKSPACE;
    }
    lp->p_all.assign(p, p + c->R);
    lp->K_all.assign(K, K + c->R);
    lp->thr_all.assign(thr, thr + c->R);
    lp->prompt_off = prompt_off;
    lp->prompt_tokens = prompt_tokens;
    // pending queue: sorted by prompt length, ties by request id
    lp->pending.resize(c->R);
    for (int32_t r = 0; r < c->R; ++r) lp->pending[r] = r;
    std::stable_sort(lp->pending.begin(), lp->pending.end(),
                     [&](int32_t a, int32_t b2) { return lp->p_all[a] < lp->p_all[b2]; });
    lp->pending_p.resize(c->R);
    for (int32_t k = 0; k < c->R; ++k) lp->pending_p[k] = lp->p_all[lp->pending[k]];
    lp->admit_idx.resize(std::max(c->R, 1));
    {
        const size_t cap = (size_t)c->capacity;
        const size_t pinned_bytes = al256(cap) + al256(cap * 4) + al256(cap * 16) + al256(cap * 4) +
                                    cap * DLLM_NUM_FEATURES * 4;
        if (cudaHostAlloc(&lp->pinned, pinned_bytes, cudaHostAllocDefault) != cudaSuccess ||
            cudaEventCreateWithFlags(&lp->staged, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            delete lp;
            return DLLM_ERR_CUDA;
        }
        unsigned char* h = static_cast<unsigned char*>(lp->pinned);
        lp->done_h = h;
        lp->quota_h = reinterpret_cast<int32_t*>(h + al256(cap));
        lp->stage_h = reinterpret_cast<int32_t*>(h + al256(cap) + al256(cap * 4));
        lp->thr_p = reinterpret_cast<float*>(h + al256(cap) + al256(cap * 4) + al256(cap * 16));
        lp->feat_p = reinterpret_cast<float*>(h + al256(cap) + al256(cap * 4) + al256(cap * 16) + al256(cap * 4));
    }
    // the step workspace must start zeroed (its counters are zero at rest)
    const int rc = dllm_workspace_init(lp->step_ws, lp->step_ws_bytes, stream);
    if (rc != DLLM_OK) {
        delete lp;
        return rc;
    }
    *out = lp;
    return DLLM_OK;
}

extern "C" void dllm_loop_destroy(dllm_loop* lp) { delete lp; }

extern "C" int dllm_loop_begin(dllm_loop* lp, void* stream) {
    if (!lp) return DLLM_ERR_INVAL;
    const dllm_loop_config& c = lp->c;
    cudaStream_t s = dllm::as_stream(stream);
    lp->admitted_last = 0;
    // ---- admission and refill (Algorithm 1, "admit"), unless in place ----
    if (!lp->in_place && !lp->pending.empty()) {
        lp->p_act.resize(lp->A);
        for (int32_t i = 0; i < lp->A; ++i) lp->p_act[i] = lp->p_all[lp->rid_h[i]];
        int32_t n = 0;
        int rc = dllm_admit((int32_t)lp->pending.size(), lp->pending_p.data(), lp->A,
                            lp->A ? lp->p_act.data() : nullptr, lp->A ? lp->b_h.data() : nullptr, c.L, c.budget,
                            lp->admit_idx.data(), &n);
        if (rc != DLLM_OK) return rc;
        if (n > 0) {
            if (lp->A + n > c.capacity) return DLLM_ERR_UNSUPPORTED;
            rc = staging_free(lp);
            if (rc != DLLM_OK) return rc;
            int32_t* st = lp->stage_h;
            for (int32_t k = 0; k < n; ++k) {
                const int32_t r = lp->pending[lp->admit_idx[k]];
                st[k] = r;
                st[n + k] = lp->p_all[r];
                st[2 * n + k] = lp->K_all[r];
                memcpy(&st[3 * n + k], &lp->thr_all[r], 4);
            }
            // drop the admitted entries from the queue (indices descending)
            std::vector<int32_t> idx(lp->admit_idx.begin(), lp->admit_idx.begin() + n);
            std::sort(idx.begin(), idx.end(), std::greater<int32_t>());
            for (int32_t k : idx) {
                lp->pending.erase(lp->pending.begin() + k);
                lp->pending_p.erase(lp->pending_p.begin() + k);
            }
            // the admitted rows' (rid, p, K, thr) in one upload
            DLLM_CUDA_TRY(cudaMemcpyAsync(lp->stage_d, st, (size_t)n * 16, cudaMemcpyHostToDevice, s));
            rc = staging_used(lp, s);
            if (rc != DLLM_OK) return rc;
            dllm_refill_args ra;
            memset(&ra, 0, sizeof(ra));
            ra.A0 = lp->A; ra.n = n; ra.L = c.L; ra.mask_id = c.mask_id;
            ra.new_rid = lp->stage_d; ra.new_p = lp->stage_d + n; ra.new_K = lp->stage_d + 2 * n;
            ra.new_thr = reinterpret_cast<const float*>(lp->stage_d + 3 * n);
            ra.rid = lp->rid; ra.p = lp->p; ra.b = lp->b; ra.K = lp->K; ra.thr = lp->thr;
            ra.input_ids = lp->ids; ra.conf_state = lp->cs;
            rc = dllm_refill(&ra, stream);
            if (rc != DLLM_OK) return rc;
            for (int32_t k = 0; k < n; ++k) {
                lp->rid_h.push_back(st[k]);
                lp->b_h.push_back(0);
                lp->s_h.push_back(0);
                lp->wait_h.push_back(0);
                lp->admit_h.push_back(lp->now);
                for (int j = 0; j < DLLM_NUM_FEATURES; ++j)
                    lp->feat_h.push_back(std::numeric_limits<float>::quiet_NaN());
            }
            lp->A += n;
            lp->admitted_last = n;
        }
    }
    // ---- the box of eq. (1) --------------------------------------------------
    dllm_pack_args pa;
    memset(&pa, 0, sizeof(pa));
    pa.A = lp->A; pa.L = c.L; pa.pad_id = c.pad_id;
    pa.p = lp->p; pa.b = lp->b; pa.rid = lp->rid; pa.prompt_off = lp->prompt_off;
    pa.prompt_tokens = lp->prompt_tokens; pa.gen_tokens = lp->gen; pa.ld_gen = (int64_t)lp->Kmax * c.L;
    pa.block_ids = lp->ids; pa.ids = lp->box_ids; pa.attn = lp->box_attn; pa.pos = lp->box_pos;
    pa.pad = lp->box_pad; pa.blk_start = lp->box_blk;
    if (lp->in_place && lp->have_box) {
        pa.W = lp->W;
        ++lp->reloops;
        return dllm_pack_block(&pa, stream);
    }
    lp->p_act.resize(lp->A);
    for (int32_t i = 0; i < lp->A; ++i) lp->p_act[i] = lp->p_all[lp->rid_h[i]];
    int rc = dllm_pack_plan(lp->A, lp->A ? lp->p_act.data() : nullptr, lp->A ? lp->b_h.data() : nullptr, c.L, &lp->W,
                            &lp->cost);
    if (rc != DLLM_OK) return rc;
    lp->have_box = lp->A > 0;
    if (lp->A == 0) return DLLM_OK;
    pa.W = lp->W;
    return dllm_pack(&pa, stream);
}

extern "C" int dllm_loop_end(dllm_loop* lp, const uint16_t* logits, int64_t ldv, void* stream) {
    if (!lp) return DLLM_ERR_INVAL;
    const dllm_loop_config& c = lp->c;
    cudaStream_t s = dllm::as_stream(stream);
    const int32_t A = lp->A;
    if (A == 0) {
        lp->thr_used.clear();
        ++lp->iteration;
        return DLLM_OK;
    }
    // ---- one denoise step over the active rows ---------------------------------
    dllm_step_args sa;
    memset(&sa, 0, sizeof(sa));
    sa.B = A; sa.L = c.L; sa.V = c.V; sa.mask_id = c.mask_id; sa.ldv = ldv; sa.logits = logits;
    sa.input_ids = lp->ids; sa.thr = lp->thr; sa.conf_state = lp->cs; sa.done = lp->done; sa.accept_len = lp->accept;
    sa.n_new = lp->n_new; sa.feats = lp->feats; sa.workspace = lp->step_ws; sa.workspace_bytes = lp->step_ws_bytes;
    int rc;
    const int32_t* quota = nullptr;
    // the thresholds of this step: the controller's, else the requests' own
    lp->thr_used.resize(A);
    if (lp->ctl_on) {
        rc = choose_thresholds(lp, A);
        if (rc != DLLM_OK) return rc;
    } else {
        for (int32_t i = 0; i < A; ++i) lp->thr_used[i] = lp->thr_all[lp->rid_h[i]];
    }
    if (c.S > 0 || lp->ctl_on) {
        rc = staging_free(lp);
        if (rc != DLLM_OK) return rc;
        if (c.S > 0) {
            for (int32_t i = 0; i < A; ++i) lp->quota_h[i] = dllm_transfer_quota(c.L, c.S, lp->s_h[i]);
            DLLM_CUDA_TRY(cudaMemcpyAsync(lp->quota, lp->quota_h, (size_t)A * 4, cudaMemcpyHostToDevice, s));
            quota = lp->quota;
        }
        if (lp->ctl_on) {
            memcpy(lp->thr_p, lp->thr_used.data(), (size_t)A * 4);
            DLLM_CUDA_TRY(cudaMemcpyAsync(lp->thr, lp->thr_p, (size_t)A * 4, cudaMemcpyHostToDevice, s));
        }
        rc = staging_used(lp, s);
        if (rc != DLLM_OK) return rc;
    }
    // FDFO: every done row advances, so the commit and compaction run in
    // the step's own launch (the advance flags are the device's done flags;
    // with none set they leave the batch unchanged)
    const bool fdfo = c.mode == 0;
    if (fdfo) {
        dllm_advance_args aa;
        dllm_compact_args ca;
        commit_args(lp, A, aa, ca);
        rc = dllm_step_commit(&sa, quota, -1, &aa, &ca, stream);
    } else {
        rc = quota ? dllm_step_quota(&sa, quota, stream) : dllm_step(&sa, stream);
    }
    if (rc != DLLM_OK) return rc;
    // the per-step readback: one byte per row (and the block features when
    // the controller needs them)
    DLLM_CUDA_TRY(cudaMemcpyAsync(lp->done_h, lp->done, (size_t)A, cudaMemcpyDeviceToHost, s));
    if (lp->ctl_on)
        DLLM_CUDA_TRY(cudaMemcpyAsync(lp->feat_p, lp->feats, (size_t)A * DLLM_NUM_FEATURES * 4,
                                      cudaMemcpyDeviceToHost, s));
    DLLM_CUDA_TRY(cudaStreamSynchronize(s));
    lp->staged_pending = false;
    if (lp->ctl_on) {
        memcpy(lp->feat_h.data(), lp->feat_p, (size_t)A * DLLM_NUM_FEATURES * 4);
        lp->now += lp->ctl_lat0 + lp->ctl_lat1 * A;
    }
    bool all_done = true, any_done = false;
    for (int32_t i = 0; i < A; ++i) {
        all_done = all_done && lp->done_h[i];
        any_done = any_done || lp->done_h[i];
    }
    // FDFO: every done row advances; sync: all of them once every row is done
    const bool advance = fdfo ? any_done : all_done;
    ++lp->iteration;
    if (!advance) {
        // nothing commits (FDFO: the commit launch changed nothing)
        for (int32_t i = 0; i < A; ++i) {
            if (!lp->wait_h[i]) ++lp->s_h[i];
            lp->wait_h[i] = lp->done_h[i];
        }
        lp->in_place = c.reloop != 0;
        return DLLM_OK;
    }
    lp->in_place = false;
    if (!fdfo) {
        rc = launch_commit(lp, A, stream);
        if (rc != DLLM_OK) return rc;
    }
    // host mirrors: b += 1 and a fresh block for the advanced rows, evict b >= K
    int32_t kept = 0;
    for (int32_t i = 0; i < A; ++i) {
        const bool adv = lp->done_h[i] != 0;
        int32_t bi = lp->b_h[i], si = lp->s_h[i] + (lp->wait_h[i] ? 0 : 1);
        uint8_t wi = 0;
        if (adv) {
            ++bi;
            si = 0;
        }
        if (adv && bi >= lp->K_all[lp->rid_h[i]]) continue;   // evicted
        lp->rid_h[kept] = lp->rid_h[i];
        lp->b_h[kept] = bi;
        lp->s_h[kept] = si;
        lp->wait_h[kept] = wi;
        lp->admit_h[kept] = lp->admit_h[i];
        for (int j = 0; j < DLLM_NUM_FEATURES; ++j)   // a fresh block has nothing unmasked yet
            lp->feat_h[(size_t)kept * DLLM_NUM_FEATURES + j] =
                adv ? std::numeric_limits<float>::quiet_NaN() : lp->feat_h[(size_t)i * DLLM_NUM_FEATURES + j];
        ++kept;
    }
    lp->rid_h.resize(kept);
    lp->b_h.resize(kept);
    lp->s_h.resize(kept);
    lp->wait_h.resize(kept);
    lp->admit_h.resize(kept);
    lp->feat_h.resize((size_t)kept * DLLM_NUM_FEATURES);
    lp->A = kept;
    return DLLM_OK;
}

extern "C" int dllm_loop_info(const dllm_loop* lp, dllm_loop_info_t* out) {
    if (!lp || !out) return DLLM_ERR_INVAL;
    memset(out, 0, sizeof(*out));
    out->A = lp->A;
    out->W = lp->W;
    out->cost = lp->cost;
    out->iteration = lp->iteration;
    out->reloops = lp->reloops;
    out->pending = (int32_t)lp->pending.size();
    out->admitted_last = lp->admitted_last;
    out->finished = lp->pending.empty() && lp->A == 0;
    out->in_place = lp->in_place ? 1 : 0;
    out->ld_gen = (int64_t)lp->Kmax * lp->c.L;
    out->block_ids = lp->ids;
    out->conf_state = lp->cs;
    out->box_ids = lp->box_ids;
    out->box_attn = lp->box_attn;
    out->box_pos = lp->box_pos;
    out->box_pad = lp->box_pad;
    out->box_blk_start = lp->box_blk;
    out->gen_tokens = lp->gen;
    out->done = lp->done;
    out->n_new = lp->n_new;
    out->accept_len = lp->accept;
    out->feats = lp->feats;
    return DLLM_OK;
}

extern "C" int dllm_loop_rows(const dllm_loop* lp, int32_t* rid, int32_t* b, int32_t* s) {
    if (!lp) return DLLM_ERR_INVAL;
    for (int32_t i = 0; i < lp->A; ++i) {
        if (rid) rid[i] = lp->rid_h[i];
        if (b) b[i] = lp->b_h[i];
        if (s) s[i] = lp->s_h[i];
    }
    return DLLM_OK;
}

extern "C" int dllm_loop_set_control(dllm_loop* lp, const dllm_loop_control* ctl) {
    if (!lp) return DLLM_ERR_INVAL;
    if (!ctl) {
        lp->ctl_on = false;
        return DLLM_OK;
    }
    if (ctl->T < 1 || !ctl->candidates || !(ctl->slo_s > 0) || !(ctl->tokens_per_s >= 0) || !(ctl->latency_s >= 0) ||
        !(ctl->latency_per_row_s >= 0))
        return DLLM_ERR_INVAL;
    for (int32_t k = 0; k < ctl->T; ++k) {
        if (!(ctl->candidates[k] == ctl->candidates[k])) return DLLM_ERR_INVAL;   // NaN
        if (k > 0 && !(ctl->candidates[k] > ctl->candidates[k - 1])) return DLLM_ERR_INVAL;
    }
    lp->ctl_cand.assign(ctl->candidates, ctl->candidates + ctl->T);
    lp->ctl_slo = ctl->slo_s;
    lp->ctl_tps = ctl->tokens_per_s;
    lp->ctl_lat0 = ctl->latency_s;
    lp->ctl_lat1 = ctl->latency_per_row_s;
    lp->ctl_on = true;
    return DLLM_OK;
}

extern "C" int dllm_loop_thresholds(const dllm_loop* lp, float* thr, int32_t* n) {
    if (!lp || !n) return DLLM_ERR_INVAL;
    *n = (int32_t)lp->thr_used.size();
    if (thr && !lp->thr_used.empty()) memcpy(thr, lp->thr_used.data(), lp->thr_used.size() * 4);
    return DLLM_OK;
}
