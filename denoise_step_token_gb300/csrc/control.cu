// Host-side confidence-threshold control (DiLaServe review, section 3.2,
// "Confidence Threshold Controller"): a stand-in step predictor over the
// step's block features, Algorithm 2 (adaptive load control) and
// Algorithm 1 (SLO-aware threshold choice).  Plain host arithmetic in
// double precision; the build turns off floating-point contraction so the
// results do not depend on the host compiler's fused multiply-add.

#include <math.h>
#include <stdint.h>

#include <vector>

#include "dllm.h"

namespace {

// P(confidence > t) from the block's features: a piecewise-linear
// distribution through (min, 0), (q25, .25), (median, .5), (q75, .75),
// (1, 1); uniform on [0, 1] when no position is unmasked yet (NaN).
double rate_above(double t, const float* f) {
    const double mn = f[0];
    if (isnan(mn)) return fmin(1.0, fmax(0.0, 1.0 - t));
    const double xs[5] = {mn, (double)f[1], (double)f[2], (double)f[4], 1.0};
    const double ps[5] = {0.0, 0.25, 0.5, 0.75, 1.0};
    if (t < xs[0]) return 1.0;
    if (t >= xs[4]) return 0.0;
    double F = 1.0;
    for (int k = 0; k < 4; ++k) {
        if (xs[k] <= t && t < xs[k + 1]) {
            const double q = (t - xs[k]) / (xs[k + 1] - xs[k]);
            F = ps[k] + q * (ps[k + 1] - ps[k]);
            break;
        }
    }
    return 1.0 - F;
}

// Steps to unmask m positions when a step unmasks a fraction P of those
// still masked, at least one: m <- m - max(1, floor(P m)).
long long steps_to_clear(long long m, double P) {
    long long n = 0;
    while (m > 0) {
        const long long take = (long long)floor(P * (double)m);
        m -= take > 1 ? take : 1;
        ++n;
    }
    return n;
}

// Algorithm 2 over load(i, k): the index of each request's highest allowed
// threshold.  worst case = committed + load(i, k) + rest[i], rest[i] = the
// later requests at the lowest threshold summed from the back:
// rest[R-1] = 0, rest[i] = load(i+1, 0) + rest[i+1].
template <typename Load>
void load_control_core(int32_t R, int32_t T, Load load, double capacity, int32_t* max_allowed) {
    std::vector<double> rest_of((size_t)R, 0.0);
    for (int32_t i = R - 2; i >= 0; --i) rest_of[i] = load(i + 1, 0) + rest_of[i + 1];
    double committed = 0.0;
    for (int32_t i = 0; i < R; ++i) {
        const double rest = rest_of[i];
        int32_t keep = 0;
        for (int32_t k = T - 1; k >= 0; --k) {
            const double worst = committed + load(i, k) + rest;
            if (worst <= capacity) {
                keep = k;
                break;
            }
        }
        max_allowed[i] = keep;
        committed += load(i, keep);
    }
}

// Algorithm 1 for request i: the highest k <= top whose remaining latency
// rem_steps[k] * step_latency fits slo_left, else 0.
int32_t slo_pick(int32_t top, const double* rem_steps, double step_latency, double slo_left) {
    for (int32_t k = top; k >= 0; --k)
        if (rem_steps[k] * step_latency <= slo_left) return k;
    return 0;
}

}  // namespace

extern "C" int dllm_predict_steps_stub(int32_t R, int32_t T, const double* cand, int32_t L, const float* feats,
                                       const int32_t* masked, const int32_t* blocks_left, double* steps_out) {
    if (R < 0 || T < 1 || L < 1) return DLLM_ERR_INVAL;
    if (R == 0) return DLLM_OK;
    if (!cand || !feats || !masked || !blocks_left || !steps_out) return DLLM_ERR_INVAL;
    for (int32_t i = 0; i < R; ++i) {
        if (masked[i] < 0 || masked[i] > L || blocks_left[i] < 0) return DLLM_ERR_INVAL;
        for (int32_t k = 0; k < T; ++k) {
            const double P = rate_above(cand[k], feats + (long long)i * DLLM_NUM_FEATURES);
            steps_out[(long long)i * T + k] =
                (double)(steps_to_clear(masked[i], P) + (long long)blocks_left[i] * steps_to_clear(L, P));
        }
    }
    return DLLM_OK;
}

extern "C" int dllm_load_control(int32_t R, int32_t T, const double* load, double capacity, int32_t* max_allowed) {
    if (R < 0 || T < 1) return DLLM_ERR_INVAL;
    if (R == 0) return DLLM_OK;
    if (!load || !max_allowed) return DLLM_ERR_INVAL;
    load_control_core(R, T, [&](int32_t i, int32_t k) { return load[(long long)i * T + k]; }, capacity,
                      max_allowed);
    return DLLM_OK;
}

extern "C" int dllm_slo_thresholds(int32_t R, int32_t T, const double* rem_steps, const double* step_latency,
                                   const double* slo_left, const int32_t* max_allowed, int32_t* choice) {
    if (R < 0 || T < 1) return DLLM_ERR_INVAL;
    if (R == 0) return DLLM_OK;
    if (!rem_steps || !step_latency || !slo_left || !choice) return DLLM_ERR_INVAL;
    for (int32_t i = 0; i < R; ++i) {
        const int32_t top = max_allowed ? max_allowed[i] : T - 1;
        if (top < 0 || top >= T) return DLLM_ERR_INVAL;
    }
    for (int32_t i = 0; i < R; ++i)
        choice[i] = slo_pick(max_allowed ? max_allowed[i] : T - 1, rem_steps + (long long)i * T, step_latency[i],
                             slo_left[i]);
    return DLLM_OK;
}

extern "C" int dllm_threshold_control(int32_t R, int32_t T, const double* cand, int32_t L, const float* feats,
                                      const int32_t* masked, const int32_t* blocks_left,
                                      const int64_t* total_tokens, const double* elapsed_s, double slo_s,
                                      double tokens_per_s, double step_latency_s, double* steps_out,
                                      int32_t* max_allowed, int32_t* choice) {
    if (R < 0 || T < 1 || L < 1) return DLLM_ERR_INVAL;
    if (R == 0) return DLLM_OK;
    if (!total_tokens || !elapsed_s || !steps_out || !max_allowed || !choice) return DLLM_ERR_INVAL;
    for (int32_t i = 0; i < R; ++i)
        if (total_tokens[i] < 0) return DLLM_ERR_INVAL;
    // item ③: remaining steps per candidate threshold
    const int rc = dllm_predict_steps_stub(R, T, cand, L, feats, masked, blocks_left, steps_out);
    if (rc != DLLM_OK) return rc;
    // item ②: load = total tokens x remaining steps, capacity = tokens/s x SLO
    load_control_core(
        R, T, [&](int32_t i, int32_t k) { return steps_out[(long long)i * T + k] * (double)total_tokens[i]; },
        tokens_per_s * slo_s, max_allowed);
    // item ①: the highest allowed threshold whose remaining latency fits the
    // SLO left since the request arrived
    for (int32_t i = 0; i < R; ++i)
        choice[i] = slo_pick(max_allowed[i], steps_out + (long long)i * T, step_latency_s, slo_s - elapsed_s[i]);
    return DLLM_OK;
}
