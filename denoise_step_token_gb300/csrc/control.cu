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
    // worst case = committed + load[i][k] + rest[i], rest[i] = the later
    // requests at the lowest threshold summed from the back:
    // rest[R-1] = 0, rest[i] = load[i+1][0] + rest[i+1]
    std::vector<double> rest_of((size_t)R, 0.0);
    for (int32_t i = R - 2; i >= 0; --i) rest_of[i] = load[(long long)(i + 1) * T] + rest_of[i + 1];
    double committed = 0.0;
    for (int32_t i = 0; i < R; ++i) {
        const double rest = rest_of[i];
        int32_t keep = 0;
        for (int32_t k = T - 1; k >= 0; --k) {
            const double worst = committed + load[(long long)i * T + k] + rest;
            if (worst <= capacity) {
                keep = k;
                break;
            }
        }
        max_allowed[i] = keep;
        committed += load[(long long)i * T + keep];
    }
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
        int32_t pick = 0;
        for (int32_t k = top; k >= 0; --k) {
            if (rem_steps[(long long)i * T + k] * step_latency[i] <= slo_left[i]) {
                pick = k;
                break;
            }
        }
        choice[i] = pick;
    }
    return DLLM_OK;
}
