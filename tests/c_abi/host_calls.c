/* Plain-C use of libdllm's host entry points, with no GPU.
 *
 * The header is C (this file compiles under -std=c99 -pedantic -Werror) and
 * the calls that need no device behave as the header documents.  Expected
 * values are hand computations of the pages' definitions:
 *   - BlockServe page, section II-D, eq. (1): Cost(A) = |A| * max_i (p_i +
 *     (b_i + 1) * L), and its sand-fill admission (hand traces);
 *   - BlockServe page, section II-E: the fixed-steps quota, floor(L / S) per
 *     step plus one for each of the first L mod S steps;
 *   - DiLaServe review, section 3.2 item 3: the stand-in step predictor,
 *     worked by hand (P read off the features, max(1, floor(P m)) per step).
 * Exit status 0 when every check holds; each failure is printed. */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "dllm.h"

static int failures = 0;

#define CHECK(cond)                                                            \
    do {                                                                       \
        if (!(cond)) {                                                         \
            fprintf(stderr, "line %d: check failed: %s\n", __LINE__, #cond);   \
            ++failures;                                                        \
        }                                                                      \
    } while (0)

static void check_struct_sizes(void) {
    /* the library's view of every argument struct against this C compiler's */
    CHECK(dllm_struct_size(0) == sizeof(dllm_step_args));
    CHECK(dllm_struct_size(1) == sizeof(dllm_pack_args));
    CHECK(dllm_struct_size(2) == sizeof(dllm_compact_args));
    CHECK(dllm_struct_size(3) == sizeof(dllm_advance_args));
    CHECK(dllm_struct_size(4) == sizeof(dllm_refill_args));
    CHECK(dllm_struct_size(5) == sizeof(dllm_loop_config));
    CHECK(dllm_struct_size(6) == sizeof(dllm_loop_info_t));
    CHECK(dllm_struct_size(7) == sizeof(dllm_vocab_shard));
    CHECK(dllm_struct_size(8) == sizeof(dllm_loop_control));
}

static void check_status_strings(void) {
    int code;
    for (code = DLLM_ERR_SCRATCH_LIMIT; code <= DLLM_OK; ++code) {
        const char* s = dllm_strerror(code);
        CHECK(s != NULL && s[0] != '\0');
    }
    CHECK(strcmp(dllm_strerror(DLLM_OK), dllm_strerror(DLLM_ERR_INVAL)) != 0);
}

static void check_pack_plan(void) {
    /* eq. (1) by hand: widths p + (b + 1) L, cost = A * max width */
    const int32_t p1[2] = {100, 50}, b1[2] = {0, 2};       /* widths 132, 146 */
    const int32_t p2[1] = {1024}, b2[1] = {7};             /* width 1280 */
    const int32_t p3[3] = {2, 3, 5}, b3[3] = {0, 0, 0};    /* L = 4: widths 6, 7, 9 */
    int32_t W = -1;
    int64_t cost = -1;
    CHECK(dllm_pack_plan(2, p1, b1, 32, &W, &cost) == DLLM_OK && W == 146 && cost == 292);
    CHECK(dllm_pack_plan(0, NULL, NULL, 32, &W, &cost) == DLLM_OK && W == 0 && cost == 0);
    CHECK(dllm_pack_plan(1, p2, b2, 32, &W, &cost) == DLLM_OK && W == 1280 && cost == 1280);
    CHECK(dllm_pack_plan(3, p3, b3, 4, &W, &cost) == DLLM_OK && W == 9 && cost == 27);
}

static int admitted(int32_t n_pending, const int32_t* pending, int32_t A, const int32_t* ap, const int32_t* ab,
                    int32_t L, int64_t budget, const int32_t* want, int32_t n_want) {
    int32_t idx[8], n = -1, k;
    if (dllm_admit(n_pending, pending, A, ap, ab, L, budget, idx, &n) != DLLM_OK || n != n_want) return 0;
    for (k = 0; k < n; ++k)
        if (idx[k] != want[k]) return 0;
    return 1;
}

static void check_admit(void) {
    /* from empty, L = 4, budget 30: widths 6, 7, 9 give costs 6, 14, 27; the
     * fourth (p = 9) would cost 4 * 13 = 52 > 30 */
    const int32_t q1[4] = {2, 3, 5, 9}, w1[3] = {0, 1, 2};
    /* active row p = 10, b = 1 (width 18): candidates with p + 4 <= 18 are
     * taken longest first (14, 4, 1: costs 36, 54, 72); then p = 20 widens
     * the box to 24 and 5 * 24 = 120 > 100 */
    const int32_t q2[4] = {1, 4, 14, 20}, ap2[1] = {10}, ab2[1] = {1}, w2[3] = {2, 1, 0};
    /* equal prompts: 1 * 9 <= 9 < 2 * 9; budget 0 admits nothing; equal
     * fitting prompts go earliest first */
    const int32_t q3[3] = {5, 5, 5}, w3[1] = {0};
    const int32_t q4[2] = {3, 3}, ap4[1] = {10}, ab4[1] = {0}, w4[2] = {0, 1};
    CHECK(admitted(4, q1, 0, NULL, NULL, 4, 30, w1, 3));
    CHECK(admitted(4, q2, 1, ap2, ab2, 4, 100, w2, 3));
    CHECK(admitted(3, q3, 0, NULL, NULL, 4, 9, w3, 1));
    CHECK(admitted(3, q3, 0, NULL, NULL, 4, 0, NULL, 0));
    CHECK(admitted(2, q4, 1, ap4, ab4, 4, 1000, w4, 2));
}

static void check_transfer_quota(void) {
    int32_t s;
    for (s = 0; s < 32; ++s) CHECK(dllm_transfer_quota(32, 32, s) == 1);
    /* L = 10 over S = 4 steps: 3, 3, 2, 2; past the schedule everything left */
    CHECK(dllm_transfer_quota(10, 4, 0) == 3 && dllm_transfer_quota(10, 4, 1) == 3);
    CHECK(dllm_transfer_quota(10, 4, 2) == 2 && dllm_transfer_quota(10, 4, 3) == 2);
    CHECK(dllm_transfer_quota(10, 4, 4) == 10);
    CHECK(dllm_transfer_quota(0, 4, 0) == -1 && dllm_transfer_quota(10, 0, 0) == -1);
    CHECK(dllm_transfer_quota(10, 4, -1) == -1);
}

static void check_step_predictor(void) {
    /* t = 0.7 on features (min .5, q25 .6, median .8, avg, q75 .9, frac):
     * F = .25 + (.7 - .6) / (.8 - .6) * .25 = .375, P = .625; 5 masked:
     * 5 -> 2 -> 1 -> 0 is 3 steps; a block of L = 8: 8 -> 3 -> 2 -> 1 -> 0,
     * 4 steps; 2 blocks left: 3 + 2 * 4 = 11.  With nothing unmasked (NaN features) at
     * t = .5, P = .5; 8 masked, L = 8, 3 blocks left: 4 + 3 * 4 = 16 */
    const double cand[1] = {0.7}, cand2[1] = {0.5};
    const float f[6] = {0.5f, 0.6f, 0.8f, 0.7f, 0.9f, 0.25f};
    float g[6];
    const int32_t m1[1] = {5}, k1[1] = {2}, m2[1] = {8}, k2[1] = {3};
    double steps = -1.0;
    int j;
    for (j = 0; j < 5; ++j) g[j] = (float)NAN;
    g[5] = 0.0f;
    CHECK(dllm_predict_steps_stub(1, 1, cand, 8, f, m1, k1, &steps) == DLLM_OK && steps == 11.0);
    CHECK(dllm_predict_steps_stub(1, 1, cand, 4, f, m1, k1, &steps) == DLLM_ERR_INVAL);   /* 5 masked > L */
    CHECK(dllm_predict_steps_stub(1, 1, cand2, 8, g, m2, k2, &steps) == DLLM_OK && steps == 16.0);
    CHECK(dllm_predict_steps_stub(1, 0, cand, 4, f, m1, k1, &steps) == DLLM_ERR_INVAL);
}

static void check_step_host_checks(void) {
    /* argument checks run before any CUDA call */
    dllm_step_args a;
    CHECK(dllm_step(NULL, NULL) == DLLM_ERR_INVAL);
    memset(&a, 0, sizeof(a));
    a.B = 0;
    a.L = 32;
    a.V = 1024;
    a.ldv = 1024;
    CHECK(dllm_step(&a, NULL) == DLLM_OK);   /* an empty batch launches nothing */
    a.L = 0;
    CHECK(dllm_step(&a, NULL) == DLLM_ERR_INVAL);
    CHECK(dllm_step_workspace_size(128, 32, 151936) > 0);
    CHECK(dllm_step_workspace_size(128, 32, 151936 + 8192 * 3) > dllm_step_workspace_size(128, 32, 151936));
}

int main(void) {
    CHECK(dllm_abi_version() == DLLM_ABI_VERSION);
    check_struct_sizes();
    check_status_strings();
    check_pack_plan();
    check_admit();
    check_transfer_quota();
    check_step_predictor();
    check_step_host_checks();
    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    printf("host calls from C: ok\n");
    return 0;
}
