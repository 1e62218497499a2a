/*
 * Seeded synthetic logits generator (test and benchmark input only).
 *
 * This file is the bulk half of the input generator that both the CUDA path
 * and the CPU oracle consume.  It holds none of the denoise step's arithmetic:
 * every output element is a table lookup addressed by a counter-based hash.
 *
 * Definition (the Python half in synth/__init__.py builds the tables and the
 * per-row keys and documents the distributions):
 *
 *   mix(z)         SplitMix64 output function (Steele, Lea & Flood, "Fast
 *                  splittable pseudorandom number generators", OOPSLA 2014):
 *                  z ^= z >> 30; z *= 0xbf58476d1ce4e5b9;
 *                  z ^= z >> 27; z *= 0x94d049bb133111eb; z ^= z >> 31.
 *   out(key, k)    the k-th SplitMix64 output of a stream seeded with key:
 *                  mix(key + (k + 1) * 0x9e3779b97f4a7c15).
 *
 *   For a row with key K and vocabulary V:
 *     element v          bg_table[out(K, v + 1) & 0xffff]
 *     planted peak       h = out(K, 0); token t = (h >> 16) % (V - 1), shifted
 *                        past mask_col when t >= mask_col; value
 *                        peak_table[h & 0xffff]
 *     column mask_col    bf16 -30.0 (0xc1f0), when 0 <= mask_col < V
 *   Columns [V, ldv) of a row are left untouched.
 *
 * Values are raw bf16 bit patterns (uint16).  Pure integer code, so x86 and
 * Arm builds give identical bytes.
 */
#include <stdint.h>
#include <stddef.h>
#include <pthread.h>

#define SYNTH_GAMMA 0x9e3779b97f4a7c15ULL
#define SYNTH_BF16_MINUS_30 ((uint16_t)0xc1f0u)

static inline uint64_t synth_mix(uint64_t z) {
    z ^= z >> 30;
    z *= 0xbf58476d1ce4e5b9ULL;
    z ^= z >> 27;
    z *= 0x94d049bb133111ebULL;
    z ^= z >> 31;
    return z;
}

static inline uint64_t synth_out(uint64_t key, uint64_t k) {
    return synth_mix(key + (k + 1u) * SYNTH_GAMMA);
}

uint64_t synth_splitmix_out(uint64_t key, uint64_t k) { return synth_out(key, k); }

typedef struct {
    uint16_t* out;
    int64_t ldv;
    int64_t V;
    const int64_t* dst_row;
    const uint64_t* row_key;
    const uint16_t* bg_table;
    const uint16_t* peak_table;
    int64_t mask_col;
    int64_t r0, r1;
} synth_job;

static void synth_fill_row(const synth_job* j, int64_t r) {
    uint16_t* row = j->out + j->dst_row[r] * j->ldv;
    const uint64_t key = j->row_key[r];
    const int64_t V = j->V;
    for (int64_t v = 0; v < V; ++v) {
        row[v] = j->bg_table[synth_out(key, (uint64_t)v + 1u) & 0xffffu];
    }
    if (V > 1) {
        const uint64_t h = synth_out(key, 0);
        int64_t t = (int64_t)((h >> 16) % (uint64_t)(V - 1));
        if (j->mask_col >= 0 && j->mask_col < V && t >= j->mask_col) t += 1;
        row[t] = j->peak_table[h & 0xffffu];
    }
    if (j->mask_col >= 0 && j->mask_col < V) row[j->mask_col] = SYNTH_BF16_MINUS_30;
}

static void* synth_worker(void* arg) {
    const synth_job* j = (const synth_job*)arg;
    for (int64_t r = j->r0; r < j->r1; ++r) synth_fill_row(j, r);
    return NULL;
}

/*
 * Fill n_rows rows of `out` (row stride ldv elements).  Row r of the request
 * list is written at out + dst_row[r] * ldv from key row_key[r].
 * Returns 0, or -1 on bad arguments.
 */
int synth_logits_rows(uint16_t* out, int64_t ldv, int64_t V, int64_t n_rows,
                      const int64_t* dst_row, const uint64_t* row_key,
                      const uint16_t* bg_table, const uint16_t* peak_table,
                      int64_t mask_col, int nthreads) {
    if (!out || !dst_row || !row_key || !bg_table || !peak_table) return -1;
    if (V < 1 || ldv < V || n_rows < 0) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n_rows) nthreads = n_rows > 0 ? (int)n_rows : 1;
    synth_job jobs[256];
    pthread_t tid[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].out = out; jobs[t].ldv = ldv; jobs[t].V = V;
        jobs[t].dst_row = dst_row; jobs[t].row_key = row_key;
        jobs[t].bg_table = bg_table; jobs[t].peak_table = peak_table;
        jobs[t].mask_col = mask_col;
        jobs[t].r0 = n_rows * t / nthreads;
        jobs[t].r1 = n_rows * (t + 1) / nthreads;
        started[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&tid[t], NULL, synth_worker, &jobs[t]) == 0;
    synth_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(tid[t], NULL);
        else synth_worker(&jobs[t]);
    }
    return 0;
}
