/*
 * synth.c -- seeded synthetic inputs for the elementwise / row ops.
 *
 * This module only draws numbers.  It holds none of the arithmetic of the ops
 * (no norm, rotation, activation, gather, sum or max): both the oracle checks
 * and the CUDA path receive the arrays it produces, and nothing else is shared
 * between them.
 *
 * Generator: splitmix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  A stream is named by
 * (seed, stream id); its k-th 64-bit output is the splitmix64 finaliser of
 * key + (k+1)*gamma, which is exactly the sequential splitmix64 sequence that
 * starts from state `key`.  Because output k depends only on (key, k), any
 * slice of a stream can be drawn on its own and by any number of threads with
 * identical results.
 *
 *   uniform double in [0,1)  : top 53 bits * 2^-53
 *   normal N(m, s)           : Box-Muller on outputs 2k and 2k+1 (cosine
 *                              branch only), s is the standard deviation,
 *                              optionally clipped at +-clip standard deviations
 *   integers U[a, b)         : a + floor(u * (b - a))
 *   f32                      : the double value rounded to nearest by a cast
 *   bf16                     : f32 rounded to nearest-even on the top 16 bits
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t syn_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Starting state of stream `stream` under `seed`. */
static uint64_t syn_key(uint64_t seed, uint64_t stream) {
    return syn_mix(syn_mix(seed + SYN_GAMMA) ^ (stream * 0xD1B54A32D192ED03ULL + 1ULL));
}

static inline uint64_t syn_draw(uint64_t key, uint64_t k) {
    return syn_mix(key + (k + 1ULL) * SYN_GAMMA);
}

static inline double syn_unit(uint64_t z) { return (double)(z >> 11) * 0x1.0p-53; }

/* ---- threading: split [0, n) into contiguous slices ------------------------ */

typedef struct {
    int kind;
    uint64_t key;
    int64_t offset, begin, end;
    double a, b, c;
    void *out;
    const void *in;
} syn_job;

enum { JOB_NORMAL = 0, JOB_UNIFORM = 1, JOB_INT = 2, JOB_UNIT = 3, JOB_BF16 = 4, JOB_U64 = 5 };

static uint16_t syn_round_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static void *syn_worker(void *arg) {
    syn_job *j = (syn_job *)arg;
    for (int64_t i = j->begin; i < j->end; ++i) {
        uint64_t k = (uint64_t)(j->offset + i);
        switch (j->kind) {
        case JOB_NORMAL: {
            double u1 = syn_unit(syn_draw(j->key, 2 * k));
            double u2 = syn_unit(syn_draw(j->key, 2 * k + 1));
            double z = sqrt(-2.0 * log(1.0 - u1)) * cos(6.283185307179586 * u2);
            if (j->c > 0.0) {
                if (z > j->c) z = j->c;
                if (z < -j->c) z = -j->c;
            }
            ((float *)j->out)[i] = (float)(j->a + j->b * z);
            break;
        }
        case JOB_UNIFORM: {
            double u = syn_unit(syn_draw(j->key, k));
            ((float *)j->out)[i] = (float)(j->a + (j->b - j->a) * u);
            break;
        }
        case JOB_INT: {
            double u = syn_unit(syn_draw(j->key, k));
            int64_t lo = (int64_t)j->a, span = (int64_t)j->b - (int64_t)j->a;
            int64_t v = lo + (int64_t)floor(u * (double)span);
            if (v >= lo + span) v = lo + span - 1;
            ((int32_t *)j->out)[i] = (int32_t)v;
            break;
        }
        case JOB_UNIT:
            ((double *)j->out)[i] = syn_unit(syn_draw(j->key, k));
            break;
        case JOB_U64:
            ((uint64_t *)j->out)[i] = syn_draw(j->key, k);
            break;
        case JOB_BF16:
            ((uint16_t *)j->out)[i] = syn_round_bf16(((const float *)j->in)[i]);
            break;
        }
    }
    return NULL;
}

#define SYN_MAX_THREADS 128

static void syn_run(syn_job proto, int64_t n, int nthreads) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > SYN_MAX_THREADS) nthreads = SYN_MAX_THREADS;
    if (n < 65536) nthreads = 1;
    syn_job jobs[SYN_MAX_THREADS];
    pthread_t tid[SYN_MAX_THREADS];
    int started[SYN_MAX_THREADS];
    int64_t per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].begin = (int64_t)t * per;
        jobs[t].end = jobs[t].begin + per < n ? jobs[t].begin + per : n;
        started[t] = 0;
        if (jobs[t].begin >= jobs[t].end) continue;
        if (t > 0 && pthread_create(&tid[t], NULL, syn_worker, &jobs[t]) == 0) started[t] = 1;
    }
    /* slice 0, and any slice whose thread could not start, runs here */
    for (int t = 0; t < nthreads; ++t)
        if (!started[t] && jobs[t].begin < jobs[t].end) syn_worker(&jobs[t]);
    for (int t = 1; t < nthreads; ++t)
        if (started[t]) pthread_join(tid[t], NULL);
}

/* ---- exported ------------------------------------------------------------- */

/* out[i] = mean + std * z_(offset+i), z standard normal, clipped at +-clip (clip <= 0: none). */
void syn_normal_f32(uint64_t seed, uint64_t stream, int64_t offset, int64_t n, double mean,
                    double std, double clip, float *out, int nthreads) {
    syn_job j = {JOB_NORMAL, syn_key(seed, stream), offset, 0, 0, mean, std, clip, out, NULL};
    syn_run(j, n, nthreads);
}

/* out[i] = lo + (hi - lo) * u_(offset+i) rounded to f32. */
void syn_uniform_f32(uint64_t seed, uint64_t stream, int64_t offset, int64_t n, double lo,
                     double hi, float *out, int nthreads) {
    syn_job j = {JOB_UNIFORM, syn_key(seed, stream), offset, 0, 0, lo, hi, 0.0, out, NULL};
    syn_run(j, n, nthreads);
}

/* out[i] uniform integer in [lo, hi). */
void syn_randint_i32(uint64_t seed, uint64_t stream, int64_t offset, int64_t n, int64_t lo,
                     int64_t hi, int32_t *out, int nthreads) {
    syn_job j = {JOB_INT, syn_key(seed, stream), offset, 0, 0, (double)lo, (double)hi, 0.0, out, NULL};
    syn_run(j, n, nthreads);
}

/* out[i] = u_(offset+i), uniform double in [0, 1). */
void syn_unit_f64(uint64_t seed, uint64_t stream, int64_t offset, int64_t n, double *out,
                  int nthreads) {
    syn_job j = {JOB_UNIT, syn_key(seed, stream), offset, 0, 0, 0.0, 0.0, 0.0, out, NULL};
    syn_run(j, n, nthreads);
}

/* Raw 64-bit outputs (used by the generator's own self-test against splitmix64). */
void syn_raw_u64(uint64_t seed, uint64_t stream, int64_t offset, int64_t n, uint64_t *out) {
    syn_job j = {JOB_U64, syn_key(seed, stream), offset, 0, 0, 0.0, 0.0, 0.0, out, NULL};
    syn_run(j, n, 1);
}

/* The starting state of a stream, so a test can replay it with plain splitmix64. */
uint64_t syn_stream_key(uint64_t seed, uint64_t stream) { return syn_key(seed, stream); }

/* Storage rounding of generated f32 values to bf16 bit patterns. */
void syn_f32_to_bf16(const float *in, uint16_t *out, int64_t n, int nthreads) {
    syn_job j = {JOB_BF16, 0, 0, 0, 0, 0.0, 0.0, 0.0, out, in};
    syn_run(j, n, nthreads);
}
