/*
 * synth.c -- seeded, counter-based synthetic inputs.
 *
 * This module only draws random numbers and rounds them to the storage types
 * the workloads name (FP32 -> BF16 round-to-nearest-even, integer codes).  It
 * holds none of the entropy-coding or GEMV arithmetic: both the CPU oracle and
 * the CUDA library receive the arrays produced here as plain inputs.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used in counter form: output number n of a
 * stream seeded with s is mix(s + (n + 1) * 0x9E3779B97F4A7C15), which equals
 * the (n+1)-th call of the sequential generator started from state s.  Every
 * element therefore depends only on (seed, index), so any index range can be
 * filled independently (and in parallel) with identical results.
 *
 * Normal deviates: Box-Muller on pairs (u1 in (0,1], u2 in [0,1)); element 2k
 * takes r*cos(2*pi*u2), element 2k+1 takes r*sin(2*pi*u2).
 *
 * Build with -ffp-contract=off so no multiply-add is fused differently on
 * different hosts.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Output number n (0-based) of the SplitMix64 stream seeded with s. */
uint64_t synth_sm64(uint64_t s, uint64_t n) { return sm64_mix(s + (n + 1) * SM64_GAMMA); }

/* Independent sub-stream seed: output number `tag` of the stream seeded with s. */
uint64_t synth_subseed(uint64_t s, uint64_t tag) { return synth_sm64(s, tag); }

static inline double u01_open0(uint64_t h) { /* (0, 1] */
    return (double)((h >> 11) + 1) * (1.0 / 9007199254740992.0);
}
static inline double u01(uint64_t h) { /* [0, 1) */
    return (double)(h >> 11) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t s, uint64_t i) {
    const uint64_t k = i >> 1;
    const double u1 = u01_open0(synth_sm64(s, 2 * k));
    const double u2 = u01(synth_sm64(s, 2 * k + 1));
    const double r = sqrt(-2.0 * log(u1));
    const double t = 6.283185307179586 * u2;
    return (i & 1) ? r * sin(t) : r * cos(t);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40); /* quiet NaN */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------------------
 * Parallel-for over an index range with pthreads.
 * ------------------------------------------------------------------------- */
typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct {
    range_fn fn;
    void* ctx;
    int64_t lo, hi;
} range_job;

static void* range_thread(void* p) {
    range_job* j = (range_job*)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < (int64_t)nthreads * 65536) nthreads = (int)(n / 65536) + 1;
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t th[256];
    range_job jobs[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].lo = n * t / nthreads;
        jobs[t].hi = n * (t + 1) / nthreads;
        if (pthread_create(&th[t], NULL, range_thread, &jobs[t]) == 0) {
            started = t + 1;
        } else {
            fn(ctx, jobs[t].lo, jobs[t].hi);
            started = t;
            for (int u = t + 1; u < nthreads; ++u) fn(ctx, n * u / nthreads, n * (u + 1) / nthreads);
            break;
        }
    }
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------------------
 * Plain streams.
 * ------------------------------------------------------------------------- */
typedef struct {
    uint64_t seed, offset;
    double scale;
    void* out;
} stream_ctx;

static void fill_normal_f64(void* c, int64_t lo, int64_t hi) {
    stream_ctx* s = (stream_ctx*)c;
    double* o = (double*)s->out;
    for (int64_t i = lo; i < hi; ++i) o[i] = normal_at(s->seed, s->offset + (uint64_t)i);
}
static void fill_uniform_f64(void* c, int64_t lo, int64_t hi) {
    stream_ctx* s = (stream_ctx*)c;
    double* o = (double*)s->out;
    for (int64_t i = lo; i < hi; ++i) o[i] = u01(synth_sm64(s->seed, s->offset + (uint64_t)i));
}
static void fill_gauss_bf16(void* c, int64_t lo, int64_t hi) {
    stream_ctx* s = (stream_ctx*)c;
    uint16_t* o = (uint16_t*)s->out;
    for (int64_t i = lo; i < hi; ++i) o[i] = f32_to_bf16_rne((float)(s->scale * normal_at(s->seed, s->offset + (uint64_t)i)));
}

/* z_i, i in [offset, offset+n), as double. */
void synth_normal_f64(uint64_t seed, uint64_t offset, int64_t n, double* out, int nthreads) {
    stream_ctx c = {seed, offset, 1.0, out};
    parallel_for(n, nthreads, fill_normal_f64, &c);
}

/* u_i in [0, 1), i in [offset, offset+n). */
void synth_uniform_f64(uint64_t seed, uint64_t offset, int64_t n, double* out, int nthreads) {
    stream_ctx c = {seed, offset, 1.0, out};
    parallel_for(n, nthreads, fill_uniform_f64, &c);
}

/* bf16(float(std * z_i)) for i in [0, n). */
void synth_gauss_bf16(uint64_t seed, int64_t n, double std_, uint16_t* out, int nthreads) {
    stream_ctx c = {seed, 0, std_, out};
    parallel_for(n, nthreads, fill_gauss_bf16, &c);
}

/* ---------------------------------------------------------------------------
 * Llama-shaped weights: w_ij = s_i * z_ij with s_i = base_std * exp(ln_sigma * zr_i),
 * then exactly round(outlier_frac * N * K) positions (a seeded partial
 * Fisher-Yates prefix of [0, N*K)) are replaced by outlier_std * zo_t.
 * Stored as bf16(float(value)).  Sub-streams: 1 = weights, 2 = row scales,
 * 3 = outlier positions, 4 = outlier values.
 * ------------------------------------------------------------------------- */
typedef struct {
    uint64_t seed_w;
    int64_t K;
    const double* row_std;
    uint16_t* out;
} llama_ctx;

static void fill_llama(void* c, int64_t lo, int64_t hi) {
    llama_ctx* s = (llama_ctx*)c;
    for (int64_t i = lo; i < hi; ++i) {
        const double v = s->row_std[i / s->K] * normal_at(s->seed_w, (uint64_t)i);
        s->out[i] = f32_to_bf16_rne((float)v);
    }
}

/* Open-addressing map int64 -> int64 for the virtual Fisher-Yates array. */
typedef struct {
    int64_t* keys;
    int64_t* vals;
    uint64_t mask;
} i64map;

static int map_init(i64map* m, int64_t want) {
    uint64_t cap = 16;
    while (cap < (uint64_t)want * 4) cap <<= 1;
    m->keys = (int64_t*)malloc(cap * sizeof(int64_t));
    m->vals = (int64_t*)malloc(cap * sizeof(int64_t));
    if (!m->keys || !m->vals) {
        free(m->keys);
        free(m->vals);
        return -1;
    }
    for (uint64_t i = 0; i < cap; ++i) m->keys[i] = -1;
    m->mask = cap - 1;
    return 0;
}
static uint64_t map_slot(const i64map* m, int64_t k) {
    uint64_t h = sm64_mix((uint64_t)k) & m->mask;
    while (m->keys[h] != -1 && m->keys[h] != k) h = (h + 1) & m->mask;
    return h;
}
static int64_t map_get(const i64map* m, int64_t k) {
    uint64_t h = map_slot(m, k);
    return m->keys[h] == -1 ? k : m->vals[h];
}
static void map_set(i64map* m, int64_t k, int64_t v) {
    uint64_t h = map_slot(m, k);
    m->keys[h] = k;
    m->vals[h] = v;
}

/* Writes the m chosen positions to pos_out (may be NULL). Returns m or -1. */
int64_t synth_llama_bf16(uint64_t seed, int64_t N, int64_t K, double base_std, double ln_sigma,
                         double outlier_frac, double outlier_std, uint16_t* out, int64_t* pos_out,
                         int nthreads) {
    if (N < 0 || K < 0) return -1;
    const int64_t NK = N * K;
    double* row_std = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!row_std) return -1;
    const uint64_t s_w = synth_subseed(seed, 1), s_r = synth_subseed(seed, 2);
    const uint64_t s_p = synth_subseed(seed, 3), s_v = synth_subseed(seed, 4);
    for (int64_t i = 0; i < N; ++i) row_std[i] = base_std * exp(ln_sigma * normal_at(s_r, (uint64_t)i));
    llama_ctx c = {s_w, K > 0 ? K : 1, row_std, out};
    parallel_for(NK, nthreads, fill_llama, &c);
    free(row_std);

    const int64_t m = (int64_t)llround(outlier_frac * (double)NK);
    if (m <= 0 || NK == 0) return 0;
    i64map map;
    if (map_init(&map, m) != 0) return -1;
    for (int64_t i = 0; i < m; ++i) {
        const uint64_t range = (uint64_t)(NK - i);
        const uint64_t r = (uint64_t)(((unsigned __int128)synth_sm64(s_p, (uint64_t)i) * range) >> 64);
        const int64_t j = i + (int64_t)r;
        const int64_t vi = map_get(&map, i), vj = map_get(&map, j);
        map_set(&map, i, vj);
        map_set(&map, j, vi);
        const int64_t p = vj; /* element now at slot i */
        if (pos_out) pos_out[i] = p;
        out[p] = f32_to_bf16_rne((float)(outlier_std * normal_at(s_v, (uint64_t)i)));
    }
    free(map.keys);
    free(map.vals);
    return m;
}

/* ---------------------------------------------------------------------------
 * Quantized codes: clip(round_half_even(std * z_i), lo, hi) as int8.
 * ------------------------------------------------------------------------- */
typedef struct {
    uint64_t seed;
    double std_;
    int lo, hi;
    int8_t* out;
} codes_ctx;

static void fill_codes(void* c, int64_t lo, int64_t hi) {
    codes_ctx* s = (codes_ctx*)c;
    for (int64_t i = lo; i < hi; ++i) {
        double v = nearbyint(s->std_ * normal_at(s->seed, (uint64_t)i)); /* default mode: ties to even */
        if (v < s->lo) v = s->lo;
        if (v > s->hi) v = s->hi;
        s->out[i] = (int8_t)v;
    }
}

void synth_codes_i8(uint64_t seed, int64_t n, double std_, int lo, int hi, int8_t* out, int nthreads) {
    codes_ctx c = {seed, std_, lo, hi, out};
    parallel_for(n, nthreads, fill_codes, &c);
}
