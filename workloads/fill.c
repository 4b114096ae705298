/*
 * Seeded synthetic values for the paged-decode workloads.
 *
 * This file only makes random numbers and converts them to the storage
 * types. It holds none of the attention arithmetic: no dot products, no
 * softmax, no page-table walk. Both the CPU oracle and the CUDA path are fed
 * from these bytes.
 *
 * Draw e of a stream with key k:
 *   u1 = U(splitmix64 output 2e), u2 = U(splitmix64 output 2e+1), both in (0, 1]
 *   x  = sqrt(-2 ln u1) * cos(2 pi u2)                      (Box-Muller, cosine branch)
 *   stored value = RNE(float(x)) to the storage type.
 * splitmix64 is Steele, Lea and Flood's generator (OOPSLA 2014): the n-th
 * output for seed k is the mix of k + n * 0x9E3779B97F4A7C15 (n counted from 1).
 * Because every draw depends only on (key, e), any slice of a stream can be
 * produced on any thread and the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t sm64_at(uint64_t key, uint64_t n) {
    uint64_t z = key + (n + 1u) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* 53 random bits mapped onto (0, 1]: never 0, so the log is finite. */
static inline double unit_open0(uint64_t r) {
    return ((double)(r >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

static inline float normal_at(uint64_t key, uint64_t e) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = unit_open0(sm64_at(key, 2u * e));
    double u2 = unit_open0(sm64_at(key, 2u * e + 1u));
    return (float)(sqrt(-2.0 * log(u1)) * cos(two_pi * u2));
}

/* float -> bfloat16, round to nearest even (NaN kept quiet). */
static inline uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* float -> IEEE binary16, round to nearest even, overflow to infinity. */
static inline uint16_t f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) return (uint16_t)(sign | (ax > 0x7f800000u ? 0x7e00u : 0x7c00u));
    if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u); /* >= 65520 rounds to inf */
    if (ax < 0x38800000u) {                                   /* below 2^-14: subnormal or 0 */
        float v;
        memcpy(&v, &ax, 4);
        uint32_t m = (uint32_t)nearbyintf(v * 16777216.0f); /* exact scale by 2^24, RNE */
        return (uint16_t)(sign | m);
    }
    uint32_t r = ax - 0x38000000u; /* rebias the exponent from 127 to 15 */
    r += 0xfffu + ((r >> 13) & 1u);
    return (uint16_t)(sign | (r >> 13));
}

enum { WL_F32 = 0, WL_F16 = 1, WL_BF16 = 2 };

typedef struct {
    void* out;
    int dtype;
    uint64_t key;
    uint64_t first; /* draw index of out[0] */
    uint64_t lo, hi;
} job_t;

static void* run_job(void* arg) {
    job_t* j = (job_t*)arg;
    for (uint64_t i = j->lo; i < j->hi; ++i) {
        float x = normal_at(j->key, j->first + i);
        if (j->dtype == WL_F32)
            ((float*)j->out)[i] = x;
        else if (j->dtype == WL_F16)
            ((uint16_t*)j->out)[i] = f32_to_f16(x);
        else
            ((uint16_t*)j->out)[i] = f32_to_bf16(x);
    }
    return 0;
}

/* Fill out[0..n) with draws first..first+n-1 of stream `key`, stored as dtype. */
int wl_fill_normal(void* out, int dtype, uint64_t n, uint64_t key, uint64_t first, int nthreads) {
    if (dtype < 0 || dtype > 2) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < (uint64_t)nthreads * 65536u) nthreads = 1;
    pthread_t th[256];
    int running[256];
    job_t jobs[256];
    uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    for (int t = 0; t < nthreads; ++t) {
        uint64_t lo = (uint64_t)t * per, hi = lo + per;
        if (lo > n) lo = n;
        if (hi > n) hi = n;
        jobs[t] = (job_t){out, dtype, key, first, lo, hi};
        running[t] = t < nthreads - 1 && pthread_create(&th[t], 0, run_job, &jobs[t]) == 0;
        if (!running[t]) run_job(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (running[t]) pthread_join(th[t], 0);
    return 0;
}

/* Round an f32 array to a 16-bit storage type (RNE); used for hand-made inputs. */
int wl_round_f32(const float* in, uint16_t* out, int dtype, uint64_t n) {
    if (dtype != WL_F16 && dtype != WL_BF16) return 1;
    for (uint64_t i = 0; i < n; ++i) out[i] = dtype == WL_F16 ? f32_to_f16(in[i]) : f32_to_bf16(in[i]);
    return 0;
}

/*
 * Random FP8 E4M3 codes: element i of stream `key` takes the bits of splitmix64
 * output i: sign = bit 0, exponent field = e_lo + (bits 1.. mod (e_hi - e_lo + 1)),
 * mantissa = bits 8..10. Only bit fields are drawn, never a rounding: with
 * 1 <= e_lo <= e_hi <= 14 no NaN code and no subnormal can occur.
 */
int wl_fill_e4m3(uint8_t* out, uint64_t n, uint64_t key, uint64_t first, int e_lo, int e_hi) {
    if (e_lo < 1 || e_hi > 14 || e_lo > e_hi) return 1;
    const uint64_t span = (uint64_t)(e_hi - e_lo + 1);
    for (uint64_t i = 0; i < n; ++i) {
        const uint64_t r = sm64_at(key, first + i);
        const unsigned e = (unsigned)e_lo + (unsigned)((r >> 1) % span);
        out[i] = (uint8_t)(((r & 1u) << 7) | (e << 3) | ((r >> 8) & 7u));
    }
    return 0;
}

/* One splitmix64 output, exposed so a test can check the generator itself. */
uint64_t wl_splitmix64_at(uint64_t key, uint64_t n) { return sm64_at(key, n); }
