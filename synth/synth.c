/*
 * Seeded synthetic-input generator shared by the oracle side and the CUDA
 * side of the tests and the benchmark.  It holds none of the paged-attention
 * arithmetic: it only turns (seed, counter) pairs into numbers.
 *
 * Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; constants from Vigna's public-domain
 * splitmix64.c).  It is counter based: the n-th output (n = 0, 1, ...) of a
 * generator seeded with s is mix(s + (n + 1) * GAMMA), so any element of a
 * stream can be produced independently and the fills below give identical
 * bits whatever the thread count.
 *
 * Derived draws:
 *   uniform  u = (x >> 11) * 2^-53                      in [0, 1)
 *   int      U[a, b] = a + floor(u * (b - a + 1))
 *   normal   element j uses counters 2j and 2j+1:
 *            n = sqrt(-2 ln(1 - u0)) * cos(2 pi u1)      (Box-Muller, cosine branch)
 *            rounded to fp32 (round-to-nearest) and, for bf16, from fp32 to
 *            bf16 with round-to-nearest-even.
 *   length mix (the skewed mix of "Simulating waste" on the ohmygp.com page):
 *            sequence i draws r = u(2i); r < 0.7 -> U[32, 511],
 *            r < 0.95 -> U[512, 2047], else U[2048, 4095], from u(2i+1).
 *   permutation: Durstenfeld's Fisher-Yates, step i = n-1 .. 1 swaps a[i]
 *            with a[j], j = U[0, i] drawn from counter n-1-i.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_u64(uint64_t seed, uint64_t counter) {
    return mix64(seed + (counter + 1ULL) * GAMMA);
}

/* Seed of a named sub-stream: keeps streams of one workload apart. */
uint64_t synth_stream_seed(uint64_t base, uint64_t tag) {
    return mix64(mix64(base) ^ (tag * GAMMA));
}

double synth_uniform(uint64_t seed, uint64_t counter) {
    return (double)(synth_u64(seed, counter) >> 11) * 0x1.0p-53;
}

int64_t synth_uniform_int(uint64_t seed, uint64_t counter, int64_t lo, int64_t hi) {
    double u = synth_uniform(seed, counter);
    return lo + (int64_t)floor(u * (double)(hi - lo + 1));
}

static double normal_at(uint64_t seed, uint64_t j) {
    const double two_pi = 6.283185307179586476925286766559;
    double u0 = synth_uniform(seed, 2 * j);
    double u1 = synth_uniform(seed, 2 * j + 1);
    return sqrt(-2.0 * log(1.0 - u0)) * cos(two_pi * u1);
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ---- threaded fills ---------------------------------------------------- */

typedef struct {
    uint64_t seed, offset, begin, end;
    void* out;
    int kind; /* 0 = f32, 1 = bf16 bits, 2 = f64 */
    double scale;
} fill_job;

static void* fill_worker(void* arg) {
    fill_job* j = (fill_job*)arg;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        double n = normal_at(j->seed, j->offset + i) * j->scale;
        if (j->kind == 0) {
            ((float*)j->out)[i] = (float)n;
        } else if (j->kind == 1) {
            ((uint16_t*)j->out)[i] = f32_to_bf16_rne((float)n);
        } else {
            ((double*)j->out)[i] = n;
        }
    }
    return NULL;
}

static int n_threads_for(uint64_t n) {
    long hw = sysconf(_SC_NPROCESSORS_ONLN);
    if (hw < 1) hw = 1;
    if (hw > 64) hw = 64;
    uint64_t by_size = n / (1u << 20) + 1; /* one thread per Mi elements */
    return (int)(by_size < (uint64_t)hw ? by_size : (uint64_t)hw);
}

static void fill_normal(uint64_t seed, uint64_t offset, uint64_t n, void* out, int kind,
                        double scale) {
    int nt = n_threads_for(n);
    pthread_t th[64];
    fill_job jobs[64];
    uint64_t per = (n + (uint64_t)nt - 1) / (uint64_t)nt;
    for (int t = 0; t < nt; ++t) {
        uint64_t b = per * (uint64_t)t, e = b + per;
        if (b > n) b = n;
        if (e > n) e = n;
        jobs[t] = (fill_job){seed, offset, b, e, out, kind, scale};
        if (nt == 1) {
            fill_worker(&jobs[t]);
        } else if (pthread_create(&th[t], NULL, fill_worker, &jobs[t]) != 0) {
            fill_worker(&jobs[t]);
            th[t] = 0;
        }
    }
    if (nt > 1)
        for (int t = 0; t < nt; ++t)
            if (th[t]) pthread_join(th[t], NULL);
}

/* Elements offset .. offset+n-1 of the N(0,1)*scale stream `seed`. */
void synth_fill_normal_f32(uint64_t seed, uint64_t offset, uint64_t n, float* out, double scale) {
    fill_normal(seed, offset, n, out, 0, scale);
}
void synth_fill_normal_bf16(uint64_t seed, uint64_t offset, uint64_t n, uint16_t* out,
                            double scale) {
    fill_normal(seed, offset, n, out, 1, scale);
}
void synth_fill_normal_f64(uint64_t seed, uint64_t offset, uint64_t n, double* out, double scale) {
    fill_normal(seed, offset, n, out, 2, scale);
}

void synth_fill_uniform_int(uint64_t seed, uint64_t offset, uint64_t n, int64_t lo, int64_t hi,
                            int32_t* out) {
    for (uint64_t i = 0; i < n; ++i) out[i] = (int32_t)synth_uniform_int(seed, offset + i, lo, hi);
}

void synth_lengths_mix(uint64_t seed, uint64_t n, int32_t* out) {
    for (uint64_t i = 0; i < n; ++i) {
        double r = synth_uniform(seed, 2 * i);
        int64_t lo, hi;
        if (r < 0.7) {
            lo = 32;
            hi = 511;
        } else if (r < 0.95) {
            lo = 512;
            hi = 2047;
        } else {
            lo = 2048;
            hi = 4095;
        }
        out[i] = (int32_t)synth_uniform_int(seed, 2 * i + 1, lo, hi);
    }
}

void synth_permutation(uint64_t seed, int32_t n, int32_t* out) {
    for (int32_t i = 0; i < n; ++i) out[i] = i;
    for (int32_t i = n - 1; i >= 1; --i) {
        int32_t j = (int32_t)synth_uniform_int(seed, (uint64_t)(n - 1 - i), 0, i);
        int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}
