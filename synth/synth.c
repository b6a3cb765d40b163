/*
 * Seeded synthetic inputs for the mHC forward workloads.
 *
 * This file holds random-number generation only: none of the mHC arithmetic.
 * Both the fp64 oracle and the CUDA path receive the arrays it fills, so the
 * two sides always see the same values.
 *
 * Generator: counter-based.  Every element is a pure function of
 * (seed, tensor id, element index, sub-stream), hashed with the splitmix64
 * output function published by S. Vigna ("Further scramblings of Marsaglia's
 * xorshift generators", splitmix64.c, 2014/2015).  Normals come from the
 * Box–Muller transform (G. E. P. Box, M. E. Muller, 1958).  The values do not
 * depend on the number of threads used to fill an array.
 *
 * bf16 results are rounded to nearest, ties to even, from the float32 value.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ull

static uint64_t splitmix64_out(uint64_t state)
{
    uint64_t z = state + GOLDEN_GAMMA;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* 64 random bits for (seed, tensor id, element index, sub-stream < 16). */
static uint64_t bits_at(uint64_t seed, uint32_t tid, uint64_t idx, uint32_t sub)
{
    uint64_t stream = splitmix64_out(seed ^ ((uint64_t)tid << 40));
    return splitmix64_out(stream ^ (idx * 16u + (uint64_t)(sub & 15u)));
}

/* Uniform on the open interval (0, 1): 53 random bits, centred in their cell. */
static double uniform_at(uint64_t seed, uint32_t tid, uint64_t idx, uint32_t sub)
{
    return ((double)(bits_at(seed, tid, idx, sub) >> 11) + 0.5) * 0x1.0p-53;
}

/* Standard normal from the Box–Muller pair of sub-streams (2p, 2p+1). */
static double normal_at(uint64_t seed, uint32_t tid, uint64_t idx, uint32_t pair)
{
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = uniform_at(seed, tid, idx, 2u * pair);
    double u2 = uniform_at(seed, tid, idx, 2u * pair + 1u);
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ---- a tiny parallel-for over element ranges -------------------------- */

enum kind { K_NORMAL_BF16, K_NORMAL_F32, K_ROWSCALE_BF16, K_STUDENT_T_BF16, K_INT_BF16 };

struct job {
    enum kind kind;
    void *out;
    int64_t count;
    uint64_t seed;
    uint32_t tid;
    double a, b;      /* kind-specific parameters */
    int64_t cols;     /* row length for K_ROWSCALE_BF16 */
    uint32_t tid2;    /* second tensor id (row scales) */
    int nu;           /* degrees of freedom for K_STUDENT_T_BF16 */
    int64_t lo, hi;   /* element range of this worker */
};

static double value_at(const struct job *j, int64_t i)
{
    switch (j->kind) {
    case K_NORMAL_BF16:
    case K_NORMAL_F32:
        return j->a * normal_at(j->seed, j->tid, (uint64_t)i, 0);
    case K_ROWSCALE_BF16: {
        /* row r has standard deviation 10^(a + (b - a) * U_r) */
        int64_t r = i / j->cols;
        double u = uniform_at(j->seed, j->tid2, (uint64_t)r, 0);
        double sigma = pow(10.0, j->a + (j->b - j->a) * u);
        return sigma * normal_at(j->seed, j->tid, (uint64_t)i, 0);
    }
    case K_STUDENT_T_BF16: {
        /* Z / sqrt(chi2_nu / nu), chi2_nu = sum of nu squared normals */
        double z = normal_at(j->seed, j->tid, (uint64_t)i, 0);
        double chi2 = 0.0;
        for (int k = 0; k < j->nu; ++k) {
            double g = normal_at(j->seed, j->tid, (uint64_t)i, (uint32_t)(1 + k));
            chi2 += g * g;
        }
        return j->a * z / sqrt(chi2 / (double)j->nu);
    }
    case K_INT_BF16: {
        /* integers uniform on [a, b] */
        double u = uniform_at(j->seed, j->tid, (uint64_t)i, 0);
        double span = j->b - j->a + 1.0;
        double v = j->a + floor(u * span);
        return v > j->b ? j->b : v;
    }
    }
    return 0.0;
}

static void *worker(void *arg)
{
    struct job *j = (struct job *)arg;
    for (int64_t i = j->lo; i < j->hi; ++i) {
        double v = value_at(j, i);
        if (j->kind == K_NORMAL_F32)
            ((float *)j->out)[i] = (float)v;
        else
            ((uint16_t *)j->out)[i] = f32_to_bf16_rne((float)v);
    }
    return NULL;
}

static void run(struct job base, int nthreads)
{
    if (nthreads <= 0) {
        long nc = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = nc > 0 ? (int)nc : 1;
    }
    if (nthreads > 256) nthreads = 256;
    if (base.count < 65536) nthreads = 1;
    struct job jobs[256];
    pthread_t th[256];
    int joined[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].lo = base.count * t / nthreads;
        jobs[t].hi = base.count * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t) {
        joined[t] = pthread_create(&th[t], NULL, worker, &jobs[t]) == 0;
        if (!joined[t]) worker(&jobs[t]); /* no thread: do the range here */
    }
    worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (joined[t]) pthread_join(th[t], NULL);
}

/* ---- exported entry points -------------------------------------------- */

void synth_normal_bf16(uint16_t *out, int64_t count, uint64_t seed, uint32_t tid,
                       double stddev, int nthreads)
{
    struct job j = {0};
    j.kind = K_NORMAL_BF16; j.out = out; j.count = count; j.seed = seed; j.tid = tid; j.a = stddev;
    run(j, nthreads);
}

void synth_normal_f32(float *out, int64_t count, uint64_t seed, uint32_t tid,
                      double stddev, int nthreads)
{
    struct job j = {0};
    j.kind = K_NORMAL_F32; j.out = out; j.count = count; j.seed = seed; j.tid = tid; j.a = stddev;
    run(j, nthreads);
}

void synth_rowscale_normal_bf16(uint16_t *out, int64_t rows, int64_t cols, uint64_t seed,
                                uint32_t tid, uint32_t sigma_tid, double log10_lo,
                                double log10_hi, int nthreads)
{
    struct job j = {0};
    j.kind = K_ROWSCALE_BF16; j.out = out; j.count = rows * cols; j.cols = cols;
    j.seed = seed; j.tid = tid; j.tid2 = sigma_tid; j.a = log10_lo; j.b = log10_hi;
    run(j, nthreads);
}

void synth_student_t_bf16(uint16_t *out, int64_t count, uint64_t seed, uint32_t tid,
                          int nu, double scale, int nthreads)
{
    struct job j = {0};
    j.kind = K_STUDENT_T_BF16; j.out = out; j.count = count; j.seed = seed; j.tid = tid;
    j.nu = nu < 1 ? 1 : (nu > 14 ? 14 : nu); j.a = scale;
    run(j, nthreads);
}

void synth_int_bf16(uint16_t *out, int64_t count, uint64_t seed, uint32_t tid,
                    int lo, int hi, int nthreads)
{
    struct job j = {0};
    j.kind = K_INT_BF16; j.out = out; j.count = count; j.seed = seed; j.tid = tid;
    j.a = (double)lo; j.b = (double)hi;
    run(j, nthreads);
}
