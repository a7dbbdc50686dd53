/*
 * Seeded synthetic input generator for the row-softmax workloads.
 *
 * This module only makes input matrices. It holds none of the softmax
 * arithmetic and is shared, unchanged, by the CPU oracle tests, the CUDA
 * parity tests and the benchmark.
 *
 * Random source: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014). The sequential generator
 * seeded with s returns, as its k-th output (k = 0, 1, ...), the 64-bit mix of
 * s + (k + 1) * 0x9E3779B97F4A7C15. We evaluate that closed form directly, so
 * any element can be generated independently of the others and the matrix is
 * the same for any thread count.
 *
 * Normal variates: Box-Muller on pairs of uniforms. Element e = i*N + j of a
 * matrix belongs to pair p = e / 2; the pair draws outputs 2p and 2p + 1 of
 * the stream, u1 in (0, 1] and u2 in [0, 1); the even element takes
 * r*cos(2*pi*u2) and the odd one r*sin(2*pi*u2), r = sqrt(-2 ln u1).
 * Uniform variates on [lo, hi): lo + (hi - lo) * u with u = (z >> 11) * 2^-53,
 * drawn from output e of a second stream seeded with seed ^ UNIFORM_STREAM.
 *
 * Casts: double -> float rounds to nearest even (C conversion), then
 * float -> bf16 / f16 rounds to nearest even (below), which is what
 * torch's tensor.float().to(torch.bfloat16 / torch.float16) does.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_F32 0
#define SYNTH_BF16 1
#define SYNTH_F16 2

#define SYNTH_DIST_NORMAL 0
#define SYNTH_DIST_UNIFORM 1

static const uint64_t GOLDEN = 0x9E3779B97F4A7C15ULL;
static const uint64_t UNIFORM_STREAM = 0xD1B54A32D192ED03ULL;

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* k-th output (k >= 0) of SplitMix64 seeded with `seed`. */
uint64_t synth_splitmix64_at(uint64_t seed, uint64_t k) {
    return mix64(seed + (k + 1) * GOLDEN);
}

static double unit_open0(uint64_t z) { /* (0, 1] */
    return (double)((z >> 11) + 1) * 0x1.0p-53;
}

static double unit_open1(uint64_t z) { /* [0, 1) */
    return (double)(z >> 11) * 0x1.0p-53;
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static uint16_t f32_to_f16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a >= 0x7F800000u) /* inf or NaN */
        return (uint16_t)(sign | 0x7C00u | (a > 0x7F800000u ? 0x0200u : 0u));
    float af;
    memcpy(&af, &a, 4);
    if (af == 0.0f)
        return sign;
    if (af >= 65520.0f) /* rounds to infinity */
        return (uint16_t)(sign | 0x7C00u);
    /* Quantum of the f16 binade that holds af (subnormal quantum 2^-24). */
    int e;
    frexpf(af, &e);              /* af = f * 2^e, f in [0.5, 1) */
    int qe = (e - 1 < -14 ? -14 : e - 1) - 10;
    float q = ldexpf(1.0f, qe);
    float r = nearbyintf(af / q); /* exact scaling, ties to even */
    uint32_t m = (uint32_t)r;     /* significand in units of q */
    uint16_t bits;
    if (qe == -24) {
        /* subnormal range; m may reach 1024, which encodes the smallest normal */
        bits = (uint16_t)m;
    } else {
        if (m == 2048u) { m = 1024u; qe += 1; }
        bits = (uint16_t)(((uint32_t)(qe + 10 + 15) << 10) | (m - 1024u));
    }
    return (uint16_t)(sign | bits);
}

typedef struct {
    void* out;
    int64_t M, N, ld;
    int dtype;
    uint64_t seed;
    int dist;
    double p0, p1;
    int64_t alt_every;
    double alt_lo, alt_hi;
    int64_t causal_period;
    int pad_nan;
    int64_t row0;               /* global index of the first row in `out` */
    int64_t row_begin, row_end; /* local row range of this job */
} job_t;

static double draw(const job_t* jb, int64_t i, int64_t j) {
    uint64_t e = (uint64_t)i * (uint64_t)jb->N + (uint64_t)j;
    if (jb->causal_period > 0 && j > i % jb->causal_period)
        return -INFINITY;
    int dist = jb->dist;
    double a = jb->p0, b = jb->p1;
    if (jb->alt_every > 0 && i % jb->alt_every == 0) {
        dist = SYNTH_DIST_UNIFORM;
        a = jb->alt_lo;
        b = jb->alt_hi;
    }
    if (dist == SYNTH_DIST_UNIFORM) {
        double u = unit_open1(synth_splitmix64_at(jb->seed ^ UNIFORM_STREAM, e));
        return a + (b - a) * u;
    }
    uint64_t p = e >> 1;
    double u1 = unit_open0(synth_splitmix64_at(jb->seed, 2 * p));
    double u2 = unit_open1(synth_splitmix64_at(jb->seed, 2 * p + 1));
    double r = sqrt(-2.0 * log(u1));
    double t = 6.283185307179586476925286766559 * u2;
    double z = (e & 1) ? r * sin(t) : r * cos(t);
    return a + b * z;
}

static void store(const job_t* jb, int64_t off, double v) {
    float f = (float)v;
    if (jb->dtype == SYNTH_F32) {
        ((float*)jb->out)[off] = f;
    } else if (jb->dtype == SYNTH_BF16) {
        ((uint16_t*)jb->out)[off] = f32_to_bf16_rne(f);
    } else {
        ((uint16_t*)jb->out)[off] = f32_to_f16_rne(f);
    }
}

static void* run_job(void* arg) {
    const job_t* jb = (const job_t*)arg;
    for (int64_t i = jb->row_begin; i < jb->row_end; ++i) {
        for (int64_t j = 0; j < jb->N; ++j)
            store(jb, i * jb->ld + j, draw(jb, jb->row0 + i, j));
        if (jb->pad_nan)
            for (int64_t j = jb->N; j < jb->ld; ++j)
                store(jb, i * jb->ld + j, NAN);
    }
    return NULL;
}

/*
 * Fill rows [row0, row0 + M) of the workload's N-column matrix into `out`,
 * row-major with leading dimension ld (elements). Row i of `out` is global
 * row row0 + i: every element depends only on its global (row, column).
 *   dist = SYNTH_DIST_NORMAL: N(p0, p1^2), i.e. p0 is the mean, p1 the standard deviation.
 *   dist = SYNTH_DIST_UNIFORM: U[p0, p1).
 *   alt_every > 0: rows i with i % alt_every == 0 are drawn from U[alt_lo, alt_hi).
 *   causal_period > 0: entry (i, j) is -inf where j > i mod causal_period.
 *   pad_nan: columns [N, ld) are set to NaN (otherwise left untouched).
 * Returns 0 on success, -1 on bad arguments.
 */
int synth_generate(void* out, int64_t row0, int64_t M, int64_t N, int64_t ld, int dtype,
                   uint64_t seed, int dist, double p0, double p1,
                   int64_t alt_every, double alt_lo, double alt_hi,
                   int64_t causal_period, int pad_nan, int nthreads) {
    if (row0 < 0 || M < 0 || N < 0 || ld < N || (M > 0 && !out)) return -1;
    if (dtype < SYNTH_F32 || dtype > SYNTH_F16) return -1;
    if (dist != SYNTH_DIST_NORMAL && dist != SYNTH_DIST_UNIFORM) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > M) nthreads = M > 0 ? (int)M : 1;
    job_t jobs[256];
    pthread_t tids[256];
    int64_t per = (M + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        job_t jb = {out, M, N, ld, dtype, seed, dist, p0, p1, alt_every, alt_lo,
                    alt_hi, causal_period, pad_nan, row0, t * per, (t + 1) * per};
        if (jb.row_begin > M) jb.row_begin = M;
        if (jb.row_end > M) jb.row_end = M;
        jobs[t] = jb;
    }
    if (nthreads == 1) {
        run_job(&jobs[0]);
        return 0;
    }
    unsigned char joined[256];
    for (int t = 0; t < nthreads; ++t) {
        joined[t] = 0;
        if (pthread_create(&tids[t], NULL, run_job, &jobs[t]) != 0) {
            run_job(&jobs[t]); /* run inline if a thread cannot be made */
            joined[t] = 1;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (!joined[t]) pthread_join(tids[t], NULL);
    return 0;
}
