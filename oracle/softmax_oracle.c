/*
 * CPU oracle for the fused row-wise softmax. TEST INFRASTRUCTURE ONLY: only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this file's library. The CUDA product path never calls it, and the two
 * share no code.
 *
 * What it computes: for every row i of an M x N row-major matrix,
 *     y[i,j] = exp(x[i,j] - m_i) / s_i,   m_i = max_j x[i,j],
 *     s_i = sum_j exp(x[i,j] - m_i),
 * which is the numerically stable softmax the source pages define
 * ("Triton: Writing GPU Kernels in Python, Measured", Step 2: subtract the
 * row maximum, exponentiate, divide by the sum; "Fused Softmax on GPU: From
 * Naive PyTorch to Persistent Triton Kernels", the four implementations).
 * As in the "Warpline" README's softmax contract (Providers), the reference
 * value is computed in FP64 and cast once to the output dtype:
 *   1. widen every input to double (exact for f32, bf16 and f16);
 *   2. m = max_j x_j, by a plain scan (NaN never compares greater, so it is
 *      skipped here and propagates through step 3 instead);
 *   3. s = sum_j exp(x_j - m), a plain sequential double sum;
 *   4. y_j = exp(x_j - m) / s;
 *   5. round y_j once, to nearest with ties to even, to the dtype.
 * Consequences of the definition, kept as they fall out: a row that is all
 * -inf gives 0/0 = NaN everywhere; a NaN or +inf anywhere in a row gives a
 * NaN sum and so NaN everywhere in that row.
 *
 * Layout: element (i, j) of the input is in[i*ld_in + j], of the output
 * out[i*ld_out + j]; columns [N, ld) are neither read nor written.
 * dtype 0 = f32 (IEEE binary32), 1 = bf16 (upper half of binary32),
 * 2 = f16 (IEEE binary16); bf16 and f16 are 16-bit patterns.
 *
 * Also here: the masked softmax (entries past a row's valid length count as
 * -inf), the softmax backward dx = y * (dy - sum_j y_j dy_j) and the residual
 * RMSNorm forward, each stated and cited where it is defined below.
 *
 * Parity pins (tests/test_oracle_pins.py) check this code against 60-digit
 * decimal brute force, closed forms and invariants, not against itself.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_F16 2

/* ---- step 1: decode one stored element to double ---------------------- */

static double decode_f32(const void* base, int64_t k) {
    float f;
    memcpy(&f, (const char*)base + 4 * k, 4);
    return (double)f;
}

static double decode_bf16(const void* base, int64_t k) {
    uint16_t h;
    memcpy(&h, (const char*)base + 2 * k, 2);
    uint32_t u = (uint32_t)h << 16; /* bf16 is the top half of a binary32 */
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double decode_f16(const void* base, int64_t k) {
    uint16_t h;
    memcpy(&h, (const char*)base + 2 * k, 2);
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double decode(const void* base, int64_t k, int dtype) {
    if (dtype == OR_F32) return decode_f32(base, k);
    if (dtype == OR_BF16) return decode_bf16(base, k);
    return decode_f16(base, k);
}

/* ---- step 5: one rounding, nearest-even, from double ------------------- */

/*
 * Round |v| to a binary format with p significand bits, smallest normal
 * exponent emin and largest finite exponent emax; return the bit pattern of
 * the result with `ebits` exponent bits. The rounding is nearbyint() of v
 * scaled by a power of two (exact), in the default nearest-even mode.
 */
static uint32_t round_to_format(double v, int p, int emin, int emax, int ebits) {
    uint32_t sign = signbit(v) ? 1u : 0u;
    int mbits = p - 1;
    uint32_t exp_all = (1u << ebits) - 1u;
    uint32_t sign_bit = sign << (ebits + mbits);
    if (isnan(v)) return sign_bit | (exp_all << mbits) | (1u << (mbits - 1));
    double a = fabs(v);
    if (isinf(a)) return sign_bit | (exp_all << mbits);
    if (a == 0.0) return sign_bit;
    int e = ilogb(a);                      /* 2^e <= a < 2^(e+1) */
    int qe = (e < emin ? emin : e) - mbits; /* exponent of one unit in the last place */
    double r = nearbyint(ldexp(a, -qe));   /* significand in units of 2^qe */
    if (r >= ldexp(1.0, p)) {              /* carried into the next binade */
        r = ldexp(r, -1);
        qe += 1;
    }
    if (qe + mbits > emax) return sign_bit | (exp_all << mbits); /* overflow */
    uint32_t m = (uint32_t)r;
    if (m < (1u << mbits))                 /* subnormal (qe == emin - mbits) */
        return sign_bit | m;
    uint32_t bexp = (uint32_t)(qe + mbits + ((1 << (ebits - 1)) - 1));
    return sign_bit | (bexp << mbits) | (m - (1u << mbits));
}

static void encode(void* base, int64_t k, int dtype, double y) {
    if (dtype == OR_F32) {
        float f = (float)y; /* C conversion: nearest-even in the default mode */
        memcpy((char*)base + 4 * k, &f, 4);
    } else if (dtype == OR_BF16) {
        uint16_t h = (uint16_t)round_to_format(y, 8, -126, 127, 8);
        memcpy((char*)base + 2 * k, &h, 2);
    } else {
        uint16_t h = (uint16_t)round_to_format(y, 11, -14, 15, 5);
        memcpy((char*)base + 2 * k, &h, 2);
    }
}

/* ---- steps 2-4 for one row ---------------------------------------------- */

/* y[j] = exp(x[j] - m) / s in double, for one row of n decoded values. */
static void softmax_row_f64(const double* x, double* y, int64_t n) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (x[j] > m) m = x[j];
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j)
        s += exp(x[j] - m);
    for (int64_t j = 0; j < n; ++j)
        y[j] = exp(x[j] - m) / s;
}

typedef struct {
    const void* in;
    void* out;      /* dtype-typed output, or NULL */
    double* out64;  /* double output before the cast, or NULL */
    int64_t N, ld_in, ld_out;
    int dtype;
    int64_t row_begin, row_end;
    double* work;   /* 2*N doubles */
    const int32_t* lens;   /* per-row valid lengths, or NULL */
    int64_t causal_period; /* used when lens is NULL: row i keeps i mod period + 1 entries */
} job_t;

/* Number of leading entries of row i that take part (the rest are -inf). */
static int64_t valid_length(const job_t* jb, int64_t i) {
    int64_t v = jb->N;
    if (jb->lens) v = jb->lens[i];
    else if (jb->causal_period > 0) v = i % jb->causal_period + 1;
    if (v < 0) v = 0;
    if (v > jb->N) v = jb->N;
    return v;
}

static void* run_rows(void* arg) {
    job_t* jb = (job_t*)arg;
    double* x = jb->work;
    double* y = jb->work + jb->N;
    for (int64_t i = jb->row_begin; i < jb->row_end; ++i) {
        /* Masked entries are -inf by definition and are never read. */
        const int64_t v = valid_length(jb, i);
        for (int64_t j = 0; j < jb->N; ++j)
            x[j] = j < v ? decode(jb->in, i * jb->ld_in + j, jb->dtype) : -INFINITY;
        softmax_row_f64(x, y, jb->N);
        for (int64_t j = 0; j < jb->N; ++j) {
            if (jb->out) encode(jb->out, i * jb->ld_out + j, jb->dtype, y[j]);
            if (jb->out64) jb->out64[i * jb->ld_out + j] = y[j];
        }
    }
    return NULL;
}

static int run(const void* in, void* out, double* out64, int64_t M, int64_t N,
               int64_t ld_in, int64_t ld_out, int dtype, int nthreads, const int32_t* lens,
               int64_t causal_period) {
    if (M < 0 || N < 1 || ld_in < N || ld_out < N) return 1;
    if (dtype < OR_F32 || dtype > OR_F16) return 2;
    if (M == 0) return 0;
    if (!in || (!out && !out64)) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > M) nthreads = (int)M;
    job_t jobs[256];
    pthread_t tids[256];
    unsigned char inline_run[256];
    double* work = (double*)malloc(sizeof(double) * 2 * (size_t)N * (size_t)nthreads);
    if (!work) return 3;
    int64_t per = (M + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = t * per, e = (t + 1) * per;
        if (b > M) b = M;
        if (e > M) e = M;
        job_t jb = {in, out, out64, N, ld_in, ld_out, dtype, b, e, work + 2 * N * (int64_t)t,
                    lens, causal_period};
        jobs[t] = jb;
    }
    if (nthreads == 1) {
        run_rows(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t) {
            inline_run[t] = 0;
            if (pthread_create(&tids[t], NULL, run_rows, &jobs[t]) != 0) {
                run_rows(&jobs[t]);
                inline_run[t] = 1;
            }
        }
        for (int t = 0; t < nthreads; ++t)
            if (!inline_run[t]) pthread_join(tids[t], NULL);
    }
    free(work);
    return 0;
}

/*
 * Softmax of every row, cast once to `dtype`. Rows are split across
 * `nthreads` host threads (each row is computed by exactly the code above, so
 * the result does not depend on the thread count). Returns 0 on success,
 * 1 on bad sizes or pointers, 2 on an unknown dtype, 3 if out of memory.
 */
int oracle_softmax_rows(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                        int64_t ld_out, int dtype, int nthreads) {
    return run(in, out, NULL, M, N, ld_in, ld_out, dtype, nthreads, NULL, 0);
}

/*
 * Masked softmax: in row i only the first L_i entries take part; the others
 * are -inf (never read) and so come out as exact zeros. L_i = lens[i] when
 * lens is not NULL, else i mod causal_period + 1 when causal_period > 0
 * (the causal attention mask of rows holding query positions i mod period),
 * else N; L_i is clamped to [0, N]. L_i = 0 leaves an all -inf row: NaN.
 */
int oracle_softmax_rows_masked(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                               int64_t ld_out, int dtype, const int32_t* lens,
                               int64_t causal_period, int nthreads) {
    return run(in, out, NULL, M, N, ld_in, ld_out, dtype, nthreads, lens, causal_period);
}

/* The same, returning the double values before the final cast (for diagnostics). */
int oracle_softmax_rows_f64(const void* in, double* out64, int64_t M, int64_t N,
                            int64_t ld_in, int64_t ld_out, int dtype, int nthreads) {
    return run(in, NULL, out64, M, N, ld_in, ld_out, dtype, nthreads, NULL, 0);
}

/*
 * Softmax backward ("Measured optimization case studies", Training: softmax
 * saves its output y and computes y * (dy - sum(y * dy))): for every row i,
 *     dot_i = sum_j y[i,j] * dy[i,j],   dx[i,j] = y[i,j] * (dy[i,j] - dot_i),
 * computed in FP64 (sequential sum) and cast once to the dtype. y, dy and dx
 * are M x N with their own pitches (elements).
 */
static void backward_rows(const void* y, const void* dy, void* dx, int64_t row_begin,
                          int64_t row_end, int64_t N, int64_t ld_y, int64_t ld_dy,
                          int64_t ld_dx, int dtype) {
    for (int64_t i = row_begin; i < row_end; ++i) {
        double dot = 0.0;
        for (int64_t j = 0; j < N; ++j)
            dot += decode(y, i * ld_y + j, dtype) * decode(dy, i * ld_dy + j, dtype);
        for (int64_t j = 0; j < N; ++j) {
            const double yj = decode(y, i * ld_y + j, dtype);
            const double gj = decode(dy, i * ld_dy + j, dtype);
            encode(dx, i * ld_dx + j, dtype, yj * (gj - dot));
        }
    }
}

int oracle_softmax_backward(const void* y, const void* dy, void* dx, int64_t M, int64_t N,
                            int64_t ld_y, int64_t ld_dy, int64_t ld_dx, int dtype) {
    if (M < 0 || N < 1 || ld_y < N || ld_dy < N || ld_dx < N) return 1;
    if (dtype < OR_F32 || dtype > OR_F16) return 2;
    if (M > 0 && (!y || !dy || !dx)) return 1;
    backward_rows(y, dy, dx, 0, M, N, ld_y, ld_dy, ld_dx, dtype);
    return 0;
}

/*
 * Residual RMSNorm forward (the "Warpline" README's K1 kernel: one program per
 * row adds the input and the residual in FP32, rounds that sum once to the
 * input dtype, reduces the RMS, applies the weight and writes one rounded
 * result; "Measured optimization case studies", Residual RMSNorm). For every
 * row i, with w the N weights:
 *     h_j    = dtype(x[i,j] + r[i,j])                 (one rounding of the sum)
 *     ms     = (1/N) * sum_j h_j^2                      (FP64, sequential)
 *     y[i,j] = dtype(h_j * w_j / sqrt(ms + eps))       (FP64, one rounding)
 * The pages add in FP32 and then round to the dtype. For bf16 and f16 inputs
 * that equals one rounding of the exact sum (FP32 carries at least twice
 * their precision plus two bits, so rounding twice changes nothing), and for
 * f32 inputs it is the FP32 sum; the double sum below, rounded once, gives
 * both (53 >= 2 * 24 + 2 bits). x, r, y are M x N with their own pitches.
 */
static double to_dtype(double v, int dtype) {
    unsigned char buf[4];
    encode(buf, 0, dtype, v);
    return decode(buf, 0, dtype);
}

int oracle_rmsnorm_residual(const void* x, const void* r, const void* w, void* y, int64_t M,
                            int64_t N, int64_t ld_x, int64_t ld_r, int64_t ld_y, double eps,
                            int dtype) {
    if (M < 0 || N < 1 || ld_x < N || ld_r < N || ld_y < N || !(eps >= 0.0)) return 1;
    if (dtype < OR_F32 || dtype > OR_F16) return 2;
    if (M > 0 && (!x || !r || !w || !y)) return 1;
    double* h = (double*)malloc((size_t)N * sizeof(double));
    if (!h) return 3;
    for (int64_t i = 0; i < M; ++i) {
        double ms = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            h[j] = to_dtype(decode(x, i * ld_x + j, dtype) + decode(r, i * ld_r + j, dtype), dtype);
            ms += h[j] * h[j];
        }
        ms /= (double)N;
        const double rms = sqrt(ms + eps);
        for (int64_t j = 0; j < N; ++j)
            encode(y, i * ld_y + j, dtype, h[j] * decode(w, j, dtype) / rms);
    }
    free(h);
    return 0;
}

/* Step 5 alone: round doubles to `dtype` storage (f32 values or 16-bit patterns). */
int oracle_cast(const double* v, void* out, int64_t n, int dtype) {
    if (dtype < OR_F32 || dtype > OR_F16) return 2;
    for (int64_t k = 0; k < n; ++k) encode(out, k, dtype, v[k]);
    return 0;
}

/* Step 1 alone: decode `dtype` storage to doubles. */
int oracle_decode(const void* in, double* v, int64_t n, int dtype) {
    if (dtype < OR_F32 || dtype > OR_F16) return 2;
    for (int64_t k = 0; k < n; ++k) v[k] = decode(in, k, dtype);
    return 0;
}
