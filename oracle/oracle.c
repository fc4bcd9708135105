/*
 * oracle.c -- plain, slow CPU oracle for the BF16 weight-streaming decode chain.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file; only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library: it was written from the definitions below, not from the kernels.
 *
 * Every sum is accumulated in IEEE double, left to right over k (the plain
 * definition; no blocking, no reordering).  Values stored as bf16/fp16 are
 * decoded exactly; results are rounded to a storage format only where the
 * caller asks for it (round-to-nearest-even, written from the IEEE 754
 * definition of the format).
 *
 * Sources (page title, section):
 *  - GEMV with BF16 inputs and FP32 accumulation, one weight matrix times one
 *    vector per sequence at small batch: "One Token, Kernel by Kernel: A Decode
 *    Step on a Laptop GPU", Step 1, "What one block launches".
 *  - RMSNorm as mean square, reciprocal square root and weight multiply:
 *    "GPU Kernel Optimization", Architecture (the Kernel bullet); the model it
 *    sits in (RMSNorm, GQA, SwiGLU MLP): "One Token, Kernel by Kernel", Step 1,
 *    "The setup".
 *  - LayerNorm -> Linear -> GELU blocks: "Making small PyTorch ops faster on a
 *    laptop GPU", "Beyond language models".
 *  - argmax over the logits: "One Token, Kernel by Kernel", "The whole step".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Storage formats                                                     */
/* ------------------------------------------------------------------ */

/* bf16 is, by definition, the upper half of an IEEE binary32 pattern. */
static inline double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double fp16_value(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int f = bits & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);    /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

/*
 * Round v to the nearest value of a binary format with p significand bits
 * (implicit bit included), minimum normal exponent emin and maximum exponent
 * emax; ties go to the even significand.  Overflow gives infinity.
 */
static double round_to_format(double v, int p, int emin, int emax)
{
    if (v == 0.0 || !isfinite(v))
        return v;
    double a = fabs(v);
    int E;
    frexp(a, &E);                    /* a = f * 2^E, 0.5 <= f < 1 */
    int lead = E - 1;                /* exponent of the leading bit */
    if (lead < emin)
        lead = emin;                 /* subnormal range: fixed quantum */
    double q = ldexp(1.0, lead - (p - 1));
    double r = nearbyint(a / q) * q; /* default mode: nearest, ties to even */
    double maxval = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (r > maxval)
        r = INFINITY;
    return copysign(r, v);
}

static uint16_t bf16_bits_of(double v)
{
    if (isnan(v))
        return 0x7fc0;
    float f = (float)round_to_format(v, 8, -126, 127); /* exact in binary32 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

static uint16_t fp16_bits_of(double v)
{
    if (isnan(v))
        return 0x7e00;
    double r = round_to_format(v, 11, -14, 15);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7c00;
    int E;
    frexp(a, &E);
    int lead = E - 1;
    if (lead < -14)                                     /* subnormal */
        return sign | (uint16_t)ldexp(a, 24);
    uint16_t frac = (uint16_t)(ldexp(a, -lead) * 1024.0 - 1024.0);
    return sign | (uint16_t)((lead + 15) << 10) | frac;
}

void ws_oracle_bf16_to_f64(const uint16_t *in, double *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = bf16_value(in[i]);
}

void ws_oracle_f64_to_bf16(const double *in, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = bf16_bits_of(in[i]);
}

void ws_oracle_fp16_to_f64(const uint16_t *in, double *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = fp16_value(in[i]);
}

void ws_oracle_f64_to_fp16(const double *in, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = fp16_bits_of(in[i]);
}

/* Round each value to binary32 (C conversion: nearest, ties to even). */
void ws_oracle_round_f32(double *v, long n)
{
    for (long i = 0; i < n; ++i)
        v[i] = (double)(float)v[i];
}

/* ------------------------------------------------------------------ */
/* Matrix-vector product                                               */
/* ------------------------------------------------------------------ */

/*
 * y[b][m] = sum_{k=0}^{K-1} W[m][k] * x[b][k]
 *
 * W: bf16 bit patterns, row-major [M][K] (the weight[out][in] layout of a
 * linear layer); x: [B][K] doubles; y: [B][M] doubles.  The sum runs k = 0..K-1
 * in double.  `threads` splits the output rows only, so the result does not
 * depend on it.
 */
void ws_oracle_gemv(const uint16_t *W, long M, long K, const double *x, long B,
                    double *y, int threads)
{
#ifdef _OPENMP
#pragma omp parallel for num_threads(threads > 0 ? threads : 1) schedule(static)
#endif
    for (long m = 0; m < M; ++m) {
        const uint16_t *row = W + m * K;
        for (long b = 0; b < B; ++b) {
            const double *xb = x + b * K;
            double s = 0.0;
            for (long k = 0; k < K; ++k)
                s += bf16_value(row[k]) * xb[k];
            y[b * M + m] = s;
        }
    }
    (void)threads;
}

/* ------------------------------------------------------------------ */
/* Normalisations and activations                                      */
/* ------------------------------------------------------------------ */

/*
 * RMSNorm of each row: r = 1 / sqrt(mean_k x^2 + eps); out = x * r * gamma.
 * (eps inside the square root; no rounding here.)
 */
void ws_oracle_rmsnorm(const double *x, long B, long K, const double *gamma,
                       double eps, double *out)
{
    for (long b = 0; b < B; ++b) {
        const double *xb = x + b * K;
        double ss = 0.0;
        for (long k = 0; k < K; ++k)
            ss += xb[k] * xb[k];
        double r = 1.0 / sqrt(ss / (double)K + eps);
        for (long k = 0; k < K; ++k)
            out[b * K + k] = xb[k] * r * gamma[k];
    }
}

/*
 * LayerNorm of each row with biased variance:
 * out = (x - mean) / sqrt(var + eps) * gamma + beta.
 */
void ws_oracle_layernorm(const double *x, long B, long N, const double *gamma,
                         const double *beta, double eps, double *out)
{
    for (long b = 0; b < B; ++b) {
        const double *xb = x + b * N;
        double s = 0.0;
        for (long i = 0; i < N; ++i)
            s += xb[i];
        double mean = s / (double)N;
        double v = 0.0;
        for (long i = 0; i < N; ++i)
            v += (xb[i] - mean) * (xb[i] - mean);
        double var = v / (double)N;
        double r = 1.0 / sqrt(var + eps);
        for (long i = 0; i < N; ++i)
            out[b * N + i] = (xb[i] - mean) * r * gamma[i] + beta[i];
    }
}

/* GELU, exact (erf) form: 0.5 * z * (1 + erf(z / sqrt(2))). */
void ws_oracle_gelu(const double *z, double *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = 0.5 * z[i] * (1.0 + erf(z[i] / sqrt(2.0)));
}

/* SwiGLU gate: silu(g) * u with silu(g) = g / (1 + exp(-g)). */
void ws_oracle_swiglu(const double *g, const double *u, double *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* Index of the largest value of each row; ties go to the lowest index. */
void ws_oracle_argmax_rows(const double *v, long rows, long cols, int32_t *idx)
{
    for (long r = 0; r < rows; ++r) {
        const double *vr = v + r * cols;
        long best = 0;
        for (long j = 1; j < cols; ++j)
            if (vr[j] > vr[best])
                best = j;
        idx[r] = (int32_t)best;
    }
}

int ws_oracle_openmp_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
