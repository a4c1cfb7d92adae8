/*
 * q4_oracle.c -- plain CPU oracle for the Q4_0-weight x Q8_0-activation
 * decode GEMV  y = W.x  (T token columns).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; the two only ever see the same input bytes.
 *
 * Every function is the plain definition written out, with no blocking,
 * fusion or reordering.  Floating-point results that the method leaves in
 * fp32 (the quantiser) are computed in fp32 exactly as defined; the GEMV
 * output is formed in fp64, where every product is exact.
 *
 * Sources (page title, section):
 *  - minfer README, "How it works": gemv_dp4a is a q4_0 GEMV with int8
 *    activations; mega streams packed q4 weights with int8 activations.
 *  - minfer README, "The optimization journey", M9: SIMD nibble masking and
 *    the folded -8 offset, sum (n-8)x = sum n.x - 8 sum x.
 *  - minfer README, M15/M16: both kernels form identical per-block integer
 *    sums, then scale and accumulate them in float.
 *  - colibri qwen36 docs, dense int8 IDOT GEMV: an int8 activation scale of
 *    amax/127, exact int32 products scaled afterwards.
 * The block formats, as the GGML q4_0 / q8_0 names denote them:
 *  - Q4_0 block: 32 weights; bytes 0-1 an fp16 scale d (little-endian);
 *    bytes 2..17 hold qs[16]; element j (j < 16) is the low nibble of qs[j],
 *    element j+16 its high nibble; the weight is (n - 8) * d.
 *  - Q8_0 block: 32 activations; d = amax/127 stored as fp16; each
 *    q = round-half-away-from-zero(x * (1/d)) as int8 (all zero if amax = 0).
 *    Byte layout: fp16 d then 32 int8 (34 bytes).
 *
 * Readings where the pages are silent:
 *  - 1/d is taken from the fp32 d, before d is rounded to fp16.
 *  - x * (1/d) is one fp32 multiply, rounded to nearest even.
 *  - amax = 0 gives d = 0, 1/d := 0, all q = 0.
 *  - argmax: lowest index among equal maxima, equality by IEEE == (so -0 == +0).
 *  - top-2: the second is the argmax of the rows other than the first.
 *  - Q4_0 encoder (requantisation at load): GGML's q4_0 encoder (see the
 *    section below).
 *  - sequence epilogue: y = W.x + bias + residual, the two terms added
 *    after the GEMV value.
 *
 * ORC_MUTANT (compile-time, default 0) plants one known mistake; the test
 * suite builds each mutant and checks that its pins reject it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

#define QK 32
#define Q4_0_BYTES 18
#define Q8_0_BYTES 34

/* ---------------------------------------------------------------- binary16 */

/* binary16 -> binary32, exact: normal (1024+m)*2^(e-25), subnormal m*2^-24. */
float orc_half_to_float(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return (float)(s ? -v : v);
}

/* Round a non-negative double with an integral-or-half fraction to the
 * nearest integer, ties to even (written out, independent of fenv). */
static double round_half_even(double q)
{
    double r = floor(q), frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    return r;
}

/* binary32 -> binary16, round to nearest even, subnormals kept, overflow to
 * infinity (IEEE 754 binary16: 1 sign, 5 exponent bits with bias 15, 10
 * fraction bits). */
uint16_t orc_float_to_half_rn(float f)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (isnan(f))
        return sign | 0x7E00;
    if (isinf(f))
        return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {                  /* subnormal: quantum 2^-24 */
        double q = a * 16777216.0;              /* exact */
#if ORC_MUTANT == 8
        double r = floor(q);                    /* MUTANT: truncation */
#else
        double r = round_half_even(q);
#endif
        return sign | (uint16_t)r;              /* r == 1024 is the smallest normal */
    }
    int e;
    frexp(a, &e);                               /* a in [2^(e-1), 2^e) */
    int E = e - 1;
    double q = ldexp(a, 10 - E);                /* in [1024, 2048), exact */
#if ORC_MUTANT == 8
    double r = floor(q);
#else
    double r = round_half_even(q);
#endif
    if (r == 2048.0) {
        r = 1024.0;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7C00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)r - 1024));
}

/* ------------------------------------------------------------ Q8_0 quantise */

static long g_range_violations = 0;

/* Number of |x * (1/d)| values that rounded beyond 127 so far (the
 * arithmetic bounds it by 127; a non-zero count flags a broken build). */
long orc_range_violations(void) { return g_range_violations; }

/* One block of 32 fp32 activations -> (fp16 d, int8 q[32]). */
void orc_quantize_block_q8_0(const float *x, uint16_t *d_out, int8_t *q)
{
    float amax = 0.0f;
    for (int j = 0; j < QK; j++) {
#if ORC_MUTANT == 7
        float a = x[j];                         /* MUTANT: signed max */
#else
        float a = fabsf(x[j]);
#endif
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    uint16_t dh = orc_float_to_half_rn(d);
#if ORC_MUTANT == 4
    float dr = orc_half_to_float(dh);           /* MUTANT: 1/d from fp16 d */
    float id = (dr != 0.0f) ? 1.0f / dr : 0.0f;
#else
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
#endif
    *d_out = dh;
    for (int j = 0; j < QK; j++) {
        float v = x[j] * id;
#if ORC_MUTANT == 3
        float r = rintf(v);                     /* MUTANT: ties to even */
#else
        float r = roundf(v);                    /* C99: halfway cases away from zero */
#endif
        if (r > 127.0f || r < -127.0f) {        /* unreachable for finite x: counted */
            g_range_violations++;
            r = r > 0.0f ? 127.0f : -127.0f;
        }
        q[j] = (int8_t)r;
    }
}

/* x fp32 [T][K] -> xq in GGML Q8_0 block layout [T][K/32][34]. */
void orc_quantize_q8_0(const float *x, int T, int64_t K, uint8_t *xq)
{
    int64_t nb = K / QK;
    for (int t = 0; t < T; t++)
        for (int64_t b = 0; b < nb; b++) {
            uint8_t *blk = xq + ((int64_t)t * nb + b) * Q8_0_BYTES;
            uint16_t d;
            int8_t q[QK];
            orc_quantize_block_q8_0(x + (int64_t)t * K + b * QK, &d, q);
            blk[0] = (uint8_t)(d & 0xFF);
            blk[1] = (uint8_t)(d >> 8);
            memcpy(blk + 2, q, QK);
        }
}

/* ------------------------------------------------------------ block sums */

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Nibble value of element e (0..31) of a Q4_0 block. */
static int q4_nibble(const uint8_t *wblk, int e)
{
#if ORC_MUTANT == 1
    e = (e + 16) % 32;                          /* MUTANT: swapped nibble halves */
#endif
    uint8_t byte = wblk[2 + (e % 16)];
    return e < 16 ? (byte & 0x0F) : (byte >> 4);
}

/* isum = sum_j (n_j - 8) * q_j over one block, exact int32 (|isum| <= 32512). */
int32_t orc_block_isum(const uint8_t *wblk, const uint8_t *xblk)
{
    const int8_t *q = (const int8_t *)(xblk + 2);
    int32_t s = 0;
    for (int j = 0; j < QK; j++) {
#if ORC_MUTANT == 2
        s += q4_nibble(wblk, j) * q[j];         /* MUTANT: -8 offset dropped */
#else
        s += (q4_nibble(wblk, j) - 8) * q[j];
#endif
    }
    return s;
}

static const uint8_t *xq_block(const uint8_t *xq, int64_t nb, int t, int64_t b)
{
#if ORC_MUTANT == 6
    b = (b + 1) % nb;                           /* MUTANT: wrong block index */
#endif
    return xq + ((int64_t)t * nb + b) * Q8_0_BYTES;
}

/* isums [T][N][nb] for W (GGML Q4_0, [N][nb][18]) and xq (GGML Q8_0). */
void orc_block_isums(const uint8_t *W, int64_t N, int64_t K, const uint8_t *xq, int T,
                     int32_t *isums)
{
    int64_t nb = K / QK;
    for (int t = 0; t < T; t++)
        for (int64_t i = 0; i < N; i++)
            for (int64_t b = 0; b < nb; b++)
                isums[((int64_t)t * N + i) * nb + b] =
                    orc_block_isum(W + (i * nb + b) * Q4_0_BYTES, xq_block(xq, nb, t, b));
}

/* ------------------------------------------------------------------ GEMV */

/* One output: y64 = sum_b d_w(i,b) * d_x(t,b) * isum(t,i,b) in fp64 (every
 * product exact), S = sum_b |same term| (the tolerance's scale). */
static void gemv_one(const uint8_t *W, int64_t nb, const uint8_t *xq, int t, int64_t i,
                     double *y, double *S)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *wblk = W + (i * nb + b) * Q4_0_BYTES;
        const uint8_t *xblk = xq_block(xq, nb, t, b);
        double dw = (double)orc_half_to_float(rd16(wblk));
#if ORC_MUTANT == 5
        double dx = 1.0;                        /* MUTANT: activation scale dropped */
#else
        double dx = (double)orc_half_to_float(rd16(xblk));
#endif
        double term = dw * dx * (double)orc_block_isum(wblk, xblk);
        acc += term;
        mag += fabs(term);
    }
    *y = acc;
    *S = mag;
}

/* y64, S: [T][N].  OpenMP over rows when built with -fopenmp. */
void orc_gemv_f64(const uint8_t *W, int64_t N, int64_t K, const uint8_t *xq, int T,
                  double *y64, double *S)
{
    int64_t nb = K / QK;
    for (int t = 0; t < T; t++) {
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < N; i++) {
#if ORC_MUTANT == 10
            int64_t o = i * T + t;              /* MUTANT: transposed output */
#else
            int64_t o = (int64_t)t * N + i;
#endif
            gemv_one(W, nb, xq, t, i, &y64[o], &S[o]);
        }
    }
}

/* The sequence epilogue (minfer README M19: the QKV bias and the residual
 * adds run in the GEMVs' epilogues): y64[t][i] = (W.x)[t][i] + bias[i] +
 * res[t][i] in fp64, either term absent when its pointer is NULL; S gains
 * |bias[i]| + |res[t][i]|, the scale of the two fp32 adds' rounding. */
void orc_gemv_ep_f64(const uint8_t *W, int64_t N, int64_t K, const uint8_t *xq, int T,
                     const float *bias, const float *res, double *y64, double *S)
{
    orc_gemv_f64(W, N, K, xq, T, y64, S);
    for (int t = 0; t < T; t++)
        for (int64_t i = 0; i < N; i++) {
            int64_t o = (int64_t)t * N + i;
            if (bias) {
                y64[o] += (double)bias[i];
                S[o] += fabs((double)bias[i]);
            }
            if (res) {
#if ORC_MUTANT == 18
                double r = (double)res[i];              /* MUTANT: residual of token 0 for every token */
#else
                double r = (double)res[o];
#endif
                y64[o] += r;
                S[o] += fabs(r);
            }
        }
}

/* Selected rows only: y64, S are [T][nrows]. */
void orc_gemv_rows_f64(const uint8_t *W, int64_t N, int64_t K, const uint8_t *xq, int T,
                       const int64_t *rows, int64_t nrows, double *y64, double *S)
{
    int64_t nb = K / QK;
    (void)N;
    for (int t = 0; t < T; t++)
        for (int64_t r = 0; r < nrows; r++)
            gemv_one(W, nb, xq, t, rows[r], &y64[(int64_t)t * nrows + r],
                     &S[(int64_t)t * nrows + r]);
}

/* ---------------------------------------------------------- Q8_0 weights */
/* A second weight format on the same path (minfer README "How it works":
 * gemv_q8_dp4a, int8 weights with int8 activations; M14: the lm_head held
 * as Q8_0): a weight block is the Q8_0 block itself, fp16 d then 32 int8 q,
 * and the weight is q * d (no offset). */

/* isum = sum_j w_j * q_j over one block, exact int32 (|isum| <= 32*127*127). */
int32_t orc_block_isum_q8(const uint8_t *wblk, const uint8_t *xblk)
{
    const int8_t *w = (const int8_t *)(wblk + 2);
    const int8_t *q = (const int8_t *)(xblk + 2);
    int32_t s = 0;
    for (int j = 0; j < QK; j++)
#if ORC_MUTANT == 13
        s += (int32_t)(uint8_t)w[j] * q[j];     /* MUTANT: weights read as unsigned */
#else
        s += (int32_t)w[j] * q[j];
#endif
    return s;
}

/* isums [T][N][nb] for W (GGML Q8_0, [N][nb][34]) and xq (GGML Q8_0). */
void orc_block_isums_q8(const uint8_t *W, int64_t N, int64_t K, const uint8_t *xq, int T, int32_t *isums)
{
    int64_t nb = K / QK;
    for (int t = 0; t < T; t++)
        for (int64_t i = 0; i < N; i++)
            for (int64_t b = 0; b < nb; b++)
                isums[((int64_t)t * N + i) * nb + b] =
                    orc_block_isum_q8(W + (i * nb + b) * Q8_0_BYTES, xq_block(xq, nb, t, b));
}

/* y64, S: [T][N], as orc_gemv_f64 with Q8_0 weight blocks. */
void orc_gemv_q8_f64(const uint8_t *W, int64_t N, int64_t K, const uint8_t *xq, int T, double *y64, double *S)
{
    int64_t nb = K / QK;
    for (int t = 0; t < T; t++) {
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < N; i++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t b = 0; b < nb; b++) {
                const uint8_t *wblk = W + (i * nb + b) * Q8_0_BYTES;
                const uint8_t *xblk = xq_block(xq, nb, t, b);
                double term = (double)orc_half_to_float(rd16(wblk)) * (double)orc_half_to_float(rd16(xblk)) *
                              (double)orc_block_isum_q8(wblk, xblk);
                acc += term;
                mag += fabs(term);
            }
            y64[(int64_t)t * N + i] = acc;
            S[(int64_t)t * N + i] = mag;
        }
    }
}

/* --------------------------------------------------------------- argmax */

/* Lowest index i with y[i] maximal; equality is IEEE == (-0 == +0). */
int64_t orc_argmax_f32(const float *y, int64_t N)
{
    int64_t best = 0;
    for (int64_t i = 1; i < N; i++) {
#if ORC_MUTANT == 9
        if (y[i] >= y[best])                    /* MUTANT: ties to highest index */
#else
        if (y[i] > y[best])
#endif
            best = i;
    }
    return best;
}

int64_t orc_argmax_f64(const double *y, int64_t N)
{
    int64_t best = 0;
    for (int64_t i = 1; i < N; i++)
        if (y[i] > y[best])
            best = i;
    return best;
}

/* ------------------------------------------------------------- FFN chain */
/* The decode FFN around the GEMVs (minfer README M15: one persistent kernel
 * runs every layer; colibri qwen36 docs: gate and up share one pass over the
 * activation): h = SiLU(g) * u with SiLU(g) = g / (1 + exp(-g)), then h is
 * quantised to Q8_0 for the down projection.  Every step is fp32, rounded to
 * nearest even, in the order written, so that the kernel's fp32 values and
 * codes can match exactly.
 *
 * exp by Cody and Waite's method (W. J. Cody, W. Waite, "Software Manual for
 * the Elementary Functions", 1980): x = k ln2 + r with k = rint(x log2 e) and
 * ln 2 split into a short head (exact k * head) and a tail, so r is formed
 * almost exactly; exp(r) by its Taylor series to r^7/7! in Horner form
 * (|r| <= ln2/2, truncation below 2^-27 relative); then the exact scale 2^k.
 * x is clamped to [-87, 88] so that 2^k stays a normal float. */
#define ORC_LOG2E 1.44269504088896340736f
#define ORC_LN2_HI 0.693145751953125f          /* 0x3F317200: 13 significant bits */
#define ORC_LN2_LO 1.42860682030941723212e-6f  /* ln 2 - ORC_LN2_HI */

float orc_exp_f32(float x)
{
    if (x > 88.0f) x = 88.0f;
    if (x < -87.0f) x = -87.0f;
    float k = rintf(x * ORC_LOG2E);
    float r = fmaf(-k, ORC_LN2_HI, x);
    r = fmaf(-k, ORC_LN2_LO, r);
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    union { uint32_t u; float f; } sc;
    sc.u = (uint32_t)((int)k + 127) << 23;
    return p * sc.f;
}

float orc_silu_f32(float g)
{
#if ORC_MUTANT == 14
    return g / (1.0f + orc_exp_f32(g));         /* MUTANT: exp(+g) */
#else
    return g / (1.0f + orc_exp_f32(-g));
#endif
}

void orc_exp_f32_n(const float *x, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_exp_f32(x[i]);
}

void orc_silu_f32_n(const float *x, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_silu_f32(x[i]);
}

/* h[t][j] = SiLU(g[t][j]) * u[t][j] (fp32 [T][F]), quantised to Q8_0 blocks
 * [T][F/32][34] as orc_quantize_q8_0 does. */
void orc_silu_mul_quantize(const float *g, const float *u, int T, int64_t F, uint8_t *hq, float *h_out)
{
    float *h = (float *)malloc(sizeof(float) * (size_t)T * (size_t)F);
    for (int64_t i = 0; i < (int64_t)T * F; i++) h[i] = orc_silu_f32(g[i]) * u[i];
    orc_quantize_q8_0(h, T, F, hq);
    if (h_out) memcpy(h_out, h, sizeof(float) * (size_t)T * (size_t)F);
    free(h);
}

/* ------------------------------------------------ top-2 and the commit rule */

/* The two best rows of y: idx[0] is the argmax (lowest index among equal
 * maxima); idx[1] is the argmax of the remaining rows, with the same rules
 * (minfer README M19 keeps the top-2 margin of every step).  idx[1] = -1
 * when N < 2. */
void orc_top2_f32(const float *y, int64_t N, int64_t idx[2])
{
    idx[0] = orc_argmax_f32(y, N);
    idx[1] = -1;
    for (int64_t i = 0; i < N; i++) {
        if (i == idx[0]) continue;
#if ORC_MUTANT == 11
        if (idx[1] < 0 || y[i] >= y[idx[1]])    /* MUTANT: second ties to highest index */
#else
        if (idx[1] < 0 || y[i] > y[idx[1]])
#endif
            idx[1] = i;
    }
}

void orc_top2_f64(const double *y, int64_t N, int64_t idx[2])
{
    idx[0] = orc_argmax_f64(y, N);
    idx[1] = -1;
    for (int64_t i = 0; i < N; i++) {
        if (i == idx[0]) continue;
        if (idx[1] < 0 || y[i] > y[idx[1]]) idx[1] = i;
    }
}

/* The lossless verify rule (minfer README M17): a verify step runs the
 * current token and its drafts, tokens[0] = current, tokens[1..T-1] =
 * drafts; pred[t] is the greedy prediction after tokens[0..t].  The step
 * commits pred[0], then pred[t] for each t >= 1 while every draft so far
 * equalled the prediction before it (tokens[t] == pred[t-1]), up to and
 * including the first prediction that disagrees with its draft.  Returns
 * the number of committed predictions, 1..T. */
int orc_verify_commit(const int64_t *tokens, const int64_t *pred, int T)
{
    int n = 1;
#if ORC_MUTANT == 12
    while (n < T && tokens[n] == pred[n]) n++;  /* MUTANT: draft compared with its own prediction */
#else
    while (n < T && tokens[n] == pred[n - 1]) n++;
#endif
    return n;
}

/* ------------------------------------ gs64 planar int4, per-vector int8 */

/* A variant format (colibri qwen36 docs: the gs64 container and its planar
 * repack; the dense int8 IDOT activation contract).  Readings where the
 * pages are silent:
 *  - a gs64 group is 64 weights in 32 bytes: byte j (j < 32) holds element
 *    j in its low nibble and element j + 32 in its high nibble (so one AND
 *    and one shift give the two halves in order), and the weight is
 *    (n - 8) * s with one fp32 scale s per group, as Q4_0's offset;
 *  - the activation is quantised once per vector: s_x = amax / 127 over the
 *    whole row of K values (fp32, not rounded to fp16), 1/s_x from it (0 when
 *    amax = 0), q = round-half-away(x * (1/s_x)) as int8;
 *  - y = sum_g s_w[g] * s_x * isum_g, isum_g the exact int32 sum over the
 *    group, formed here in fp64 (every product exact). */

/* x fp32 [T][K] -> q int8 [T][K], s [T]. */
void orc_quantize_vec_i8(const float *x, int T, int64_t K, int8_t *q, float *s)
{
    for (int t = 0; t < T; t++) {
        const float *xr = x + (int64_t)t * K;
        float amax = 0.0f;
#if ORC_MUTANT == 20
        for (int64_t k = 0; k < (K < 32 ? K : 32); k++) {   /* MUTANT: the first block's maximum only */
#else
        for (int64_t k = 0; k < K; k++) {
#endif
            float a = fabsf(xr[k]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        s[t] = d;
        for (int64_t k = 0; k < K; k++) {
            float r = roundf(xr[k] * id);
            if (r > 127.0f) r = 127.0f;             /* unreachable for finite x */
            if (r < -127.0f) r = -127.0f;
            q[(int64_t)t * K + k] = (int8_t)r;
        }
    }
}

/* Nibble of element e (0..63) of a 32-byte gs64 group. */
static int gs64_nibble(const uint8_t *grp, int e)
{
#if ORC_MUTANT == 19
    return e % 2 == 0 ? (grp[e / 2] & 0x0F) : (grp[e / 2] >> 4);   /* MUTANT: GGML-style pairs */
#else
    return e < 32 ? (grp[e] & 0x0F) : (grp[e - 32] >> 4);
#endif
}

/* W nibbles [N][K/64][32], scales [N][K/64] fp32; q int8 [T][K], s [T]:
 * y64 = sum_g ws * s * isum_g, S = sum_g |same term|, both [T][N]. */
void orc_gemv_gs64_f64(const uint8_t *Wq, const float *Ws, int64_t N, int64_t K, const int8_t *q,
                       const float *s, int T, double *y64, double *S)
{
    int64_t ng = K / 64;
    for (int t = 0; t < T; t++) {
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < N; i++) {
            double acc = 0.0, sc = 0.0;
            for (int64_t g = 0; g < ng; g++) {
                const uint8_t *grp = Wq + (i * ng + g) * 32;
                const int8_t *qg = q + (int64_t)t * K + g * 64;
                int32_t isum = 0;
                for (int e = 0; e < 64; e++) isum += (gs64_nibble(grp, e) - 8) * (int32_t)qg[e];
                double term = (double)Ws[i * ng + g] * (double)s[t] * (double)isum;
                acc += term;
                sc += fabs(term);
            }
            y64[(int64_t)t * N + i] = acc;
            S[(int64_t)t * N + i] = sc;
        }
    }
}

/* ------------------------------------------ Q4_0 requantisation at load */

/* Weights requantised to Q4_0 blocks at load (minfer README M14: the
 * lm_head requantised from Q8_0 to q4_0, 248 MB to 131 MB; M18: the Q8_0
 * head of the smallest model requantised to q4_0 at load).  The pages fix
 * the block format, not its encoder; the reading here is the encoder of the
 * GGML q4_0 format the pages' models ship in:
 *  - m = the block's element of largest magnitude (the first on ties; a
 *    block of zeros gives m = +0);
 *  - d = m / -8 in fp32, so that m is code 0 (value -8d) and the code range
 *    0..15 covers [-8d, 7d];
 *  - 1/d from the fp32 d (0 when d = 0);
 *  - code n = min(15, floor(x * (1/d) + 8.5)): one fp32 multiply and one
 *    fp32 add, each rounded to nearest even (x * (1/d) lies in [-8, 8] up
 *    to rounding, so the sum is at least 0.49...);
 *  - d stored as fp16, round to nearest even.
 * When d is so small (an fp32 subnormal) that 1/d overflows to infinity,
 * the same operations give codes 0 (x < 0), 15 (x > 0) and 0 (x = 0, a NaN
 * sum), the clamp taken before the conversion.  Non-finite inputs give
 * unspecified codes. */
void orc_quantize_block_q4_0(const float *x, uint8_t *blk)
{
    float amax = 0.0f, m = 0.0f;
    for (int j = 0; j < QK; j++) {
        float a = fabsf(x[j]);
        if (a > amax) {
            amax = a;
#if ORC_MUTANT == 15
            m = a;                              /* MUTANT: the magnitude, not the signed value */
#else
            m = x[j];
#endif
        }
    }
    float d = m / -8.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    uint16_t dh = orc_float_to_half_rn(d);
    blk[0] = (uint8_t)(dh & 0xFF);
    blk[1] = (uint8_t)(dh >> 8);
    int n[QK];
    for (int j = 0; j < QK; j++) {
        float v = x[j] * id;
#if ORC_MUTANT == 16
        float s = v + 8.0f;                     /* MUTANT: rounds down instead of to nearest */
#else
        float s = v + 8.5f;
#endif
        /* min(15, floor(s)), taken so that an infinite s (1/d overflows when
         * d is an fp32 subnormal) gives 15 or 0 and a NaN gives 0 */
        int c = (s >= 15.0f) ? 15 : (s >= 0.0f) ? (int)floorf(s) : 0;
        n[j] = c;
    }
    for (int j = 0; j < 16; j++) blk[2 + j] = (uint8_t)(n[j] | (n[j + 16] << 4));
}

/* w fp32 [N][K] -> GGML Q4_0 blocks [N][K/32][18]. */
void orc_requant_f32_q4_0(const float *w, int64_t N, int64_t K, uint8_t *out)
{
    int64_t nb = N * (K / QK);
    for (int64_t b = 0; b < nb; b++) orc_quantize_block_q4_0(w + b * QK, out + b * Q4_0_BYTES);
}

/* GGML Q8_0 weight blocks [N][K/32][34] -> GGML Q4_0 blocks [N][K/32][18]:
 * each block decoded to fp32 (q * d, exact: an 8-bit integer times an
 * 11-bit significand), then encoded as above. */
void orc_requant_q8_0_q4_0(const uint8_t *w, int64_t N, int64_t K, uint8_t *out)
{
    int64_t nb = N * (K / QK);
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *src = w + b * Q8_0_BYTES;
        float d = orc_half_to_float(rd16(src));
        float x[QK];
        for (int j = 0; j < QK; j++) {
#if ORC_MUTANT == 17
            x[j] = (float)src[2 + j] * d;       /* MUTANT: codes read as unsigned */
#else
            x[j] = (float)(int8_t)src[2 + j] * d;
#endif
        }
        orc_quantize_block_q4_0(x, out + b * Q4_0_BYTES);
    }
}

/* ------------------------------------------------------------------ misc */

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the row loops from now on (n >= 1); returns the new count. */
int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int orc_mutant(void) { return ORC_MUTANT; }
