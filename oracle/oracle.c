/*
 * oracle.c -- plain, slow, obviously-correct CPU definition of the
 * weight-quantized linear layer (W4A16, W4A8, W8A16), the per-token int8
 * activation quantizer, the int8 group-128 weight round trip, the int8
 * group-128 embedding gather and the top-k over logits.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * Source: "What this repo does that stock vLLM doesn't" (qwen38-27b-rtx3090
 * docs/optimizations.md), section "In full", item 4 ("int8 tensor cores for the
 * batched GEMMs, with a bug fix"): weights stay int4 with symmetric group
 * scales (about half of them negative), activations are quantized to int8 per
 * token, and the fix keeps the sign of each group scale.  Item 1 of the same
 * section: lm_head / embed_tokens requantized to int8 group-128 with a ~0.6 %
 * round-trip error.  Item 5: the 248k-row lm_head.
 *
 * The pages give no formula, so each function below writes out the plain
 * definition ("dequantize, then multiply"):
 *
 *   y[m,n] = fp16_rne( sum_g s[n,g] * sum_{k in g} x[m,k] * q[n,k] )      (W4A16/W8A16)
 *   y[m,n] = fp16_rne( sx[m] * sum_g s[n,g] * sum_{k in g} qa[m,k]*q[n,k] ) (W4A8)
 *
 * with g = k / 128 and all arithmetic in IEEE binary64 (the W4A8 inner sums
 * are exact 64-bit integers).  The activation quantizer follows the symmetric
 * per-token reading:  amax = max_k |x|,  s = amax / 127 (binary32, IEEE
 * divide, round-to-nearest-even),  q = clamp(rne(x / s), -127, 127), and an
 * all-zero row gives s = 0 and q = 0.
 *
 * Build: cc -O2 -std=c11 -fopenmp -ffp-contract=off -fno-fast-math -fPIC -shared
 * (no contraction, so that float expressions are evaluated exactly as written).
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#include <fenv.h>
#include <stdlib.h>

#define GROUP 128

/* ---------- IEEE binary16 <-> binary64, written from the format definition ---------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)            /* zero or subnormal: f * 2^-24 */
        v = ldexp((double)f, -24);
    else if (e == 31)      /* inf / nan */
        v = f ? NAN : INFINITY;
    else                   /* normal: (1024 + f) * 2^(e - 25) */
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Round a binary64 value to the nearest binary16, ties to even. */
uint16_t oracle_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return 0x7e00;
    /* 65504 is the largest finite half; halfway to the next binade step (65520)
       and beyond rounds to infinity (65520 ties to the even value 2^16). */
    if (a >= 65520.0) return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: integer multiple n of 2^-24, n in [0, 1024];
           n == 1024 is the smallest normal and its bits are exactly 0x0400 */
        double n = nearbyint(ldexp(a, 24));   /* scaling by 2^24 is exact */
        return sign | (uint16_t)n;
    }
    int e;
    (void)frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) -> unbiased exp e-1 */
    int ue = e - 1;              /* a in [2^ue, 2^(ue+1)) */
    double n = nearbyint(ldexp(a, 10 - ue));  /* n in [1024, 2048] */
    if (n == 2048.0) { n = 1024.0; ue += 1; }
    if (ue > 15) return sign | 0x7c00;
    return sign | (uint16_t)(((ue + 15) << 10) | ((int)n - 1024));
}

/* ---------- per-token int8 activation quantizer ---------- */

/* x: [M,K] binary16 bits, row-major.  q: [M,K] int8.  s: [M] binary32. */
int oracle_quant_act_int8(const uint16_t *x, int64_t M, int64_t K,
                          int8_t *q, float *s)
{
    if (M < 0 || K < 0) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = x + m * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = (float)oracle_half_to_double(row[k]);   /* exact */
            float b = fabsf(a);
            if (b > amax) amax = b;
        }
        float sm = amax / 127.0f;             /* IEEE binary32 divide, RNE */
        s[m] = (amax == 0.0f) ? 0.0f : sm;
        for (int64_t k = 0; k < K; ++k) {
            if (amax == 0.0f) { q[m * K + k] = 0; continue; }
            float a = (float)oracle_half_to_double(row[k]);
            float r = nearbyintf(a / sm);      /* IEEE divide, then RNE */
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[m * K + k] = (int8_t)r;
        }
    }
    return 0;
}

/* ---------- weight-only GEMM with fp16 activations (W4A16 and W8A16) ---------- */

static int check_codes(const int8_t *codes, int64_t count, int lo, int hi)
{
    for (int64_t i = 0; i < count; ++i)
        if (codes[i] < lo || codes[i] > hi) return -3;
    return 0;
}

/*
 * x: [M,K] binary16, codes: [N,K] int8 (logical weight W[n,k] = codes*scale),
 * scales: [N, K/128] binary16 (signed), y: [M,N] binary16.
 * y[m,n] = fp16( sum_g s[n,g] * sum_{k in g} x[m,k] * codes[n,k] ), all in binary64.
 */
static int gemm_wxa16(const uint16_t *x, const int8_t *codes, const uint16_t *scales,
                      int64_t M, int64_t N, int64_t K, uint16_t *y)
{
    if (M < 0 || N < 0 || K < 0 || K % GROUP) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
    int64_t G = K / GROUP;
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                double inner = 0.0;
                for (int64_t k = g * GROUP; k < (g + 1) * GROUP; ++k)
                    inner += oracle_half_to_double(x[m * K + k]) * (double)codes[n * K + k];
                acc += oracle_half_to_double(scales[n * G + g]) * inner;
            }
            y[m * N + n] = oracle_double_to_half(acc);
        }
    }
    return 0;
}

/* W4A16: codes must lie in [-8, 7] (signed int4). */
int oracle_w4a16(const uint16_t *x, const int8_t *codes, const uint16_t *scales,
                 int64_t M, int64_t N, int64_t K, uint16_t *y)
{
    int rc = check_codes(codes, N * K, -8, 7);
    if (rc) return rc;
    return gemm_wxa16(x, codes, scales, M, N, K, y);
}

/* W8A16: any int8 code. */
int oracle_w8a16(const uint16_t *x, const int8_t *codes, const uint16_t *scales,
                 int64_t M, int64_t N, int64_t K, uint16_t *y)
{
    return gemm_wxa16(x, codes, scales, M, N, K, y);
}

/*
 * W4A8: qa: [M,K] int8 activation codes, sx: [M] binary32 token scales,
 * codes [N,K] in [-8,7], scales [N,K/128] binary16.
 * y[m,n] = fp16( sx[m] * sum_g s[n,g] * (int64) sum_{k in g} qa[m,k]*codes[n,k] ).
 */
int oracle_w4a8(const int8_t *qa, const float *sx, const int8_t *codes,
                const uint16_t *scales, int64_t M, int64_t N, int64_t K, uint16_t *y)
{
    if (M < 0 || N < 0 || K < 0 || K % GROUP) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
    int rc = check_codes(codes, N * K, -8, 7);
    if (rc) return rc;
    int64_t G = K / GROUP;
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                int64_t inner = 0;
                for (int64_t k = g * GROUP; k < (g + 1) * GROUP; ++k)
                    inner += (int64_t)qa[m * K + k] * (int64_t)codes[n * K + k];
                acc += oracle_half_to_double(scales[n * G + g]) * (double)inner;
            }
            y[m * N + n] = oracle_double_to_half((double)sx[m] * acc);
        }
    }
    return 0;
}

/* ---------- int8 group-128 weight round trip (lm_head / embed requantizer) ---------- */

/*
 * w: [N,K] binary32 weights.  Per row n and group g:
 *   amax = max |w|,  s = fp16(amax / 127) (the stored scale),
 *   q = clamp(rne(w / s), -127, 127),  w_hat = q * s.
 * Writes codes [N,K], scales [N,K/128] (binary16 bits) and returns, through
 * rel_err, ||w - w_hat||_F / ||w||_F computed in binary64.
 */
int oracle_roundtrip_int8_g128(const float *w, int64_t N, int64_t K,
                               int8_t *codes, uint16_t *scales, double *rel_err)
{
    if (N < 0 || K < 0 || K % GROUP) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
    int64_t G = K / GROUP;
    double num = 0.0, den = 0.0;
    #pragma omp parallel for schedule(static) reduction(+:num, den)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const float *wg = w + n * K + g * GROUP;
            double amax = 0.0;
            for (int k = 0; k < GROUP; ++k)
                if (fabs((double)wg[k]) > amax) amax = fabs((double)wg[k]);
            uint16_t sh = oracle_double_to_half(amax / 127.0);
            double s = oracle_half_to_double(sh);
            scales[n * G + g] = sh;
            for (int k = 0; k < GROUP; ++k) {
                double r = 0.0;
                if (s != 0.0) {
                    r = nearbyint((double)wg[k] / s);
                    if (r > 127.0) r = 127.0;
                    if (r < -127.0) r = -127.0;
                }
                codes[n * K + g * GROUP + k] = (int8_t)r;
                double d = (double)wg[k] - r * s;
                num += d * d;
                den += (double)wg[k] * (double)wg[k];
            }
        }
    }
    *rel_err = den > 0.0 ? sqrt(num / den) : 0.0;
    return 0;
}

/* ---------- dequant-on-gather embedding (int8 group-128 table) ---------- */

/*
 * "What this repo does that stock vLLM doesn't", "In full" items 1 and 2: the
 * embedding table is requantized to int8 with group-128 fp16 scales and read
 * through a dequant-on-gather kernel.  For token t and feature k:
 *   out[t,k] = fp16_rne( codes[ids[t],k] * scales[ids[t], k/128] )
 * (the product of an 8-bit code and an 11-bit scale is exact in binary64).
 * ids [T] int64, codes [V,D] int8, scales [V,D/128] binary16, out [T,D] binary16.
 * Returns -4 (rows set to zero) when an id lies outside [0, V).
 */
int oracle_embed_w8(const int64_t *ids, int64_t T, const int8_t *codes, const uint16_t *scales,
                    int64_t V, int64_t D, uint16_t *out)
{
    if (T < 0 || V < 0 || D < 0 || D % GROUP) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
    int64_t G = D / GROUP;
    int bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        int64_t v = ids[t];
        if (v < 0 || v >= V) {
            for (int64_t k = 0; k < D; ++k) out[t * D + k] = 0;
            bad = 1;
            continue;
        }
        for (int64_t k = 0; k < D; ++k) {
            double s = oracle_half_to_double(scales[v * G + k / GROUP]);
            out[t * D + k] = oracle_double_to_half((double)codes[v * D + k] * s);
        }
    }
    return bad ? -4 : 0;
}

/* ---------- top-k over logits ---------- */

/*
 * "What this repo does that stock vLLM doesn't", "In full" item 6: with top-k
 * known on the host the sampler's mask is a small top-k over the logits.  Per
 * row: the k largest values, largest first, ties broken by the smaller index
 * (values compared as numbers, so -0 and +0 tie).
 * logits [M,N] binary16 (no NaN), vals [M,k] binary16, idx [M,k] int64.
 */
static const uint16_t *g_topk_row;
static int topk_cmp(const void *a, const void *b)
{
    int64_t i = *(const int64_t *)a, j = *(const int64_t *)b;
    double vi = oracle_half_to_double(g_topk_row[i]), vj = oracle_half_to_double(g_topk_row[j]);
    if (vi > vj) return -1;
    if (vi < vj) return 1;
    return (i < j) ? -1 : (i > j) ? 1 : 0;
}

int oracle_topk(const uint16_t *logits, int64_t M, int64_t N, int64_t k, uint16_t *vals, int64_t *idx)
{
    if (M < 0 || N < 0 || k < 0 || k > N) return -1;
    int64_t *order = (int64_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
    if (!order) return -5;
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = logits + m * N;
        for (int64_t n = 0; n < N; ++n) {
            if (oracle_half_to_double(row[n]) != oracle_half_to_double(row[n])) { free(order); return -6; }
            order[n] = n;
        }
        g_topk_row = row;           /* qsort has no context argument; single-threaded */
        qsort(order, (size_t)N, sizeof(int64_t), topk_cmp);
        for (int64_t j = 0; j < k; ++j) {
            idx[m * k + j] = order[j];
            vals[m * k + j] = row[order[j]];
        }
    }
    free(order);
    return 0;
}
