/*
 * mcc1d_oracle.c - CPU oracle for the masked causal depthwise conv1d backward.
 *
 * TEST INFRASTRUCTURE ONLY. This is the slow, plain, fp64 statement of what
 * the operation computes, kept to check the GPU library against. Only the
 * test suite, the package smoke check and the benchmark's CPU-baseline leg
 * load it. The GPU library never calls it and shares no code, header, table
 * or helper with it.
 *
 * Source: CANN operator page "aclnnMaskedCausalConv1dBackward",
 * section 功能说明 (function description), 计算公式 (formulas). With the
 * tensors gradY, x and gradX laid out [S,B,H], weight [W,H] and the bool
 * mask [B,S], i the S index, j the B index and k the tap index:
 *
 *   gradYMasked(i,j,h) = mask(j,i) * gradY(i,j,h)
 *   gradX(i,j,h)       = sum over k=0..W-1 of gradYMasked(i+k,j,h) * weight(W-1-k,h)
 *   gradWeight(k,h)    = sum over j=0..B-1, i=0..S-1 of
 *                        gradYMasked(i+W-1-k,j,h) * x(i,j,h)
 *
 * A term whose S index lands outside [0,S) is zero (the page pads invalid
 * positions with zeros); the sequences of different batches never touch;
 * H is the elementwise (depthwise) axis that the page leaves out of the
 * formulas. A null mask means every position is kept (the mask input is
 * optional and defaults to nullptr in the parameter table, 参数说明).
 *
 * Arithmetic: every 16-bit input is decoded exactly to double, every sum is
 * taken in double in the formula's own order, and each result is rounded
 * once, to nearest with ties to even, straight from double to the 16-bit
 * output format by the converter in this file. The page fixes neither the
 * accumulation precision nor the rounding; fp64 with a single final rounding
 * is the reading taken here.
 *
 * Nothing here is blocked, fused or reordered: loops run over the formula's
 * indices, and the only parallelism (OpenMP, optional) splits independent
 * outputs (rows of gradX, columns h of gradWeight), never one sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* 16-bit floating formats of the page's parameter table: BFLOAT16, FLOAT16. */
enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1 };

typedef struct {
    int man_bits; /* stored mantissa bits */
    int exp_bits; /* exponent field width */
    int bias;     /* exponent bias */
    int emin;     /* exponent of the smallest normal */
    int emax;     /* exponent of the largest finite binade */
} fmt16;

static fmt16 fmt_of(int dtype)
{
    fmt16 f;
    if (dtype == ORACLE_BF16) {
        f.man_bits = 7; f.exp_bits = 8; f.bias = 127; f.emin = -126; f.emax = 127;
    } else {
        f.man_bits = 10; f.exp_bits = 5; f.bias = 15; f.emin = -14; f.emax = 15;
    }
    return f;
}

/* Exact value of a bf16 / fp16 bit pattern (IEEE 754 binary16 layout for fp16,
 * the upper half of binary32 for bf16), subnormals included. */
double mcc1d_oracle_to_double(uint16_t bits, int dtype)
{
    fmt16 f = fmt_of(dtype);
    unsigned sign = bits >> 15;
    unsigned e = (bits >> f.man_bits) & ((1u << f.exp_bits) - 1u);
    unsigned m = bits & ((1u << f.man_bits) - 1u);
    double v;
    if (e == (1u << f.exp_bits) - 1u)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, f.emin - f.man_bits);
    else
        v = ldexp((double)(m | (1u << f.man_bits)), (int)e - f.bias - f.man_bits);
    return sign ? -v : v;
}

/* Round a double once to the 16-bit format: nearest, ties to even, with
 * gradual underflow and overflow to infinity. */
uint16_t mcc1d_oracle_from_double(double v, int dtype)
{
    fmt16 f = fmt_of(dtype);
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    uint16_t inf_bits = (uint16_t)(sign | (((1u << f.exp_bits) - 1u) << f.man_bits));
    if (isnan(v))
        return (uint16_t)(inf_bits | (1u << (f.man_bits - 1)));
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return inf_bits;
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;            /* a lies in [2^E, 2^(E+1)) */
    if (E < f.emin)
        E = f.emin;            /* below the normals the spacing stays 2^(emin-man_bits) */
    double q = ldexp(a, f.man_bits - E); /* a in units of the target spacing; exact */
    double r = floor(q);
    double d = q - r;
    if (d > 0.5 || (d == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    if (r >= ldexp(1.0, f.man_bits + 1)) { /* carried into the next binade */
        r = ldexp(1.0, f.man_bits);
        E += 1;
    }
    if (E > f.emax)
        return inf_bits;
    unsigned ri = (unsigned)r;
    if (ri < (1u << f.man_bits)) /* subnormal (E == emin) */
        return (uint16_t)(sign | ri);
    return (uint16_t)(sign | ((unsigned)(E + f.bias) << f.man_bits) | (ri - (1u << f.man_bits)));
}

static double *decode_table(int dtype)
{
    double *t = (double *)malloc(65536 * sizeof(double));
    if (!t)
        return NULL;
    for (uint32_t b = 0; b < 65536u; ++b)
        t[b] = mcc1d_oracle_to_double((uint16_t)b, dtype);
    return t;
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
    return nthreads;
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of threads a call with this request actually uses. */
int mcc1d_oracle_threads(int nthreads) { return set_threads(nthreads); }

/* gradYMasked(i,j,h): the literal product mask(j,i) * gradY(i,j,h), zero
 * outside [0,S). */
static inline double gym(const double *tab, const uint16_t *gy, const uint8_t *mask,
                         int64_t S, int64_t B, int64_t H, int64_t i, int64_t j, int64_t h)
{
    if (i < 0 || i >= S)
        return 0.0;
    double m = mask ? (mask[j * S + i] ? 1.0 : 0.0) : 1.0;
    return m * tab[gy[(i * B + j) * H + h]];
}

/*
 * Full backward. gradY, x: [S,B,H]; weight: [W,H]; mask: [B,S] bytes or NULL.
 * Outputs (each may be NULL): gx_bits / gx_exact [S,B,H], gw_bits / gw_exact /
 * gw_abs [W,H]. gw_abs(k,h) is the sum of the absolute values of the terms of
 * gradWeight(k,h), the scale its tolerance is stated against.
 * Returns 0, or -1 on a bad argument or allocation failure.
 */
int mcc1d_oracle_bwd(int64_t S, int64_t B, int64_t H, int64_t W, int dtype,
                     const uint16_t *gy, const uint16_t *x, const uint16_t *w,
                     const uint8_t *mask,
                     uint16_t *gx_bits, double *gx_exact,
                     uint16_t *gw_bits, double *gw_exact, double *gw_abs,
                     int nthreads)
{
    if (S < 1 || B < 1 || H < 1 || W < 1 || (dtype != ORACLE_BF16 && dtype != ORACLE_FP16))
        return -1;
    if (!gy || !w || ((gw_bits || gw_exact || gw_abs) && !x))
        return -1;
    double *tab = decode_table(dtype);
    if (!tab)
        return -1;
    int nt = set_threads(nthreads);

    /* gradX(i,j,h) = sum_k gradYMasked(i+k,j,h) * weight(W-1-k,h) */
    if (gx_bits || gx_exact) {
        int64_t rows = S * B;
#pragma omp parallel for schedule(static) num_threads(nt)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t i = r / B, j = r % B;
            for (int64_t h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int64_t k = 0; k < W; ++k)
                    acc += gym(tab, gy, mask, S, B, H, i + k, j, h) * tab[w[(W - 1 - k) * H + h]];
                int64_t o = (i * B + j) * H + h;
                if (gx_exact)
                    gx_exact[o] = acc;
                if (gx_bits)
                    gx_bits[o] = mcc1d_oracle_from_double(acc, dtype);
            }
        }
    }

    /* gradWeight(k,h) = sum_j sum_i gradYMasked(i+W-1-k,j,h) * x(i,j,h) */
    if (gw_bits || gw_exact || gw_abs) {
        double *acc = (double *)calloc((size_t)(W * H), sizeof(double));
        double *mag = (double *)calloc((size_t)(W * H), sizeof(double));
        if (!acc || !mag) {
            free(acc); free(mag); free(tab);
            return -1;
        }
        /* Each thread owns a range of h and runs the whole j, i loop for it,
         * so every (k,h) sum is taken in the order j, then i. */
#pragma omp parallel num_threads(nt)
        {
            int tid = 0, nth = 1;
#ifdef _OPENMP
            tid = omp_get_thread_num();
            nth = omp_get_num_threads();
#endif
            int64_t h0 = H * tid / nth, h1 = H * (tid + 1) / nth;
            for (int64_t j = 0; j < B; ++j)
                for (int64_t i = 0; i < S; ++i)
                    for (int64_t k = 0; k < W; ++k)
                        for (int64_t h = h0; h < h1; ++h) {
                            double t = gym(tab, gy, mask, S, B, H, i + W - 1 - k, j, h) *
                                       tab[x[(i * B + j) * H + h]];
                            acc[k * H + h] += t;
                            mag[k * H + h] += fabs(t);
                        }
        }
        for (int64_t c = 0; c < W * H; ++c) {
            if (gw_exact)
                gw_exact[c] = acc[c];
            if (gw_abs)
                gw_abs[c] = mag[c];
            if (gw_bits)
                gw_bits[c] = mcc1d_oracle_from_double(acc[c], dtype);
        }
        free(acc);
        free(mag);
    }
    free(tab);
    return 0;
}

/*
 * gradX at n chosen flat positions idx[] of the [S,B,H] tensor, one at a
 * time, by the same formula. For tensors too large to check in full.
 */
int mcc1d_oracle_gradx_at(int64_t S, int64_t B, int64_t H, int64_t W, int dtype,
                          const uint16_t *gy, const uint16_t *w, const uint8_t *mask,
                          int64_t n, const int64_t *idx, uint16_t *out_bits, double *out_exact)
{
    if (S < 1 || B < 1 || H < 1 || W < 1 || !gy || !w || !idx || n < 0)
        return -1;
    for (int64_t t = 0; t < n; ++t) {
        int64_t o = idx[t];
        if (o < 0 || o >= S * B * H)
            return -1;
        int64_t h = o % H, r = o / H, j = r % B, i = r / B;
        double acc = 0.0;
        for (int64_t k = 0; k < W; ++k) {
            double g = 0.0; /* gradYMasked(i+k,j,h), zero past the end of S */
            if (i + k < S) {
                double m = mask ? (mask[j * S + i + k] ? 1.0 : 0.0) : 1.0;
                g = m * mcc1d_oracle_to_double(gy[((i + k) * B + j) * H + h], dtype);
            }
            acc += g * mcc1d_oracle_to_double(w[(W - 1 - k) * H + h], dtype);
        }
        if (out_exact)
            out_exact[t] = acc;
        if (out_bits)
            out_bits[t] = mcc1d_oracle_from_double(acc, dtype);
    }
    return 0;
}

/*
 * The forward pass that this backward differentiates. The page names the
 * forward operator (MaskedCausalConv1d) but prints only the backward;
 * transposing the two backward formulas gives
 *
 *   y(t,j,h) = mask(j,t) * sum over k=0..W-1 of weight(k,h) * x(t-(W-1)+k, j, h)
 *
 * with x zero at negative S indices: a causal depthwise convolution with W-1
 * positions of left padding and the mask on its output (the parameter table
 * describes the mask as the convolution's output mask).
 * Outputs (either may be NULL): y [S,B,H] fp64, y_bits [S,B,H] the same
 * values rounded once to the 16-bit type.
 */
int mcc1d_oracle_fwd(int64_t S, int64_t B, int64_t H, int64_t W, int dtype,
                     const uint16_t *x, const uint16_t *w, const uint8_t *mask, double *y,
                     uint16_t *y_bits, int nthreads)
{
    if (S < 1 || B < 1 || H < 1 || W < 1 || !x || !w || (!y && !y_bits))
        return -1;
    double *tab = decode_table(dtype);
    if (!tab)
        return -1;
    int nt = set_threads(nthreads);
    int64_t rows = S * B;
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t t = r / B, j = r % B;
        double m = mask ? (mask[j * S + t] ? 1.0 : 0.0) : 1.0;
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t k = 0; k < W; ++k) {
                int64_t s = t - (W - 1) + k;
                if (s >= 0)
                    acc += tab[w[k * H + h]] * tab[x[(s * B + j) * H + h]];
            }
            int64_t o = (t * B + j) * H + h;
            if (y)
                y[o] = m * acc;
            if (y_bits)
                y_bits[o] = mcc1d_oracle_from_double(m * acc, dtype);
        }
    }
    free(tab);
    return 0;
}
