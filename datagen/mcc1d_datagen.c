/*
 * mcc1d_datagen.c - seeded synthetic inputs for the masked causal conv1d
 * backward: normal / uniform 16-bit tensors and the four mask patterns.
 *
 * This module holds none of the operation's arithmetic. It only draws
 * numbers. Both the GPU tests and the CPU oracle consume the bit patterns it
 * writes, so neither side regenerates anything.
 *
 * Generator: counter-based. Value n of stream s under seed k is
 *   mix(mix(k * G + s + 1) + (n + 1) * G)
 * with G = 0x9E3779B97F4A7C15 and mix() the output function of SplitMix64
 * (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014). Being a pure function of (k, s, n), it gives the
 * same numbers for any thread count and on any host.
 * Normals use the Box-Muller transform (cosine branch) on draws 2n and 2n+1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return mix(seed * GOLDEN + stream + 1);
}

static inline uint64_t draw(uint64_t key, uint64_t n) { return mix(key + (n + 1) * GOLDEN); }

/* uniform in [0,1) with 53 random bits */
static inline double unit_open1(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }
/* uniform in (0,1] */
static inline double unit_open0(uint64_t r) { return (double)((r >> 11) + 1) * 0x1.0p-53; }

/*
 * Double to 16-bit float (0 = bf16, 1 = fp16), round to nearest even, by
 * integer arithmetic on the double's IEEE bits. Values far outside the
 * format's range never arise from the distributions used here; they
 * saturate to infinity.
 */
static uint16_t to16(double v, int dtype)
{
    const int man = dtype == 0 ? 7 : 10, bias = dtype == 0 ? 127 : 15;
    const int emax_field = dtype == 0 ? 255 : 31;
    union { double d; uint64_t u; } c;
    c.d = v;
    uint16_t sign = (uint16_t)((c.u >> 63) << 15);
    int e = (int)((c.u >> 52) & 0x7FF);
    uint64_t frac = c.u & ((1ull << 52) - 1);
    if (e == 0 && frac == 0)
        return sign;
    if (e == 0x7FF)
        return (uint16_t)(sign | (emax_field << man) | (frac ? 1u << (man - 1) : 0));
    /* value = sig * 2^(e - 1075) with the implicit bit in sig (double subnormals
     * are far below either format's range and flush through the shift) */
    uint64_t sig = e ? (frac | (1ull << 52)) : frac;
    int ue = (e ? e : 1) - 1023;          /* unbiased exponent of the leading bit position 52 */
    int te = ue + bias;                   /* target exponent field if normal */
    int shift = 52 - man;                 /* bits to drop for a normal result */
    if (te <= 0) {                        /* subnormal in the target */
        shift += 1 - te;
        te = 0;
    }
    if (shift > 63)
        return sign;
    uint64_t kept = sig >> shift;
    uint64_t rest = sig & ((1ull << shift) - 1);
    uint64_t half = 1ull << (shift - 1);
    if (rest > half || (rest == half && (kept & 1)))
        kept += 1;
    /* kept includes the implicit bit for normals; add the exponent field so a
     * carry out of the mantissa bumps the exponent naturally */
    uint32_t out;
    if (te == 0)
        out = (uint32_t)kept;             /* may carry into the smallest normal */
    else
        out = ((uint32_t)(te - 1) << man) + (uint32_t)kept;
    if ((out >> man) >= (uint32_t)emax_field)
        out = (uint32_t)emax_field << man;
    return (uint16_t)(sign | out);
}

static int nthreads_of(int n)
{
#ifdef _OPENMP
    return n > 0 ? n : omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* out[n] = 16-bit(mean + std * N(0,1)) for n < count */
void mcc1d_gen_normal(uint16_t *out, int64_t count, int dtype, double mean, double std,
                      uint64_t seed, uint64_t stream, int nthreads)
{
    const uint64_t key = stream_key(seed, stream);
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static) num_threads(nthreads_of(nthreads))
    for (int64_t n = 0; n < count; ++n) {
        double u1 = unit_open0(draw(key, 2 * (uint64_t)n));
        double u2 = unit_open1(draw(key, 2 * (uint64_t)n + 1));
        double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        out[n] = to16(mean + std * z, dtype);
    }
}

/* out[n] = 16-bit(lo + (hi - lo) * U[0,1)) */
void mcc1d_gen_uniform(uint16_t *out, int64_t count, int dtype, double lo, double hi,
                       uint64_t seed, uint64_t stream, int nthreads)
{
    const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static) num_threads(nthreads_of(nthreads))
    for (int64_t n = 0; n < count; ++n)
        out[n] = to16(lo + (hi - lo) * unit_open1(draw(key, (uint64_t)n)), dtype);
}

/* 16-bit pattern of a double, exposed for the generator's own tests */
uint16_t mcc1d_gen_to16(double v, int dtype) { return to16(v, dtype); }

/* mask[j*S+i] = 1 with probability p, independently per position */
void mcc1d_gen_mask_bernoulli(uint8_t *mask, int64_t B, int64_t S, double p,
                              uint64_t seed, uint64_t stream)
{
    const uint64_t key = stream_key(seed, stream);
    for (int64_t n = 0; n < B * S; ++n)
        mask[n] = unit_open1(draw(key, (uint64_t)n)) < p ? 1 : 0;
}

/* Padding-style mask: batch j keeps a prefix of length L_j drawn uniformly
 * from the integers floor(S/2) .. S inclusive; the rest is zero. */
void mcc1d_gen_mask_prefix(uint8_t *mask, int64_t B, int64_t S, uint64_t seed, uint64_t stream,
                           int64_t *lengths_out)
{
    const uint64_t key = stream_key(seed, stream);
    const int64_t lo = S / 2, span = S - lo + 1;
    for (int64_t j = 0; j < B; ++j) {
        int64_t L = lo + (int64_t)(unit_open1(draw(key, (uint64_t)j)) * (double)span);
        if (L > S)
            L = S;
        if (lengths_out)
            lengths_out[j] = L;
        for (int64_t i = 0; i < S; ++i)
            mask[j * S + i] = i < L ? 1 : 0;
    }
}

/* Span mask: per batch, zero spans with start uniform in 0..S-1 and length
 * uniform in lmin..lmax (clipped at S) are laid down, overlaps allowed,
 * until at least frac*S positions of that batch are zero. */
void mcc1d_gen_mask_spans(uint8_t *mask, int64_t B, int64_t S, double frac, int64_t lmin,
                          int64_t lmax, uint64_t seed, uint64_t stream)
{
    const uint64_t key = stream_key(seed, stream);
    for (int64_t j = 0; j < B; ++j) {
        uint8_t *m = mask + j * S;
        for (int64_t i = 0; i < S; ++i)
            m[i] = 1;
        int64_t zeros = 0;
        uint64_t n = (uint64_t)j << 32; /* each batch has its own counter range */
        while ((double)zeros < frac * (double)S) {
            int64_t start = (int64_t)(unit_open1(draw(key, n++)) * (double)S);
            int64_t len = lmin + (int64_t)(unit_open1(draw(key, n++)) * (double)(lmax - lmin + 1));
            if (start >= S)
                start = S - 1;
            int64_t end = start + len < S ? start + len : S;
            for (int64_t i = start; i < end; ++i)
                if (m[i]) {
                    m[i] = 0;
                    ++zeros;
                }
        }
    }
}
