/*
 * q4_0_oracle.c -- plain, slow, obviously-correct CPU reference for the
 * Q4_0 weight-only matmul.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg load this file's library; the
 * product library never does, and this file shares no code, header, table or
 * constant with the CUDA sources.
 *
 * What is computed, and where it comes from:
 *   - "Vertical disaggregation: maximizing model throughput on heterogeneous
 *     silicon", section "Every cycle counts: custom kernels": CPU and GPU share
 *     ONE Q4_0 weight format, the output is deterministic, and the kernels are
 *     built from nibble unpack, dot product and scale apply.  The page names
 *     Q4_0 but prints no byte layout, quantizer or precision.
 *   - The Q4_0 block this library fixes: 32 consecutive weights along K, one
 *     IEEE binary16 scale d followed by 16 bytes of 4-bit codes q; element j
 *     (0..15) is the low nibble of code byte j, element j+16 its high nibble;
 *     w = d * (q - 8).  Quantizer: d = (signed value of the max-|w| element)
 *     / -8 and q = clamp(round(w / d) + 8, 0, 15).
 *   - Where the above leaves a step open, the reading taken is (all listed in
 *     the design notes): first index wins a tie on max-|w|; d is formed in
 *     fp32 and w is divided by that fp32 d (correctly rounded IEEE division);
 *     round() is half-away-from-zero; an all-zero block stores d = +0 and
 *     codes 8; the stored scale is fp32 d rounded to binary16, nearest-even.
 *   - The matmul is the plain definition y[m,n] = sum_k w[n,k] * x[m,k] with
 *     w decoded exactly into fp64 and x (bf16) widened exactly, summed in fp64
 *     in ascending k.
 *
 * The quantizer's integer decision (the code) is taken in fp32 because that
 * is the precision the device quantizer decides it in; everything else is
 * fp64.  Build flags: -O2 -fno-fast-math -ffp-contract=off -fopenmp.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake; the
 * CPU tests build each mutant and check that at least one pin fails.  Never
 * set it for a real build.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_QK 32          /* weights per block */

/* The scale's bits from the first two bytes of a block (little-endian). */
#if ORACLE_MUTANT == 10
#define ORACLE_D_BITS(blk) ((uint16_t)((blk)[1] | ((blk)[0] << 8))) /* mutant: scale bytes swapped */
#else
#define ORACLE_D_BITS(blk) ((uint16_t)((blk)[0] | ((blk)[1] << 8)))
#endif
#define ORACLE_BLOCK_BYTES 18 /* 2 bytes of d + 16 bytes of codes */

/* ---------------------------------------------------------------- binary16 */

static int oracle_lead_bit(uint64_t v) {
    int p = -1;
    while (v) { v >>= 1; ++p; }
    return p;
}

/* IEEE 754 binary32 -> binary16, round to nearest, ties to even, with
 * subnormals, overflow to infinity and quiet NaNs. */
uint16_t oracle_f32_to_f16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t ex = (u >> 23) & 0xFFu, man = u & 0x7FFFFFu;
    if (ex == 0xFFu)
        return man ? (uint16_t)(sign | 0x7E00u | (man >> 13)) : (uint16_t)(sign | 0x7C00u);
    if (ex == 0 && man == 0) return sign;
    uint64_t sig;
    int e2; /* |f| = sig * 2^e2 exactly */
    if (ex == 0) { sig = man; e2 = -149; }
    else { sig = man | 0x800000u; e2 = (int)ex - 150; }
    int expo = oracle_lead_bit(sig) + e2;  /* |f| in [2^expo, 2^(expo+1)) */
    int quantum = expo - 10;               /* binary16 spacing at this magnitude */
    if (quantum < -24) quantum = -24;      /* ... floored by the subnormal spacing */
    int shift = quantum - e2;              /* n = sig / 2^shift, rounded */
    uint64_t n;
    if (shift <= 0) {
        n = sig << (-shift);
    } else if (shift >= 63) {
        n = 0;
    } else {
        uint64_t rem = sig & ((1ull << shift) - 1), half = 1ull << (shift - 1);
        n = sig >> shift;
#if ORACLE_MUTANT == 8
        (void)rem; (void)half;           /* mutant: truncate instead of rounding */
#else
        if (rem > half || (rem == half && (n & 1u))) ++n;
#endif
    }
    if (n == 2048) { n = 1024; ++quantum; } /* rounding carried into the exponent */
    if (quantum == -24 && n < 1024) return (uint16_t)(sign | n); /* subnormal */
    int biased = quantum + 25;
    if (biased >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | ((uint32_t)biased << 10) | (uint32_t)(n - 1024));
}

/* Array form of the converter above (used by the exhaustive pin). */
void oracle_f32_to_f16_array(const float *in, uint16_t *out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16_bits(in[i]);
}

/* IEEE 754 binary16 -> double, exact. */
double oracle_f16_bits_to_f64(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);
    return s ? -v : v;
}

/* bfloat16 -> double, exact: the bf16 bits are the top half of a binary32. */
double oracle_bf16_bits_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* --------------------------------------------------------------- quantizer */

static float oracle_round_half_away(float r) {
#if ORACLE_MUTANT == 2
    return nearbyintf(r);                /* mutant: ties to even */
#else
    return roundf(r);
#endif
}

/* One block: 32 fp32 weights -> 18 bytes. */
static void oracle_quantize_block(const float *w, uint8_t *out) {
    int imax = 0;
    float amax = fabsf(w[0]);
    for (int j = 1; j < ORACLE_QK; ++j) {
#if ORACLE_MUTANT == 4
        if (fabsf(w[j]) >= amax) { amax = fabsf(w[j]); imax = j; } /* mutant: last index wins */
#else
        if (fabsf(w[j]) > amax) { amax = fabsf(w[j]); imax = j; }
#endif
    }
    uint8_t q[ORACLE_QK];
    uint16_t dbits;
    if (amax == 0.0f) {
        dbits = 0;
        for (int j = 0; j < ORACLE_QK; ++j) q[j] = 8;
    } else {
#if ORACLE_MUTANT == 3
        float d = w[imax] / 8.0f;        /* mutant: wrong sign of d */
#else
        float d = w[imax] / -8.0f;
#endif
        dbits = oracle_f32_to_f16_bits(d);
#if ORACLE_MUTANT == 7
        d = (float)oracle_f16_bits_to_f64(dbits); /* mutant: divide by the stored fp16 d */
#endif
        for (int j = 0; j < ORACLE_QK; ++j) {
            float r = w[j] / d;
            int c = (int)oracle_round_half_away(r) + 8;
            if (c < 0) c = 0;
#if ORACLE_MUTANT == 11
            if (c > 14) c = 14; /* mutant: codes clamped one short of 15 */
#else
            if (c > 15) c = 15;
#endif
            q[j] = (uint8_t)c;
        }
    }
#if ORACLE_MUTANT == 10
    out[0] = (uint8_t)(dbits >> 8); /* mutant: scale bytes swapped */
    out[1] = (uint8_t)(dbits & 0xFFu);
#else
    out[0] = (uint8_t)(dbits & 0xFFu);
    out[1] = (uint8_t)(dbits >> 8);
#endif
    for (int j = 0; j < 16; ++j) {
#if ORACLE_MUTANT == 1
        out[2 + j] = (uint8_t)((q[j] << 4) | q[j + 16]); /* mutant: nibbles swapped */
#else
        out[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
#endif
    }
}

/* w: fp32 [N][K] row-major; wq: N * (K/32) blocks of 18 bytes, row-major. */
void oracle_quantize(const float *w, uint8_t *wq, int64_t N, int64_t K) {
    int64_t nb = K / ORACLE_QK;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            oracle_quantize_block(w + n * K + b * ORACLE_QK,
                                  wq + (n * nb + b) * ORACLE_BLOCK_BYTES);
}

/* -------------------------------------------------------- unpack / decode */

/* codes: uint8 [N][K] (q in 0..15), dbits: uint16 [N][K/32]. */
void oracle_unpack(const uint8_t *wq, uint8_t *codes, uint16_t *dbits, int64_t N, int64_t K) {
    int64_t nb = K / ORACLE_QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = wq + (n * nb + b) * ORACLE_BLOCK_BYTES;
            dbits[n * nb + b] = ORACLE_D_BITS(blk);
            uint8_t *c = codes + n * K + b * ORACLE_QK;
            for (int j = 0; j < 16; ++j) {
#if ORACLE_MUTANT == 1
                c[j] = blk[2 + j] >> 4;
                c[j + 16] = blk[2 + j] & 15;
#else
                c[j] = blk[2 + j] & 15;
                c[j + 16] = blk[2 + j] >> 4;
#endif
            }
        }
}

/* Row n of W, decoded exactly into fp64: w = d * (q - 8). */
static void oracle_decode_row(const uint8_t *wq, int64_t n, int64_t K, double *row) {
    int64_t nb = K / ORACLE_QK;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = wq + (n * nb + b) * ORACLE_BLOCK_BYTES;
        double d = oracle_f16_bits_to_f64(ORACLE_D_BITS(blk));
        for (int j = 0; j < 16; ++j) {
#if ORACLE_MUTANT == 1
            int lo = blk[2 + j] >> 4, hi = blk[2 + j] & 15;
#else
            int lo = blk[2 + j] & 15, hi = blk[2 + j] >> 4;
#endif
#if ORACLE_MUTANT == 5
            row[b * ORACLE_QK + j] = d * lo;            /* mutant: offset 8 dropped */
            row[b * ORACLE_QK + j + 16] = d * hi;
#else
            row[b * ORACLE_QK + j] = d * (lo - 8);
            row[b * ORACLE_QK + j + 16] = d * (hi - 8);
#endif
        }
    }
}

void oracle_dequantize(const uint8_t *wq, double *w, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) oracle_decode_row(wq, n, K, w + n * K);
}

/* ------------------------------------------------------------------ matmul */

/* y[m][n] = sum_k w[n][k] * x[m][k] (fp64, k ascending); optional
 * abssum[m][n] = sum_k |w[n][k] * x[m][k]|, the scale of the per-element
 * tolerance.  x: bf16 bits [M][K]; y, abssum: [M][N]. */
void oracle_matmul(const uint16_t *x, const uint8_t *wq, double *y, double *abssum,
                   int64_t M, int64_t N, int64_t K) {
#pragma omp parallel
    {
        double *row = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t n = 0; n < N; ++n) {
            oracle_decode_row(wq, n, K, row);
            for (int64_t m = 0; m < M; ++m) {
                const uint16_t *xr = x + m * K;
                double s = 0.0, a = 0.0;
#if ORACLE_MUTANT == 9
                for (int64_t k = 0; k + 1 < K; ++k) {   /* mutant: last term dropped */
#else
                for (int64_t k = 0; k < K; ++k) {
#endif
#if ORACLE_MUTANT == 6
                    double p = row[k] * oracle_bf16_bits_to_f64(x[(k % M) * K + (k / M) + m * 0]);
                    (void)xr;                             /* mutant: x indexed transposed */
#else
                    double p = row[k] * oracle_bf16_bits_to_f64(xr[k]);
#endif
                    s += p;
                    a += fabs(p);
                }
                y[m * N + n] = s;
                if (abssum) abssum[m * N + n] = a;
            }
        }
        free(row);
    }
}

/* The same definition evaluated only at the listed (m, n) pairs. */
void oracle_matmul_sampled(const uint16_t *x, const uint8_t *wq, int64_t M, int64_t N, int64_t K,
                           const int64_t *ms, const int64_t *ns, int64_t count,
                           double *y, double *abssum) {
    (void)N;
#pragma omp parallel
    {
        double *row = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < count; ++i) {
            oracle_decode_row(wq, ns[i], K, row);
            const uint16_t *xr = x + ms[i] * K;
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = row[k] * oracle_bf16_bits_to_f64(xr[k]);
                s += p;
                a += fabs(p);
            }
            (void)M;
            y[i] = s;
            if (abssum) abssum[i] = a;
        }
        free(row);
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_mutant(void) { return ORACLE_MUTANT; }
