/*
 * arf_oracle.c: plain, single-threaded CPU oracle for the all-reduce fusion
 * epilogue (patterns kAllReduce and kARResidualRMSNorm).
 *
 * TEST INFRASTRUCTURE, not part of the library. The test suite, the package's
 * smoke check and the benchmark's CPU-baseline leg are the only callers. It
 * shares no code, header, table, constant or helper with the CUDA library.
 *
 * What it computes. The pattern names come from tokenspeed PR #1075 "route
 * generic MNNVL AR patterns to upstream flashinfer" (description and Summary):
 * kAllReduce is the cross-rank elementwise sum of the W per-rank partials;
 * kARResidualRMSNorm is that sum followed by a residual add and an RMSNorm.
 * fp16 alongside bf16 follows flashinfer PR #1321 "Optimizations for TRTLLM
 * MNNVL Allreduce" (Highlights, __nv_half support). The numeric contract the
 * library states, and this file writes out:
 *   acc   = 0.0f; for r = 0..W-1: acc = acc + f32(P_r[m,i])   (binary32, RN,
 *           rank order as given, no reassociation)
 *   AR:   out[m,i]          = rn(acc)
 *   RMS:  residual_out[m,i] = rn(acc + f32(R[m,i]))           (one rounding)
 *         x_i = f32(residual_out[m,i])                         (stored value)
 *         inv = 1 / sqrt(sum_i x_i^2 / H + eps)                (binary64)
 *         out[m,i] = rn(x_i * inv * gamma_i)                   (binary64, one
 *                                                               final rounding)
 * rn() is round-to-nearest-even to the I/O type, written below from the
 * IEEE-754 definition of the binary16 and bfloat16 formats.
 *
 * Build: any C99 compiler, with -ffp-contract=off and without fast-math, so
 * that every binary32 add is a separate IEEE round-to-nearest operation.
 */
#include "arf_oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* 16-bit formats, from their IEEE-754-style definitions.                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    int p;         /* significand precision, implicit bit included           */
    int emin;      /* exponent of the smallest normal binade                 */
    int emax;      /* exponent of the largest finite binade                  */
    int bias;      /* exponent field bias                                    */
    unsigned qnan; /* default quiet NaN, sign bit clear                      */
} fmt16_t;

/* bfloat16: 1 sign, 8 exponent, 7 fraction bits (binary32's upper half). */
static const fmt16_t FMT_BF16 = {8, -126, 127, 127, 0x7fc0u};
/* binary16: 1 sign, 5 exponent, 10 fraction bits. */
static const fmt16_t FMT_F16 = {11, -14, 15, 15, 0x7e00u};

static const fmt16_t* fmt_of(int dtype) { return dtype == 0 ? &FMT_BF16 : &FMT_F16; }

/* Round v to the nearest value of format f, ties to the even significand,
 * and return its encoding. The value is written as K * 2^(E - (p-1)) with
 * E its binade exponent clamped below at emin (subnormals share the smallest
 * quantum); K = v / quantum is exact in binary64, and rounding K to an
 * integer is exactly rounding v to the format's grid. */
static unsigned encode16(double v, const fmt16_t* f)
{
    const int mbits = f->p - 1;
    const int ebits = 15 - mbits;
    const unsigned sign = signbit(v) ? 0x8000u : 0u;
    const unsigned inf = ((1u << ebits) - 1u) << mbits;

    if (isnan(v)) return sign | f->qnan;
    double a = fabs(v);
    if (isinf(a)) return sign | inf;
    if (a == 0.0) return sign;

    int e2;
    (void)frexp(a, &e2); /* a = m * 2^e2 with m in [0.5, 1) */
    int E = e2 - 1;      /* binade: a in [2^E, 2^(E+1)) */
    if (E < f->emin) E = f->emin;

    double k = ldexp(a, mbits - E); /* a / 2^(E - mbits): exact */
    double kf = floor(k);
    double rem = k - kf; /* exact */
    if (rem > 0.5 || (rem == 0.5 && fmod(kf, 2.0) != 0.0)) kf += 1.0;
    if (kf >= ldexp(1.0, f->p)) { /* rounded up into the next binade */
        kf = ldexp(1.0, mbits);
        E += 1;
    }
    if (E > f->emax) return sign | inf; /* overflow */

    unsigned K = (unsigned)kf;
    if (K < (1u << mbits)) return sign | K; /* subnormal: exponent field 0 */
    return sign | ((unsigned)(E + f->bias) << mbits) | (K - (1u << mbits));
}

static float decode_bf16(unsigned h)
{
    /* bfloat16 is the upper half of a binary32 encoding. */
    unsigned u = h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float decode_f16(unsigned h)
{
    unsigned ex = (h >> 10) & 0x1fu, man = h & 0x3ffu;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24); /* subnormal: man * 2^(emin - 10) */
    else if (ex == 31)
        v = man ? (double)NAN : (double)INFINITY;
    else
        v = ldexp((double)(man | 0x400u), (int)ex - 25); /* 1.man * 2^(ex-15) */
    return (float)((h & 0x8000u) ? -v : v);
}

float arf_oracle_widen(int dtype, uint16_t bits)
{
    return dtype == 0 ? decode_bf16(bits) : decode_f16(bits);
}

uint16_t arf_oracle_narrow_f32(int dtype, float v)
{
    return (uint16_t)encode16((double)v, fmt_of(dtype)); /* exact widening first */
}

uint16_t arf_oracle_narrow_f64(int dtype, double v)
{
    return (uint16_t)encode16(v, fmt_of(dtype));
}

void arf_oracle_widen_n(int dtype, const uint16_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = arf_oracle_widen(dtype, in[i]);
}

void arf_oracle_narrow_f32_n(int dtype, const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = arf_oracle_narrow_f32(dtype, in[i]);
}

void arf_oracle_narrow_f64_n(int dtype, const double* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = arf_oracle_narrow_f64(dtype, in[i]);
}

/* ------------------------------------------------------------------------ */
/* The epilogue.                                                             */
/* ------------------------------------------------------------------------ */

/* RMSNorm statistic of one stored row (the standard root-mean-square norm:
 * mean over all H elements, eps inside the root, added after the mean). */
double arf_oracle_inv_rms(int dtype, const uint16_t* x, int64_t H, float eps,
                          double* ss_out)
{
    double ss = 0.0;
    for (int64_t i = 0; i < H; ++i) {
        double xi = (double)arf_oracle_widen(dtype, x[i]);
        ss += xi * xi; /* sequential i = 0..H-1 */
    }
    if (ss_out) *ss_out = ss;
    return 1.0 / sqrt(ss / (double)H + (double)eps);
}

/* Value of partial element i of rank r: 16-bit codes of the I/O dtype, or
 * binary32 as stored (pdtype 2). */
static float partial_at(const void* p, int pdtype, int dtype, int64_t i)
{
    if (pdtype == 2) return ((const float*)p)[i];
    return arf_oracle_widen(dtype, ((const uint16_t*)p)[i]);
}

int arf_oracle_run_general(int pattern, int W, const void* const* partials, int pdtype, int64_t ld_partials,
                           const void* residual, int64_t ld_residual, const void* gamma, float eps,
                           void* out, int64_t ld_out, void* residual_out, int64_t ld_residual_out,
                           int64_t M, int64_t H, int dtype)
{
    if (pattern != 0 && pattern != 1) return 1;
    if (dtype != 0 && dtype != 1) return 1;
    if (pdtype != dtype && pdtype != 2) return 1;
    if (W < 1 || M < 0 || H < 1) return 1;
    if (ld_partials < H || ld_out < H) return 1;
    if (partials == NULL || out == NULL) return 1;
    for (int r = 0; r < W; ++r)
        if (partials[r] == NULL) return 1;
    if (pattern == 1) {
        if (residual == NULL || gamma == NULL || residual_out == NULL) return 1;
        if (ld_residual < H || ld_residual_out < H) return 1;
    }

    const uint16_t* R = (const uint16_t*)residual;
    const uint16_t* G = (const uint16_t*)gamma;
    uint16_t* O = (uint16_t*)out;
    uint16_t* RO = (uint16_t*)residual_out;

    for (int64_t m = 0; m < M; ++m) {
        const int64_t pb = m * ld_partials, ob = m * ld_out;
        const int64_t rb = m * ld_residual, rob = m * ld_residual_out;

        /* Cross-rank sum, binary32, ranks in the order given. */
        for (int64_t i = 0; i < H; ++i) {
            float acc = 0.0f;
            for (int r = 0; r < W; ++r) acc = acc + partial_at(partials[r], pdtype, dtype, pb + i);
            if (pattern == 0) {
                O[ob + i] = arf_oracle_narrow_f32(dtype, acc);
            } else {
                /* Residual add on the unrounded sum: one rounding in total. */
                float t = acc + arf_oracle_widen(dtype, R[rb + i]);
                RO[rob + i] = arf_oracle_narrow_f32(dtype, t);
            }
        }
        if (pattern == 0) continue;

        /* RMSNorm of the stored residual_out row. */
        double inv = arf_oracle_inv_rms(dtype, RO + rob, H, eps, NULL);
        for (int64_t i = 0; i < H; ++i) {
            double x = (double)arf_oracle_widen(dtype, RO[rob + i]);
            double g = (double)arf_oracle_widen(dtype, G[i]);
            O[ob + i] = arf_oracle_narrow_f64(dtype, x * inv * g);
        }
    }
    return 0;
}

int arf_oracle_run(int pattern, int W, const void* const* partials,
                   const void* residual, const void* gamma, float eps,
                   void* out, void* residual_out, int64_t M, int64_t H,
                   int dtype)
{
    return arf_oracle_run_general(pattern, W, partials, dtype, H, residual, H, gamma, eps, out, H,
                                  residual_out, H, M, H, dtype);
}
