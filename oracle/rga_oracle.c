/*
 * rga_oracle.c -- CPU oracle for the residual-gate update  y = residual + gate * update.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite and the
 * benchmark's CPU-baseline leg load this library.  The CUDA library never
 * links, includes or calls it, and this file shares no header, helper or
 * constant with it.
 *
 * What it computes (the prhub digest of sglang PR #33823, FLUX.2 bit-exact
 * residual-gate fusion, sections "Functions and motivation" and
 * "Implementation breakdown", items 1-3): the
 * transformer's residual stream update `residual + gate * update` with
 * residual and update of shape [rows, D] and gate one broadcast row [D], in
 * half precision (bf16 or fp16), bit for bit equal to the eager two-kernel
 * evaluation: first the product gate * update as its own half-precision
 * tensor, then the sum with the residual.  Each eager kernel works in fp32
 * and rounds its result to the half format once (round to nearest, ties to
 * even), so per element:
 *
 *   p = half( f32(gate[d]) * f32(update[r, d]) )      (the fp32 product of
 *                                                       two half values is
 *                                                       exact)
 *   y = half( f32( f32(residual[r, d]) + f32(p) ) )    (fp32 sum, rounded to
 *                                                       fp32, then to half)
 *
 * Reading where the pages are silent: the "eager" semantics are those of
 * PyTorch's elementwise kernels for half dtypes (fp32 arithmetic, one
 * rounding to the storage format per kernel); NaN results are quiet NaNs
 * (any NaN payload counts as the same value).
 *
 * (The intermediate fp32 rounding of the sum never changes the final half
 * value: the two operands carry 8 (bf16) or 11 (fp16) significant bits, so
 * the exact sum needs more than 24 bits only when the smaller operand lies
 * far below the half format's rounding midpoints.  It is kept because it is
 * what the eager kernel does.)
 *
 * Here every value is decoded exactly to fp64, the product is formed in
 * fp64 (exact), and the two roundings are written out from their
 * definitions: to binary32 by the C cast (round to nearest even), to bf16 /
 * fp16 by the bit-level routines below.  Nothing is fused (built with
 * -ffp-contract=off).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { RGA_OK = 0, RGA_BAD_ARG = 1 };
enum { FMT_BF16 = 0, FMT_F16 = 1 };

/* ---- exact decodes ------------------------------------------------------- */
static double bf16_decode(uint16_t h)
{
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double f16_decode(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int ex = (h >> 10) & 0x1f;
    const int man = h & 0x3ff;
    double v;
    if (ex == 0x1f) {
        v = man ? NAN : INFINITY;
    } else if (ex == 0) {
        v = ldexp((double)man, -24);              /* subnormal: man * 2^-24 */
    } else {
        v = ldexp((double)(man | 0x400), ex - 25); /* (1.man) * 2^(ex-15) */
    }
    return sign ? -v : v;
}

/* ---- roundings to the half formats (round to nearest, ties to even) ------ */
/* A binary32 value (given exactly) to bf16 bits. */
static uint16_t f32_to_bf16(float f)
{
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    if ((w & 0x7f800000u) == 0x7f800000u && (w & 0x007fffffu)) return 0x7fc0; /* NaN */
    const uint32_t lsb = (w >> 16) & 1u;
    w += 0x7fffu + lsb;                          /* carries into the exponent as needed */
    return (uint16_t)(w >> 16);
}

/* A binary32 value (given exactly) to fp16 bits. */
static uint16_t f32_to_f16(float f)
{
    if (isnan(f)) return 0x7e00;
    const uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (isinf(a)) return sign | 0x7c00;
    /* the fp16 spacing at |a|: 2^(e-10) for normals (e >= -14), 2^-24 below */
    int e;
    frexp(a, &e);                                /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 1 - 10;                          /* exponent of one ulp */
    if (q < -24) q = -24;
    const double ulp = ldexp(1.0, q);
    double n = a / ulp;                          /* exact: a power-of-two scaling */
    double fl = floor(n);
    double rem = n - fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    const double r = fl * ulp;                   /* the rounded magnitude */
    if (r >= 65536.0) return sign | 0x7c00;      /* overflow to infinity */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -14)) return sign | (uint16_t)(r / ldexp(1.0, -24));   /* subnormal */
    int re;
    const double rm = frexp(r, &re);             /* r = rm * 2^re, rm in [0.5, 1) */
    const uint16_t exf = (uint16_t)(re - 1 + 15);
    const uint16_t man = (uint16_t)((rm * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)(exf << 10) | man;
}

static double decode(uint16_t h, int fmt) { return fmt == FMT_BF16 ? bf16_decode(h) : f16_decode(h); }

static uint16_t round_half(float f, int fmt) { return fmt == FMT_BF16 ? f32_to_bf16(f) : f32_to_f16(f); }

/* One output element from its three inputs (raw half bit patterns). */
static uint16_t residual_gate_one(uint16_t res, uint16_t upd, uint16_t gat, int fmt)
{
    const double prod = decode(gat, fmt) * decode(upd, fmt);   /* exact in fp64 */
    const uint16_t p = round_half((float)prod, fmt);            /* (float) is exact here */
    const double sum = decode(res, fmt) + decode(p, fmt);
    return round_half((float)sum, fmt);                         /* to fp32, then to half */
}

/* out[r, d] for a [rows, D] residual and update and a [D] gate. */
int rga_oracle_forward(const uint16_t *residual, const uint16_t *update, const uint16_t *gate,
                       uint16_t *out, int64_t rows, int64_t D, int fmt)
{
    if (!residual || !update || !gate || !out) return RGA_BAD_ARG;
    if (rows < 0 || D <= 0 || (fmt != FMT_BF16 && fmt != FMT_F16)) return RGA_BAD_ARG;
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        for (int64_t d = 0; d < D; ++d) {
            const int64_t at = r * D + d;
            out[at] = residual_gate_one(residual[at], update[at], gate[d], fmt);
        }
    }
    return RGA_OK;
}

/* The same at selected flat indices of the [rows, D] tensors. */
int rga_oracle_at(const uint16_t *residual, const uint16_t *update, const uint16_t *gate,
                  int64_t rows, int64_t D, int fmt, const int64_t *index, int64_t count, uint16_t *out)
{
    if (!residual || !update || !gate || !index || !out) return RGA_BAD_ARG;
    if (rows < 0 || D <= 0 || count < 0 || (fmt != FMT_BF16 && fmt != FMT_F16)) return RGA_BAD_ARG;
    int bad = 0;
    int64_t k;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (k = 0; k < count; ++k) {
        const int64_t at = index[k];
        if (at < 0 || at >= rows * D) { bad |= 1; out[k] = 0; continue; }
        out[k] = residual_gate_one(residual[at], update[at], gate[at % D], fmt);
    }
    return bad ? RGA_BAD_ARG : RGA_OK;
}
