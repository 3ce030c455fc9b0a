/*
 * gn_oracle.c -- fp64 CPU oracle for channels-last GroupNorm followed by SiLU.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference arm load this library.
 * The CUDA library never links, includes or calls it, and this file shares
 * no header, helper or constant with it.
 *
 * What it computes (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
 * quality=high", section "Modifications", item 1): GroupNorm over (N, L, C)
 * rows with C innermost (a channels_last 4D tensor seen through a permute
 * view), with per-(batch, group) statistics, the per-channel affine, and an
 * optional SiLU applied after it (the "GroupNorm -> SiLU" chain named in the
 * "Motivation" section).  The method itself reaches this result through
 * re-associations (partial sums, scale/shift folding); the oracle instead
 * writes out the plain definition:
 *
 *   for each n and each group g, S = { x[n,l,c] : 0 <= l < L,
 *                                      g*Cg <= c < (g+1)*Cg },  m = L*Cg
 *   mean = (1/m) * sum_S x                        (first pass, fp64)
 *   var  = (1/m) * sum_S (x - mean)^2             (second pass, fp64; biased)
 *   rstd = 1 / sqrt(var + eps)
 *   z    = (x - mean) * rstd * gamma[c] + beta[c]
 *   y    = z / (1 + exp(-z))   if SiLU is on,  else  y = z
 *
 * Readings where the pages are silent: biased variance (GroupNorm's own
 * definition, which the pages' "mathematically exact re-associations" keep),
 * eps inside the square root, affine before SiLU, SiLU = z * sigmoid(z).
 *
 * Everything is fp64; x arrives as raw bf16 bit patterns and is decoded
 * here exactly (a bf16 value is the upper 16 bits of an IEEE binary32).
 * Sums run in a fixed order inside each (n, g), so results do not depend on
 * the number of OpenMP threads.  Nothing is rounded to bf16 or fp32 on the
 * way out.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1 };

/* Exact decode of one bf16 bit pattern: widen to binary32 by appending 16
 * zero bits, then to binary64 (both widenings are exact). */
static double bf16_to_f64(uint16_t bits)
{
    uint32_t wide = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &wide, sizeof f);
    return (double)f;
}

static int check_geometry(int64_t N, int64_t L, int64_t C, int64_t G)
{
    if (N <= 0 || L <= 0 || C <= 0 || G <= 0) return ORACLE_BAD_ARG;
    if (C % G != 0) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads OpenMP will use for the next parallel region. */
int gn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Per-(n, g) mean, biased variance and rstd, each [N*G] fp64 (var may be
 * NULL).  Two passes over the group's elements, in row order then channel
 * order. */
int gn_oracle_stats(const uint16_t *x, int64_t N, int64_t L, int64_t C, int64_t G,
                    double eps, double *mean, double *var, double *rstd, int nthreads)
{
    if (!x || !mean || !rstd) return ORACLE_BAD_ARG;
    if (check_geometry(N, L, C, G) != ORACLE_OK) return ORACLE_BAD_ARG;
    const int64_t Cg = C / G;
    const double m = (double)L * (double)Cg;
    set_threads(nthreads);

    int64_t task;
#pragma omp parallel for schedule(dynamic, 1)
    for (task = 0; task < N * G; ++task) {
        const int64_t n = task / G;
        const int64_t g = task % G;
        const uint16_t *xn = x + n * L * C;

        double sum = 0.0;
        for (int64_t l = 0; l < L; ++l)
            for (int64_t c = g * Cg; c < (g + 1) * Cg; ++c)
                sum += bf16_to_f64(xn[l * C + c]);
        const double mu = sum / m;

        double sq = 0.0;
        for (int64_t l = 0; l < L; ++l)
            for (int64_t c = g * Cg; c < (g + 1) * Cg; ++c) {
                const double d = bf16_to_f64(xn[l * C + c]) - mu;
                sq += d * d;
            }
        const double v = sq / m;

        mean[task] = mu;
        if (var) var[task] = v;
        rstd[task] = 1.0 / sqrt(v + eps);
    }
    return ORACLE_OK;
}

/* The normalised, affine-transformed value followed by the optional SiLU,
 * for one element whose group statistics are known. */
static double normalize_one(double xv, double mu, double r, double gam, double bet,
                            int apply_silu)
{
    const double z = (xv - mu) * r * gam + bet;
    if (!apply_silu) return z;
    return z / (1.0 + exp(-z));
}

/* Full forward pass: y [N*L*C] fp64 plus mean / rstd [N*G] fp64. */
int gn_oracle_forward(const uint16_t *x, const float *gamma, const float *beta,
                      int64_t N, int64_t L, int64_t C, int64_t G, double eps,
                      int apply_silu, double *y, double *mean, double *rstd, int nthreads)
{
    if (!x || !gamma || !beta || !y || !mean || !rstd) return ORACLE_BAD_ARG;
    int rc = gn_oracle_stats(x, N, L, C, G, eps, mean, NULL, rstd, nthreads);
    if (rc != ORACLE_OK) return rc;
    const int64_t Cg = C / G;

    int64_t row;
#pragma omp parallel for schedule(static)
    for (row = 0; row < N * L; ++row) {
        const int64_t n = row / L;
        for (int64_t c = 0; c < C; ++c) {
            const int64_t g = c / Cg;
            const int64_t at = row * C + c;
            y[at] = normalize_one(bf16_to_f64(x[at]), mean[n * G + g], rstd[n * G + g],
                                  (double)gamma[c], (double)beta[c], apply_silu);
        }
    }
    return ORACLE_OK;
}

/* y at selected flat indices of the [N][L][C] tensor, given the statistics
 * (e.g. from gn_oracle_stats).  Used to check sampled outputs of tensors too
 * large to materialise in fp64. */
int gn_oracle_apply_at(const uint16_t *x, const float *gamma, const float *beta,
                       int64_t N, int64_t L, int64_t C, int64_t G,
                       const double *mean, const double *rstd, int apply_silu,
                       const int64_t *index, int64_t count, double *y, int nthreads)
{
    if (!x || !gamma || !beta || !mean || !rstd || !index || !y) return ORACLE_BAD_ARG;
    if (check_geometry(N, L, C, G) != ORACLE_OK || count < 0) return ORACLE_BAD_ARG;
    const int64_t Cg = C / G;
    const int64_t total = N * L * C;
    int bad = 0;
    set_threads(nthreads);

    int64_t k;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (k = 0; k < count; ++k) {
        const int64_t at = index[k];
        if (at < 0 || at >= total) { bad |= 1; y[k] = NAN; continue; }
        const int64_t n = at / (L * C);
        const int64_t c = at % C;
        const int64_t g = c / Cg;
        y[k] = normalize_one(bf16_to_f64(x[at]), mean[n * G + g], rstd[n * G + g],
                             (double)gamma[c], (double)beta[c], apply_silu);
    }
    return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}
