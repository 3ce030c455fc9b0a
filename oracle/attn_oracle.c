/*
 * attn_oracle.c -- CPU oracle for the decoder's single-head attention block
 * with its output projection (the operation whose V projection the fast
 * path folds the output projection into).
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite and the
 * benchmark's CPU-baseline leg load this library.  The CUDA library never
 * links, includes or calls it, and this file shares no header, helper or
 * constant with it.
 *
 * What it computes (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
 * quality=high", section "Modifications", item 2, the attention bullet): the
 * VAE mid-block attention after its GroupNorm and its query / key
 * projections, single head of width D, as defined -- NOT folded:
 *
 *   v[j][c]   = bv[c] + sum_i xn[j][i] * wv[c][i]                 (value projection)
 *   s[r][j]   = (1 / sqrt(D)) * sum_d q[r][d] * k[j][d]
 *   a[r][j]   = exp(s[r][j] - max_j s[r][.]) / sum_j exp(s[r][j] - max_j s[r][.])
 *   o[r][c]   = sum_j a[r][j] * v[j][c]
 *   out[r][e] = bo[e] + sum_c o[r][c] * wo[e][c] + residual[r][e]  (output projection,
 *                                                                    residual optional)
 *
 * The page's fold (W' = wo wv, b' = wo bv + bo, out = a (xn W'^T + b') +
 * residual, exact because every row of a sums to 1) is NOT used here; the
 * tests check it against this definition.
 *
 * Alongside out it can return mag[r][e] = |bo[e]| + |residual[r][e]| +
 * sum_c |wo[e][c]| * sum_j a[r][j] * (|bv[c]| + sum_i |xn[j][i] * wv[c][i]|),
 * the magnitude against which the rounding of any evaluation order is
 * bounded.  Inputs are bf16 bit patterns decoded exactly; everything is
 * fp64 (built with -ffp-contract=off).  Linear weights use PyTorch's layout
 * [out][in].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ATT_OK = 0, ATT_BAD_ARG = 1, ATT_NO_MEM = 2 };

static double bf(uint16_t h)
{
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

typedef struct {
    int64_t S, D;
    const uint16_t *q, *k, *res;
    double *v;      /* [S][D] value projection */
    double *va;     /* [S][D] |bv| + sum |xn * wv| */
    double *wo;     /* [D][D] decoded */
    double *bo;     /* [D] */
} Att;

static void att_free(Att *t)
{
    free(t->v);
    free(t->va);
    free(t->wo);
    free(t->bo);
}

static int att_setup(Att *t, const uint16_t *q, const uint16_t *k, const uint16_t *xn, const uint16_t *wv,
                     const uint16_t *bv, const uint16_t *wo, const uint16_t *bo, const uint16_t *res, int64_t S,
                     int64_t D)
{
    memset(t, 0, sizeof *t);
    if (!q || !k || !xn || !wv || !bv || !wo || !bo || S <= 0 || D <= 0) return ATT_BAD_ARG;
    t->S = S;
    t->D = D;
    t->q = q;
    t->k = k;
    t->res = res;
    t->v = (double *)malloc((size_t)(S * D) * sizeof(double));
    t->va = (double *)malloc((size_t)(S * D) * sizeof(double));
    t->wo = (double *)malloc((size_t)(D * D) * sizeof(double));
    t->bo = (double *)malloc((size_t)D * sizeof(double));
    double *wvd = (double *)malloc((size_t)(D * D) * sizeof(double));
    if (!t->v || !t->va || !t->wo || !t->bo || !wvd) {
        free(wvd);
        att_free(t);
        return ATT_NO_MEM;
    }
    for (int64_t i = 0; i < D * D; ++i) {
        wvd[i] = bf(wv[i]);
        t->wo[i] = bf(wo[i]);
    }
    for (int64_t c = 0; c < D; ++c) t->bo[c] = bf(bo[c]);
    int64_t j;
#pragma omp parallel for schedule(static)
    for (j = 0; j < S; ++j) {
        for (int64_t c = 0; c < D; ++c) {
            double acc = bf(bv[c]), mag = fabs(bf(bv[c]));
            for (int64_t i = 0; i < D; ++i) {
                const double p = bf(xn[j * D + i]) * wvd[c * D + i];
                acc += p;
                mag += fabs(p);
            }
            t->v[j * D + c] = acc;
            t->va[j * D + c] = mag;
        }
    }
    free(wvd);
    return ATT_OK;
}

/* one query row r: out[D] (and mag[D] if not NULL); work holds 2 S + 2 D doubles */
static void att_row(const Att *t, int64_t r, double *out, double *mag, double *work)
{
    const int64_t S = t->S, D = t->D;
    double *a = work, *o = work + S, *oa = work + S + D;
    const double scale = 1.0 / sqrt((double)D);
    double mx = -INFINITY;
    for (int64_t j = 0; j < S; ++j) {
        double s = 0.0;
        for (int64_t d = 0; d < D; ++d) s += bf(t->q[r * D + d]) * bf(t->k[j * D + d]);
        a[j] = scale * s;
        if (a[j] > mx) mx = a[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < S; ++j) {
        a[j] = exp(a[j] - mx);
        l += a[j];
    }
    for (int64_t j = 0; j < S; ++j) a[j] /= l;
    for (int64_t c = 0; c < D; ++c) {
        double acc = 0.0, am = 0.0;
        for (int64_t j = 0; j < S; ++j) {
            acc += a[j] * t->v[j * D + c];
            am += a[j] * t->va[j * D + c];
        }
        o[c] = acc;
        oa[c] = am;
    }
    for (int64_t e = 0; e < D; ++e) {
        const double rv = t->res ? bf(t->res[r * D + e]) : 0.0;
        double acc = t->bo[e], m = fabs(t->bo[e]) + fabs(rv);
        for (int64_t c = 0; c < D; ++c) {
            acc += o[c] * t->wo[e * D + c];
            m += oa[c] * fabs(t->wo[e * D + c]);
        }
        out[e] = acc + rv;
        if (mag) mag[e] = m;
    }
}

/* out (and mag) for the query rows listed in rows[count] (all rows if rows
 * is NULL and count == S), [count][D] */
int attn_oracle_rows(const uint16_t *q, const uint16_t *k, const uint16_t *xn, const uint16_t *wv,
                     const uint16_t *bv, const uint16_t *wo, const uint16_t *bo, const uint16_t *residual,
                     int64_t S, int64_t D, const int64_t *rows, int64_t count, double *out, double *mag)
{
    if (!out || count < 0 || (!rows && count != S)) return ATT_BAD_ARG;
    if (rows) {
        for (int64_t i = 0; i < count; ++i)
            if (rows[i] < 0 || rows[i] >= S) return ATT_BAD_ARG;
    }
    Att t;
    int rc = att_setup(&t, q, k, xn, wv, bv, wo, bo, residual, S, D);
    if (rc) return rc;
    int bad = 0;
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (i = 0; i < count; ++i) {
        double *work = (double *)malloc((size_t)(2 * S + 2 * D) * sizeof(double));
        if (!work) {
            bad |= 1;
            continue;
        }
        att_row(&t, rows ? rows[i] : i, out + i * D, mag ? mag + i * D : NULL, work);
        free(work);
    }
    att_free(&t);
    return bad ? ATT_NO_MEM : ATT_OK;
}

/* out (and mag) over all S query rows, [S][D] */
int attn_oracle_forward(const uint16_t *q, const uint16_t *k, const uint16_t *xn, const uint16_t *wv,
                        const uint16_t *bv, const uint16_t *wo, const uint16_t *bo, const uint16_t *residual,
                        int64_t S, int64_t D, double *out, double *mag)
{
    if (!out) return ATT_BAD_ARG;
    return attn_oracle_rows(q, k, xn, wv, bv, wo, bo, residual, S, D, NULL, S, out, mag);
}
