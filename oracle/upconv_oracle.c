/*
 * upconv_oracle.c -- CPU oracle for the fused nearest-2x upsample + 3x3 conv.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite and the
 * benchmark's CPU-baseline leg load this library.  The CUDA library never
 * links, includes or calls it, and this file shares no header, helper or
 * constant with it.
 *
 * What it computes (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
 * quality=high", section "Modifications", item 2, the fused-upsample bullet):
 * the decoder's up-sampling step, a nearest-neighbour 2x upsample followed by
 * a 3x3 convolution with padding 1 (the page notes that this equals a
 * transposed convolution with kernel 4, stride 2, padding 1 whose taps are
 * sums of the 3x3 taps; this file does NOT use that identity, it writes out
 * the two steps as defined, and the tests check the identity separately).
 *
 * Layouts: x is channels-last [N][H][W][Cin] bf16, the weight is the
 * convolution's own [Cout][Cin][3][3] bf16, the optional bias [Cout] bf16.
 * The output is [N][2H][2W][Cout], returned unrounded in fp64:
 *
 *   u[n][p][q][ci] = x[n][p/2][q/2][ci]   for 0 <= p < 2H, 0 <= q < 2W
 *                  = 0                    otherwise (the conv's zero padding)
 *   y[n][P][Q][co] = bias[co] + sum_{ky,kx in 0..2} sum_ci
 *                        u[n][P+ky-1][Q+kx-1][ci] * w[co][ci][ky][kx]
 *
 * Alongside y it can return a[n][P][Q][co] = sum |u * w| over the same terms:
 * the scale against which rounding errors of any evaluation order are
 * bounded.  Every bf16 value is decoded exactly; products and sums are fp64
 * (built with -ffp-contract=off, so nothing is fused).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { UPC_OK = 0, UPC_BAD_ARG = 1, UPC_NO_MEM = 2 };

static double bf16_value(uint16_t h)
{
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

typedef struct {
    int64_t N, H, W, Cin, Cout;
    const uint16_t *x, *bias;
    double *wd;   /* the weight decoded to fp64, same [Cout][Cin][3][3] order */
} Problem;

/* the upsampled input u at (n, p, q, ci), zero outside the 2H x 2W image */
static double upsampled(const Problem *pr, int64_t n, int64_t p, int64_t q, int64_t ci)
{
    if (p < 0 || q < 0 || p >= 2 * pr->H || q >= 2 * pr->W) return 0.0;
    const int64_t i = p / 2, j = q / 2;
    return bf16_value(pr->x[((n * pr->H + i) * pr->W + j) * pr->Cin + ci]);
}

/* one output element y[n][P][Q][co] and its absolute-term sum */
static void one_output(const Problem *pr, int64_t n, int64_t P, int64_t Q, int64_t co,
                       double *y, double *a)
{
    double s = pr->bias ? bf16_value(pr->bias[co]) : 0.0;
    double t = fabs(s);
    for (int ky = 0; ky < 3; ++ky) {
        for (int kx = 0; kx < 3; ++kx) {
            for (int64_t ci = 0; ci < pr->Cin; ++ci) {
                const double u = upsampled(pr, n, P + ky - 1, Q + kx - 1, ci);
                const double w = pr->wd[((co * pr->Cin + ci) * 3 + ky) * 3 + kx];
                s += u * w;
                t += fabs(u * w);
            }
        }
    }
    *y = s;
    if (a) *a = t;
}

static int setup(Problem *pr, const uint16_t *x, const uint16_t *w, const uint16_t *bias,
                 int64_t N, int64_t H, int64_t W, int64_t Cin, int64_t Cout)
{
    if (!x || !w || N < 0 || H <= 0 || W <= 0 || Cin <= 0 || Cout <= 0) return UPC_BAD_ARG;
    pr->N = N; pr->H = H; pr->W = W; pr->Cin = Cin; pr->Cout = Cout;
    pr->x = x; pr->bias = bias;
    const int64_t nw = Cout * Cin * 9;
    pr->wd = (double *)malloc((size_t)nw * sizeof(double));
    if (!pr->wd) return UPC_NO_MEM;
    for (int64_t k = 0; k < nw; ++k) pr->wd[k] = bf16_value(w[k]);
    return UPC_OK;
}

/* y (and a, if not NULL) over the whole [N][2H][2W][Cout] output */
int upconv_oracle_forward(const uint16_t *x, const uint16_t *w, const uint16_t *bias,
                          int64_t N, int64_t H, int64_t W, int64_t Cin, int64_t Cout,
                          double *y, double *a)
{
    if (!y) return UPC_BAD_ARG;
    Problem pr;
    int rc = setup(&pr, x, w, bias, N, H, W, Cin, Cout);
    if (rc) return rc;
    const int64_t OH = 2 * H, OW = 2 * W;
    int64_t pix;
#pragma omp parallel for schedule(dynamic, 16)
    for (pix = 0; pix < N * OH * OW; ++pix) {
        const int64_t n = pix / (OH * OW), P = (pix / OW) % OH, Q = pix % OW;
        for (int64_t co = 0; co < Cout; ++co) {
            const int64_t at = pix * Cout + co;
            one_output(&pr, n, P, Q, co, &y[at], a ? &a[at] : NULL);
        }
    }
    free(pr.wd);
    return UPC_OK;
}

/* The same at selected flat indices of the [N][2H][2W][Cout] output. */
int upconv_oracle_at(const uint16_t *x, const uint16_t *w, const uint16_t *bias,
                     int64_t N, int64_t H, int64_t W, int64_t Cin, int64_t Cout,
                     const int64_t *index, int64_t count, double *y, double *a)
{
    if (!index || !y || count < 0) return UPC_BAD_ARG;
    Problem pr;
    int rc = setup(&pr, x, w, bias, N, H, W, Cin, Cout);
    if (rc) return rc;
    const int64_t OH = 2 * H, OW = 2 * W, total = N * OH * OW * Cout;
    int bad = 0;
    int64_t k;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (k = 0; k < count; ++k) {
        const int64_t at = index[k];
        if (at < 0 || at >= total) {
            bad |= 1;
            y[k] = 0.0;
            if (a) a[k] = 0.0;
            continue;
        }
        const int64_t co = at % Cout, pix = at / Cout;
        const int64_t n = pix / (OH * OW), P = (pix / OW) % OH, Q = pix % OW;
        one_output(&pr, n, P, Q, co, &y[k], a ? &a[k] : NULL);
    }
    free(pr.wd);
    return bad ? UPC_BAD_ARG : UPC_OK;
}
