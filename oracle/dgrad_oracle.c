/*
 * dgrad_oracle.c -- plain fp64 CPU oracle for 2-D convolution backward-data.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg load it (through oracle/__init__.py).  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * What is computed (page "Non-unit stride input backward different input and
 * dispatches between BOO and Fusilli", torch-IR input, op
 * `torch.aten.convolution_backward` with output_mask [true, false, false]):
 * the gradient of a forward cross-correlation with respect to its input,
 *
 *   dx[n, c, hi, wi] = sum over k in group(c), y < Y, x < X, ho < Ho, wo < Wo
 *                      with ho*sh - ph + y*dh == hi and wo*sw - pw + x*dw == wi
 *                      of dy[n, k, ho, wo] * w[k, c mod Cg, y, x]
 *
 * where Ho/Wo are the forward output sizes.  dx is fully overwritten (the
 * same torch-IR ends with `torch.overwrite.tensor.contents`), so every pixel
 * that no tap reaches is exactly zero.
 *
 * Entry points (all arithmetic in double):
 *   oracle_out_dims       forward output size Ho, Wo
 *   oracle_dgrad_scatter  the definition above as a scatter loop, plus the
 *                         per-element magnitude sum  sum |dy*w|  used for
 *                         tolerances; optional image / channel ranges for
 *                         bounded samples
 *   oracle_dgrad_point    the same definition gathered at one dx element
 *   oracle_dgrad_zero_insert  second formulation: zero-insert dy with the
 *                         stride, pad, then correlate with the flipped filter
 *                         (the BOO IR on the same page: `tensor.insert_slice`
 *                         with strides [1,1,2,1], the `1 - x` filter flip and
 *                         the 7-D `linalg.generic` contraction)
 *   oracle_conv_fwd       forward cross-correlation (gather loop), used by the
 *                         adjoint-identity pin <fwd(x,w), dy> = <x, dgrad(dy,w)>
 *
 * Layouts: layout 0 = dy [N][K][Ho][Wo], w [K][Cg][Y][X] (GKCYX with the group
 * index folded into K), dx [N][C][Hi][Wi]; layout 1 = dy [N][Ho][Wo][K],
 * w [K][Y][X][Cg], dx [N][Hi][Wi][C].  Group g owns input channels
 * [g*Cg, (g+1)*Cg) and output channels [g*Kg, (g+1)*Kg).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

typedef struct {
    int64_t N, C, K, Hi, Wi, Y, X;
    int64_t pad_h, pad_w, stride_h, stride_w, dil_h, dil_w, groups;
    int64_t Ho, Wo; /* filled by oracle_out_dims */
} oracle_geom;

/* ---- index helpers (layout-aware element offsets) ---- */
static int64_t dy_off(const oracle_geom *g, int layout, int64_t n, int64_t k, int64_t ho, int64_t wo) {
    if (layout == 0) return ((n * g->K + k) * g->Ho + ho) * g->Wo + wo;
    return ((n * g->Ho + ho) * g->Wo + wo) * g->K + k;
}
static int64_t dx_off(const oracle_geom *g, int layout, int64_t n, int64_t c, int64_t hi, int64_t wi) {
    if (layout == 0) return ((n * g->C + c) * g->Hi + hi) * g->Wi + wi;
    return ((n * g->Hi + hi) * g->Wi + wi) * g->C + c;
}
static int64_t w_off(const oracle_geom *g, int layout, int64_t k, int64_t cg, int64_t y, int64_t x) {
    int64_t Cg = g->C / g->groups;
    if (layout == 0) return ((k * Cg + cg) * g->Y + y) * g->X + x;
    return ((k * g->Y + y) * g->X + x) * Cg + cg;
}

/* Forward output size of a cross-correlation (the dy extent).  Returns 0 on
 * success, -1 for an invalid geometry. */
int oracle_out_dims(oracle_geom *g) {
    if (g->N < 1 || g->C < 1 || g->K < 1 || g->Hi < 1 || g->Wi < 1 || g->Y < 1 || g->X < 1) return -1;
    if (g->stride_h < 1 || g->stride_w < 1 || g->dil_h < 1 || g->dil_w < 1) return -1;
    if (g->pad_h < 0 || g->pad_w < 0 || g->groups < 1) return -1;
    if (g->C % g->groups || g->K % g->groups) return -1;
    int64_t eh = g->Hi + 2 * g->pad_h - g->dil_h * (g->Y - 1) - 1;
    int64_t ew = g->Wi + 2 * g->pad_w - g->dil_w * (g->X - 1) - 1;
    if (eh < 0 || ew < 0) return -1;
    g->Ho = eh / g->stride_h + 1;
    g->Wo = ew / g->stride_w + 1;
    return 0;
}

/* The definition as a scatter loop.  Only images n in [n_begin, n_end) and
 * channels c with c mod Cg in [cg_begin, cg_end) are computed (those dx /
 * absdot entries are zeroed first); the rest of dx is not touched, which is
 * how bounded samples of a large problem are taken.  absdot may be NULL.  Work items are (image, group, channel block):
 * each owns a disjoint slice of dx, so the OpenMP split needs no atomics. */
void oracle_dgrad_scatter(const oracle_geom *g, int layout, const double *dy, const double *w,
                          double *dx, double *absdot, int64_t n_begin, int64_t n_end,
                          int64_t cg_begin, int64_t cg_end) {
    const int64_t G = g->groups, Kg = g->K / G;
    const int64_t CB = 16; /* channel block per work item (the OpenMP grain) */
    const int64_t cspan = cg_end - cg_begin;
    const int64_t ncb = (cspan + CB - 1) / CB;
    const int64_t items = (n_end - n_begin) * G * ncb;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < items; ++it) {
        int64_t n = n_begin + it / (G * ncb);
        int64_t gi = (it / ncb) % G;
        int64_t c0 = cg_begin + (it % ncb) * CB, c1 = c0 + CB < cg_end ? c0 + CB : cg_end;
        const int64_t Cg = g->C / G;
        /* zero this item's slice */
        for (int64_t hi = 0; hi < g->Hi; ++hi)
            for (int64_t wi = 0; wi < g->Wi; ++wi)
                for (int64_t c = c0; c < c1; ++c) {
                    int64_t o = dx_off(g, layout, n, gi * Cg + c, hi, wi);
                    dx[o] = 0.0;
                    if (absdot) absdot[o] = 0.0;
                }
        for (int64_t kk = 0; kk < Kg; ++kk) {
            int64_t k = gi * Kg + kk;
            for (int64_t ho = 0; ho < g->Ho; ++ho)
                for (int64_t wo = 0; wo < g->Wo; ++wo) {
                    double v = dy[dy_off(g, layout, n, k, ho, wo)];
                    for (int64_t y = 0; y < g->Y; ++y) {
                        int64_t hi = ho * g->stride_h - g->pad_h + y * g->dil_h;
                        if (hi < 0 || hi >= g->Hi) continue;
                        for (int64_t x = 0; x < g->X; ++x) {
                            int64_t wi = wo * g->stride_w - g->pad_w + x * g->dil_w;
                            if (wi < 0 || wi >= g->Wi) continue;
                            for (int64_t c = c0; c < c1; ++c) {
                                double p = v * w[w_off(g, layout, k, c, y, x)];
                                int64_t o = dx_off(g, layout, n, gi * Cg + c, hi, wi);
                                dx[o] += p;
                                if (absdot) absdot[o] += fabs(p);
                            }
                        }
                    }
                }
        }
    }
}

/* The definition gathered at one element dx[n, c, hi, wi] (c is the global
 * input channel): every (k, y, x) whose forward window position lands on
 * (hi, wi) contributes, i.e. ho = (hi + ph - y*dh) / sh must be an integer in
 * [0, Ho), likewise wo.  Writes the value and sum |dy*w|. */
void oracle_dgrad_point(const oracle_geom *g, int layout, const double *dy, const double *w,
                        int64_t n, int64_t c, int64_t hi, int64_t wi, double *val, double *absdot) {
    const int64_t G = g->groups, Cg = g->C / G, Kg = g->K / G;
    const int64_t gi = c / Cg, cg = c % Cg;
    double s = 0.0, a = 0.0;
    for (int64_t y = 0; y < g->Y; ++y) {
        int64_t th = hi + g->pad_h - y * g->dil_h;
        if (th < 0 || th % g->stride_h) continue;
        int64_t ho = th / g->stride_h;
        if (ho >= g->Ho) continue;
        for (int64_t x = 0; x < g->X; ++x) {
            int64_t tw = wi + g->pad_w - x * g->dil_w;
            if (tw < 0 || tw % g->stride_w) continue;
            int64_t wo = tw / g->stride_w;
            if (wo >= g->Wo) continue;
            for (int64_t kk = 0; kk < Kg; ++kk) {
                int64_t k = gi * Kg + kk;
                double p = dy[dy_off(g, layout, n, k, ho, wo)] * w[w_off(g, layout, k, cg, y, x)];
                s += p;
                a += fabs(p);
            }
        }
    }
    *val = s;
    if (absdot) *absdot = a;
}

/* Second formulation.  Per spatial dim with stride s, dilation d, pad p and
 * filter length R: place dy[ho] at position ho*s + d*(R-1) - p of a zero
 * buffer of length Hi + d*(R-1) (positions outside are dropped), then
 *   dx[hi] = sum_r dyz[hi + r*d] * w[R-1-r]
 * i.e. a stride-1 correlation of the zero-inserted, padded dy with the
 * flipped filter.  Allocates the buffer; intended for tiny shapes. */
int oracle_dgrad_zero_insert(const oracle_geom *g, int layout, const double *dy, const double *w, double *dx) {
    const int64_t G = g->groups, Cg = g->C / G, Kg = g->K / G;
    const int64_t eh = g->dil_h * (g->Y - 1), ew = g->dil_w * (g->X - 1);
    const int64_t Hz = g->Hi + eh, Wz = g->Wi + ew;
    double *z = (double *)calloc((size_t)(g->N * g->K * Hz * Wz), sizeof(double));
    if (!z) return -1;
    for (int64_t n = 0; n < g->N; ++n)
        for (int64_t k = 0; k < g->K; ++k)
            for (int64_t ho = 0; ho < g->Ho; ++ho) {
                int64_t hz = ho * g->stride_h + eh - g->pad_h;
                if (hz < 0 || hz >= Hz) continue;
                for (int64_t wo = 0; wo < g->Wo; ++wo) {
                    int64_t wz = wo * g->stride_w + ew - g->pad_w;
                    if (wz < 0 || wz >= Wz) continue;
                    z[((n * g->K + k) * Hz + hz) * Wz + wz] = dy[dy_off(g, layout, n, k, ho, wo)];
                }
            }
    for (int64_t n = 0; n < g->N; ++n)
        for (int64_t c = 0; c < g->C; ++c) {
            int64_t gi = c / Cg, cg = c % Cg;
            for (int64_t hi = 0; hi < g->Hi; ++hi)
                for (int64_t wi = 0; wi < g->Wi; ++wi) {
                    double s = 0.0;
                    for (int64_t kk = 0; kk < Kg; ++kk) {
                        int64_t k = gi * Kg + kk;
                        for (int64_t r = 0; r < g->Y; ++r)
                            for (int64_t q = 0; q < g->X; ++q)
                                s += z[((n * g->K + k) * Hz + hi + r * g->dil_h) * Wz + wi + q * g->dil_w] *
                                     w[w_off(g, layout, k, cg, g->Y - 1 - r, g->X - 1 - q)];
                    }
                    dx[dx_off(g, layout, n, c, hi, wi)] = s;
                }
        }
    free(z);
    return 0;
}

/* Forward cross-correlation y = fwd(x, w) with the same geometry: x has dx's
 * shape, the result has dy's shape (a textbook gather loop). */
void oracle_conv_fwd(const oracle_geom *g, int layout, const double *x, const double *w, double *out) {
    const int64_t G = g->groups, Cg = g->C / G, Kg = g->K / G;
    for (int64_t n = 0; n < g->N; ++n)
        for (int64_t k = 0; k < g->K; ++k) {
            int64_t gi = k / Kg;
            for (int64_t ho = 0; ho < g->Ho; ++ho)
                for (int64_t wo = 0; wo < g->Wo; ++wo) {
                    double s = 0.0;
                    for (int64_t cg = 0; cg < Cg; ++cg)
                        for (int64_t y = 0; y < g->Y; ++y) {
                            int64_t hi = ho * g->stride_h - g->pad_h + y * g->dil_h;
                            if (hi < 0 || hi >= g->Hi) continue;
                            for (int64_t q = 0; q < g->X; ++q) {
                                int64_t wi = wo * g->stride_w - g->pad_w + q * g->dil_w;
                                if (wi < 0 || wi >= g->Wi) continue;
                                s += x[dx_off(g, layout, n, gi * Cg + cg, hi, wi)] * w[w_off(g, layout, k, cg, y, q)];
                            }
                        }
                    out[dy_off(g, layout, n, k, ho, wo)] = s;
                }
        }
}

/* Number of OpenMP threads the scatter loop would use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
