/*
 * msssim_oracle.c — plain CPU reference of MS-SSIM on the luma plane.
 *
 * TEST INFRASTRUCTURE ONLY (see ss2_oracle.h).  Shares no code with the
 * CUDA library.
 *
 * Source: "Research-1363: Device-resident ssimulacra2 and a single-wait
 * MS-SSIM on SYCL" (vmafx documentation), Findings 6 and 9: float_ms_ssim
 * computes every scale of a frame and reports one score (and, with
 * enable_lcs, the per-scale terms); the page gives no formula.  The method is
 * the one published by Wang, Simoncelli and Bovik, "Multi-scale structural
 * similarity for image quality assessment" (Asilomar 2003), read as:
 *   - M = 5 scales; scale 1 is the luma plane, scale j + 1 the scale-j
 *     plane low-passed by a 2x2 average and decimated by two, with the edge
 *     sample repeated for odd sizes (out(X, Y) = mean of in(min(2X + dx,
 *     w - 1), min(2Y + dy, h - 1)), dx, dy in {0, 1}), ceil(w / 2) x
 *     ceil(h / 2);
 *   - at every scale the SSIM statistics of an 11x11 Gaussian window
 *     (sigma 1.5, normalised to sum 1) wherever it fits; K1 = 0.01,
 *     K2 = 0.03, C3 = C2 / 2, and per position
 *       l  = (2 mu1 mu2 + C1) / (mu1^2 + mu2^2 + C1),
 *       c  = (2 s1 s2 + C2) / (s1^2 + s2^2 + C2),
 *       s  = (s12 + C3) / (s1 s2 + C3),
 *       cs = (2 s12 + C2) / (s1^2 + s2^2 + C2)    (= c s, as C3 = C2 / 2),
 *     with s1, s2 the square roots of the variances clamped at zero;
 *   - the per-scale means of l, c, s, cs and l cs over the positions;
 *   - MS-SSIM = prod_{j<5} mean(cs_j)^beta_j * mean(l cs)_5^beta_5 with
 *     beta = (0.0448, 0.2856, 0.3001, 0.2363, 0.1333) (the published
 *     exponents; a negative mean gives NaN, as pow does).
 * Samples are taken in the 8-bit range, raw / 2^(depth - 8), with L = 255
 * (the reading the float_ssim oracle takes for the same family of features).
 * With enable_chroma (Finding 6 lists it among float_ms_ssim's outputs and
 * asks for a span per (plane, scale)), the Cb and Cr planes are scored too,
 * each on its own at chroma resolution (ceil(w / 2^sx) x ceil(h / 2^sy))
 * with the same method and constants: the page names the option only, so
 * the plainest reading is one MS-SSIM score per plane.
 * Everything is fp64.  Frames whose scale-5 plane is below 11x11 are refused
 * (-95).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "ss2_oracle.h"

#define WIN 11
#define NSCALE 5

static const double kBeta[NSCALE] = {0.0448, 0.2856, 0.3001, 0.2363, 0.1333};

void ss2o_msssim_dims(int w, int h, int *dims)
{
    for (int j = 0; j < NSCALE; ++j) {
        dims[2 * j] = w;
        dims[2 * j + 1] = h;
        w = (w + 1) / 2;
        h = (h + 1) / 2;
    }
}

/* Scale-1 plane: luma in the 8-bit range.                                  */
static void luma_plane(const void *frame, int w, int h, int depth, double *out)
{
    const double norm = 1.0 / (double)(1 << (depth - 8));
    const size_t n = (size_t)w * h;
    if (depth == 8) {
        const uint8_t *f = (const uint8_t *)frame;
        for (size_t i = 0; i < n; ++i) out[i] = (double)f[i] * norm;
    } else {
        const uint8_t *f = (const uint8_t *)frame;
        for (size_t i = 0; i < n; ++i)
            out[i] = (double)((int)f[2 * i] | ((int)f[2 * i + 1] << 8)) * norm;
    }
}

/* 2x2 average with the edge sample repeated.                               */
static void halve(const double *in, int w, int h, double *out)
{
    const int wo = (w + 1) / 2, ho = (h + 1) / 2;
    for (int y = 0; y < ho; ++y) {
        const int y0 = 2 * y, y1 = 2 * y + 1 < h ? 2 * y + 1 : h - 1;
        for (int x = 0; x < wo; ++x) {
            const int x0 = 2 * x, x1 = 2 * x + 1 < w ? 2 * x + 1 : w - 1;
            out[(size_t)y * wo + x] = (in[(size_t)y0 * w + x0] + in[(size_t)y0 * w + x1] +
                                       in[(size_t)y1 * w + x0] + in[(size_t)y1 * w + x1]) / 4.0;
        }
    }
}

/* Means of l, c, s, cs and l cs over the valid windows of one scale.       */
static void scale_means(const double *a, const double *b, int w, int h, double *m5)
{
    double g[WIN], gs = 0.0;
    for (int i = 0; i < WIN; ++i) {
        const double t = (double)(i - WIN / 2);
        g[i] = exp(-t * t / (2.0 * 1.5 * 1.5));
        gs += g[i];
    }
    for (int i = 0; i < WIN; ++i) g[i] /= gs;
    const double L = 255.0;
    const double C1 = (0.01 * L) * (0.01 * L), C2 = (0.03 * L) * (0.03 * L), C3 = C2 / 2.0;
    double acc[5] = {0, 0, 0, 0, 0};
    long n = 0;
    for (int y = 0; y + WIN <= h; ++y) {
        for (int x = 0; x + WIN <= w; ++x) {
            double m1 = 0, m2 = 0, s11 = 0, s22 = 0, s12 = 0;
            for (int j = 0; j < WIN; ++j)
                for (int i = 0; i < WIN; ++i) {
                    const double wgt = g[j] * g[i];
                    const double p = a[(size_t)(y + j) * w + x + i];
                    const double q = b[(size_t)(y + j) * w + x + i];
                    m1 += wgt * p;
                    m2 += wgt * q;
                    s11 += wgt * p * p;
                    s22 += wgt * q * q;
                    s12 += wgt * p * q;
                }
            double v1 = s11 - m1 * m1, v2 = s22 - m2 * m2;
            const double cv = s12 - m1 * m2;
            if (v1 < 0.0) v1 = 0.0;
            if (v2 < 0.0) v2 = 0.0;
            const double sd1 = sqrt(v1), sd2 = sqrt(v2);
            const double l = (2.0 * m1 * m2 + C1) / (m1 * m1 + m2 * m2 + C1);
            const double c = (2.0 * sd1 * sd2 + C2) / (v1 + v2 + C2);
            const double s = (cv + C3) / (sd1 * sd2 + C3);
            const double cs = (2.0 * cv + C2) / (v1 + v2 + C2);
            acc[0] += l;
            acc[1] += c;
            acc[2] += s;
            acc[3] += cs;
            acc[4] += l * cs;
            ++n;
        }
    }
    for (int k = 0; k < 5; ++k) m5[k] = acc[k] / (double)n;
}

int ss2o_msssim_pyramid(const void *frame, int w, int h, int depth, double *levels)
{
    if (w < 1 || h < 1 || depth < 8 || depth > 16) return -22;
    int dims[2 * NSCALE];
    ss2o_msssim_dims(w, h, dims);
    luma_plane(frame, w, h, depth, levels);
    double *cur = levels;
    for (int j = 1; j < NSCALE; ++j) {
        double *next = cur + (size_t)dims[2 * (j - 1)] * dims[2 * (j - 1) + 1];
        halve(cur, dims[2 * (j - 1)], dims[2 * (j - 1) + 1], next);
        cur = next;
    }
    return 0;
}

size_t ss2o_msssim_pyramid_len(int w, int h)
{
    int dims[2 * NSCALE];
    ss2o_msssim_dims(w, h, dims);
    size_t n = 0;
    for (int j = 0; j < NSCALE; ++j) n += (size_t)dims[2 * j] * dims[2 * j + 1];
    return n;
}

int ss2o_msssim(const void *ref, const void *dis, int w, int h, int depth, double *score,
                double *values)
{
    if (w < 1 || h < 1 || depth < 8 || depth > 16) return -22;
    int dims[2 * NSCALE];
    ss2o_msssim_dims(w, h, dims);
    if (dims[2 * (NSCALE - 1)] < WIN || dims[2 * (NSCALE - 1) + 1] < WIN) return -95;
    const size_t len = ss2o_msssim_pyramid_len(w, h);
    double *pa = malloc(sizeof(double) * len), *pb = malloc(sizeof(double) * len);
    if (!pa || !pb) {
        free(pa);
        free(pb);
        return -12;
    }
    ss2o_msssim_pyramid(ref, w, h, depth, pa);
    ss2o_msssim_pyramid(dis, w, h, depth, pb);
    double m[NSCALE][5];
    size_t off = 0;
    for (int j = 0; j < NSCALE; ++j) {
        scale_means(pa + off, pb + off, dims[2 * j], dims[2 * j + 1], m[j]);
        off += (size_t)dims[2 * j] * dims[2 * j + 1];
    }
    double ms = 1.0;
    for (int j = 0; j < NSCALE - 1; ++j) ms *= pow(m[j][3], kBeta[j]);
    ms *= pow(m[NSCALE - 1][4], kBeta[NSCALE - 1]);
    if (score) *score = ms;
    if (values) memcpy(values, m, sizeof(m));
    free(pa);
    free(pb);
    return 0;
}

/* Per-plane scores of a packed frame pair: plane 0 is luma, 1 Cb, 2 Cr
 * (nplanes 1 or 3).  scores[p], values[p][5][5] (values may be NULL).    */
int ss2o_msssim_planes(const void *ref, const void *dis, int w, int h, int depth,
                       int chroma, int nplanes, double *scores, double *values)
{
    int sx, sy;
    switch (chroma) {
    case 420: sx = 1; sy = 1; break;
    case 422: sx = 1; sy = 0; break;
    case 444: sx = 0; sy = 0; break;
    default: return -22;
    }
    if (nplanes != 1 && nplanes != 3) return -22;
    const size_t bps = depth > 8 ? 2 : 1;
    const int cw = (w + sx) >> sx, ch = (h + sy) >> sy;
    for (int p = 0; p < nplanes; ++p) {
        const int pw = p ? cw : w, ph = p ? ch : h;
        const size_t off = p == 0 ? 0 : (size_t)w * h + (size_t)(p - 1) * cw * ch;
        const int rc = ss2o_msssim((const uint8_t *)ref + off * bps,
                                   (const uint8_t *)dis + off * bps, pw, ph, depth,
                                   scores + p, values ? values + (size_t)p * 25 : NULL);
        if (rc) return rc;
    }
    return 0;
}
