/*
 * fssim_oracle.c — plain CPU reference of float_ssim with decimation.
 *
 * TEST INFRASTRUCTURE ONLY (see ss2_oracle.h).  Shares no code with the
 * CUDA library.
 *
 * Source: "ADR-1405: float_ssim_hip decimates on the device, bit-identical
 * to the CPU" (vmafx documentation), Context and Decision 1 and 4:
 *   - decimation factor max(1, round(min(w, h) / 256));
 *   - each plane is low-passed with a scale x scale box of weight
 *     1.0f / (scale * scale) and decimated: output (x, y) is the filter at
 *     (x * scale, y * scale) with offsets -scale/2 .. scale-1-scale/2 and
 *     symmetric edges; every tap is the fp32 product sample * weight and the
 *     taps are summed exactly (an int64 count of 2^-52 units on the page),
 *     then rounded once to fp32;
 *   - SSIM on the decimated planes with an 11x11 Gaussian window; planes
 *     smaller than the window or scales above 128 are refused.
 * Readings (the page is silent): samples are taken in the 8-bit range,
 * raw / 2^(depth - 8) (exact in fp32), and L = 255 -- the page's window sum
 * in 2^-52 units is exact "up to scale 128" and its planes byte-identical at
 * 10, 12 and 16 bits only if every sample stays below 2^11, which raw 12- and
 * 16-bit samples do not; decimated dims ceil(w / scale) x ceil(h / scale);
 * "symmetric" edges mirror with the edge sample repeated (-1 -> 0,
 * w -> w-1); SSIM as Wang et al. (2004): Gaussian window sigma 1.5
 * normalised to sum 1, evaluated where the window fits ("valid"), K1 = 0.01,
 * K2 = 0.03, the score the mean of the map; luma only.
 *
 * The exact window sum: a tap is sample * w rounded to float with sample a
 * multiple of 2^-8 below 256 and w = RN(1 / scale^2) >= 2^-14 (scale <= 128),
 * so every nonzero tap is at least 2^-22, a multiple of 2^-45, and the window
 * sum stays below 256 = 2^53 * 2^-45: an fp64 running sum of the taps is
 * exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "ss2_oracle.h"

#define EINVAL_RC (-22)
#define ENOTSUP_RC (-95)
#define WIN 11

int ss2o_fssim_scale(int w, int h)
{
    int m = w < h ? w : h;
    int s = (int)lround((double)m / 256.0);
    return s < 1 ? 1 : s;
}

int ss2o_fssim_dims(int w, int h, int *wd, int *hd)
{
    int s = ss2o_fssim_scale(w, h);
    *wd = (w + s - 1) / s;
    *hd = (h + s - 1) / s;
    return s;
}

static int mirror(int i, int n)
{
    while (i < 0 || i >= n) {
        if (i < 0) i = -1 - i;
        if (i >= n) i = 2 * n - 1 - i;
    }
    return i;
}

static int luma(const uint8_t *f, int w, int x, int y, int bps)
{
    size_t i = (size_t)y * w + x;
    if (bps == 1) return f[i];
    return (int)f[2 * i] | ((int)f[2 * i + 1] << 8);
}

/* A luma sample in the 8-bit range: raw / 2^(depth - 8), exact in fp32.     */
static float sample8(const uint8_t *f, int w, int x, int y, int bps, float norm)
{
    return (float)luma(f, w, x, y, bps) * norm;
}

int ss2o_fssim_decimate(const void *frame, int w, int h, int depth, float *out)
{
    if (w < 1 || h < 1 || depth < 8 || depth > 16) return EINVAL_RC;
    const int s = ss2o_fssim_scale(w, h);
    if (s > 128) return ENOTSUP_RC;
    const int bps = depth > 8 ? 2 : 1;
    const float norm = 1.0f / (float)(1 << (depth - 8));
    const uint8_t *f = (const uint8_t *)frame;
    int wd, hd;
    ss2o_fssim_dims(w, h, &wd, &hd);
    if (s == 1) {
        for (int y = 0; y < h; ++y)
            for (int x = 0; x < w; ++x) out[(size_t)y * w + x] = sample8(f, w, x, y, bps, norm);
        return 0;
    }
    const float wt = 1.0f / (float)(s * s);
    const int lo = -(s / 2), hi = s - 1 - s / 2;
    for (int y = 0; y < hd; ++y) {
        for (int x = 0; x < wd; ++x) {
            double sum = 0.0;   /* exact: see the file header */
            for (int dy = lo; dy <= hi; ++dy) {
                int yy = mirror(y * s + dy, h);
                for (int dx = lo; dx <= hi; ++dx) {
                    int xx = mirror(x * s + dx, w);
                    float tap = sample8(f, w, xx, yy, bps, norm) * wt;
                    sum += (double)tap;
                }
            }
            out[(size_t)y * wd + x] = (float)sum;
        }
    }
    return 0;
}

/* SSIM of two planes (fp64): Gaussian-weighted means, variances and
 * covariance over every 11x11 window inside the plane, map averaged.       */
static double ssim_planes(const float *a, const float *b, int w, int h, double L)
{
    double g[WIN], gs = 0.0;
    for (int i = 0; i < WIN; ++i) {
        double t = (double)(i - WIN / 2);
        g[i] = exp(-t * t / (2.0 * 1.5 * 1.5));
        gs += g[i];
    }
    for (int i = 0; i < WIN; ++i) g[i] /= gs;
    const double C1 = (0.01 * L) * (0.01 * L), C2 = (0.03 * L) * (0.03 * L);
    double total = 0.0;
    long count = 0;
    for (int y = 0; y + WIN <= h; ++y) {
        for (int x = 0; x + WIN <= w; ++x) {
            double m1 = 0, m2 = 0, s11 = 0, s22 = 0, s12 = 0;
            for (int j = 0; j < WIN; ++j) {
                for (int i = 0; i < WIN; ++i) {
                    double wgt = g[j] * g[i];
                    double p = a[(size_t)(y + j) * w + x + i];
                    double q = b[(size_t)(y + j) * w + x + i];
                    m1 += wgt * p;
                    m2 += wgt * q;
                    s11 += wgt * p * p;
                    s22 += wgt * q * q;
                    s12 += wgt * p * q;
                }
            }
            double v1 = s11 - m1 * m1, v2 = s22 - m2 * m2, cv = s12 - m1 * m2;
            double num = (2.0 * m1 * m2 + C1) * (2.0 * cv + C2);
            double den = (m1 * m1 + m2 * m2 + C1) * (v1 + v2 + C2);
            total += num / den;
            ++count;
        }
    }
    return total / (double)count;
}

int ss2o_fssim(const void *ref, const void *dis, int w, int h, int depth, double *score,
               float *dec_ref, float *dec_dis)
{
    if (w < 1 || h < 1 || depth < 8 || depth > 16) return EINVAL_RC;
    int wd, hd;
    const int s = ss2o_fssim_dims(w, h, &wd, &hd);
    if (s > 128 || wd < WIN || hd < WIN) return ENOTSUP_RC;
    const size_t n = (size_t)wd * hd;
    float *a = malloc(sizeof(float) * n), *b = malloc(sizeof(float) * n);
    if (!a || !b) {
        free(a);
        free(b);
        return -12;
    }
    ss2o_fssim_decimate(ref, w, h, depth, a);
    ss2o_fssim_decimate(dis, w, h, depth, b);
    if (score) *score = ssim_planes(a, b, wd, hd, 255.0);
    if (dec_ref) memcpy(dec_ref, a, sizeof(float) * n);
    if (dec_dis) memcpy(dec_dis, b, sizeof(float) * n);
    free(a);
    free(b);
    return 0;
}
