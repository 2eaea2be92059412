/*
 * cambi_oracle.c — plain CPU reference of CAMBI's c-values and top-K pool.
 *
 * TEST INFRASTRUCTURE ONLY (see ss2_oracle.h).  Shares no code with the
 * CUDA library.
 *
 * Source: "ADR-1357: Run the SYCL CAMBI extractor entirely on the device"
 * (vmafx documentation), Decision.  The two stages this covers:
 *   - c-values: for every pixel, counts of levels in its window (at most
 *     65 x 65: window^2 < 4226), and the per-pixel value w * p0 * pm /
 *     (p0 + pm) formed "float for float" as (float)(w p0 pm) times a
 *     reciprocal table entry, with p0, pm counts of at least one;
 *   - top-K pooling: the k-th largest c-value T, and the exact sum
 *     sum(v > T) + (k - #(v > T)) T in units of 2^-24 (every nonzero
 *     c-value is a multiple of 2^-24 in [0.5, 2^14)).
 * Readings (the page leaves these open; the stages before, 10-bit
 * conversion, spatial mask, decimation and mode filter, are inputs here):
 *   - the window of (x, y) is the W x W square centred on it, clipped to the
 *     plane; a pixel counts when its mask byte is nonzero (no mask: all);
 *   - p0 = count of the pixel's own level L, pm = count of level L + d for
 *     each (d, w) of a diff table (d >= 1, w in 1..9); the c-value is the
 *     largest term over the table, 0 when pm = 0, and 0 for an unmasked
 *     pixel;
 *   - the reciprocal table is R[n] = 1/n rounded to nearest fp32 (the page
 *     says 42 entries of cambi.c's table are one ulp away from 1.0f / n but
 *     does not list them);
 *   - the pool is the mean S / k of the exact top-K sum S.
 * Everything here is exact integer counting plus the one fp32 product per
 * term the page specifies; the top-K sum uses unsigned __int128.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "ss2_oracle.h"

#define CAMBI_LEVELS 1024
#define CAMBI_MAX_WIN2 4225

float ss2o_cambi_recip(int n)
{
    return 1.0f / (float)n;   /* IEEE division: correctly rounded */
}

/* The c-value of pixel (x, y): counts over its clipped window by a direct
 * scan, then the largest term of the diff table.                          */
static float cvalue_at(const uint16_t *levels, const uint8_t *mask, int w, int h, int window,
                       int ndiff, const int *diffs, const int *weights, int x, int y)
{
    const size_t at = (size_t)y * w + x;
    if (mask && !mask[at]) return 0.0f;
    const int r = window / 2;
    const int L = levels[at];
    long p0 = 0, pm[4] = {0, 0, 0, 0};
    for (int yy = y - r; yy <= y + r; ++yy) {
        if (yy < 0 || yy >= h) continue;
        for (int xx = x - r; xx <= x + r; ++xx) {
            if (xx < 0 || xx >= w) continue;
            const size_t j = (size_t)yy * w + xx;
            if (mask && !mask[j]) continue;
            const int v = levels[j];
            if (v == L) ++p0;
            for (int i = 0; i < ndiff; ++i)
                if (v == L + diffs[i]) ++pm[i];
        }
    }
    float best = 0.0f;
    for (int i = 0; i < ndiff; ++i) {
        if (pm[i] == 0) continue;
        const long num = (long)weights[i] * p0 * pm[i];
        const float c = (float)num * ss2o_cambi_recip((int)(p0 + pm[i]));
        if (c > best) best = c;
    }
    return best;
}

int ss2o_cambi_cvalues(const uint16_t *levels, const uint8_t *mask, int w, int h, int window,
                       int ndiff, const int *diffs, const int *weights, float *out)
{
    if (w < 1 || h < 1 || window < 1 || !(window & 1) || window * window > CAMBI_MAX_WIN2)
        return -22;
    if (ndiff < 1 || ndiff > 4) return -22;
    for (int i = 0; i < ndiff; ++i)
        if (diffs[i] < 1 || diffs[i] >= CAMBI_LEVELS || weights[i] < 1 || weights[i] > 9)
            return -22;
    for (size_t i = 0; i < (size_t)w * h; ++i)
        if (levels[i] >= CAMBI_LEVELS) return -22;
    for (int y = 0; y < h; ++y)
        for (int x = 0; x < w; ++x)
            out[(size_t)y * w + x] = cvalue_at(levels, mask, w, h, window, ndiff, diffs,
                                               weights, x, y);
    return 0;
}

int ss2o_cambi_cvalue_at(const uint16_t *levels, const uint8_t *mask, int w, int h, int window,
                         int ndiff, const int *diffs, const int *weights, int x, int y,
                         float *out)
{
    if (x < 0 || x >= w || y < 0 || y >= h) return -22;
    *out = cvalue_at(levels, mask, w, h, window, ndiff, diffs, weights, x, y);
    return 0;
}

/* Exact top-K sum of non-negative c-values (multiples of 2^-24 below 2^14)
 * in units of 2^-24, by its definition: the k-th largest value T found by
 * sorting, then the elements above T plus (k - #above) copies of T.        */
static int cmp_desc(const void *a, const void *b)
{
    const float x = *(const float *)a, y = *(const float *)b;
    return (x < y) - (x > y);
}

int ss2o_cambi_topk(const float *c, long n, long k, uint64_t *sum_lo, uint64_t *sum_hi,
                    float *threshold, double *mean)
{
    if (n < 1 || k < 1 || k > n) return -22;
    float *s = malloc(sizeof(float) * (size_t)n);
    if (!s) return -12;
    memcpy(s, c, sizeof(float) * (size_t)n);
    qsort(s, (size_t)n, sizeof(float), cmp_desc);
    const float T = s[k - 1];
    unsigned __int128 S = 0;
    long above = 0;
    for (long i = 0; i < n; ++i) {
        if (!(c[i] >= 0.0f) || c[i] >= 16384.0f) {
            free(s);
            return -22;
        }
        const double units = (double)c[i] * 16777216.0;   /* exact: c is on the 2^-24 grid */
        if ((double)(uint64_t)units != units) {
            free(s);
            return -22;
        }
        if (c[i] > T) {
            S += (uint64_t)units;
            ++above;
        }
    }
    S += (unsigned __int128)(uint64_t)(k - above) * (uint64_t)((double)T * 16777216.0);
    *sum_lo = (uint64_t)S;
    *sum_hi = (uint64_t)(S >> 64);
    *threshold = T;
    /* the mean S 2^-24 / k: S and k are exact, one division in long double */
    *mean = (double)((long double)S / 16777216.0L / (long double)k);
    free(s);
    return 0;
}
