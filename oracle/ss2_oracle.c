/*
 * ss2_oracle.c — plain single-threaded CPU reference of the per-frame
 * SSIMULACRA2 scoring pipeline.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the CPU
 * baseline leg of the benchmark, never by the CUDA library, with which it
 * shares no code.
 *
 * What is computed follows "Research-1363: Device-resident ssimulacra2 and a
 * single-wait MS-SSIM on SYCL" (vmafx documentation):
 *   - "Sources": the CPU pipeline steps picture_to_linear_rgb,
 *     linear_rgb_to_xyb, fast_gaussian_1d / blur_plane, multiply_3plane,
 *     ssim_map, edge_diff_map, downsample_2x2, pool_score, with the per-pixel
 *     fp64 terms accumulated in sequential order;
 *   - Finding 2: contraction off, products in named temporaries, fma for the
 *     YUV matrix, an sRGB EOTF table, a cube root with a correctly rounded
 *     division step (here: a correctly rounded cube root);
 *   - Finding 3: the sums are fp64, one term after the other;
 *   - Finding 4: the per-pixel SSIM term is built from the product
 *     num_m * num_s of two floats, a quotient and 1 - q; the edge term is the
 *     ratio (1 + |r2 - mu2|) / (1 + |r1 - mu1|) - 1; fourth powers; six sums
 *     per channel;
 *   - Finding 7: the IIR is a sequential recurrence along each line,
 *     horizontal pass then vertical pass.
 *
 * Readings taken where the pages are silent (each restated at its function):
 *   chroma siting (nearest), BT.709 limited-range matrix, EOTF table size and
 *   interpolation, the XYB opsin parameters, the scale loop on linear RGB with
 *   a stop below 8 pixels, ceil-halving downsample with edge clamp, the
 *   truncated-cosine recursive Gaussian (three odd harmonics, support |m|<=4,
 *   least-squares fit to the sigma = 1.5 Gaussian), C2 = 0.0009 with no C1
 *   term, the clamps d >= 0 and art/det >= 0, the 108-value ordering and the
 *   final polynomial map.
 *
 * Default parameters: the opsin mixing matrix and bias are the XYB colour
 * space's published values (JPEG XL, ISO/IEC 18181-1).  The 108 pooling
 * weights, the final map and the "make positive" affine are SSIMULACRA2's
 * tuned constants, which the pages do not give: the defaults are labelled
 * placeholders (uniform weights 1/108, score = 100 - 100 P, identity affine
 * with B' = B - Y).  Any real table can be passed in the parameter vector.
 *
 * Build with -ffp-contract=off and without fast-math.
 */
#include "ss2_oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EINVAL_RC (-22)
#define NQ 5            /* blurred quantities per channel: mu1 mu2 s11 s22 s12 */
#define NSUM 6          /* d, d^4, art, art^4, det, det^4                      */

/* ------------------------------------------------------------------------ */
/* Parameters                                                                */
/* ------------------------------------------------------------------------ */

void ss2o_default_params(double *p)
{
    memset(p, 0, sizeof(double) * SS2O_NPARAMS);
    for (int i = 0; i < SS2O_NVALUES; ++i)
        p[SS2O_P_WEIGHTS + i] = 1.0 / 108.0;          /* placeholder */
    p[SS2O_P_POLY + 0] = 100.0;                        /* placeholder map */
    p[SS2O_P_POLY + 1] = -100.0;
    p[SS2O_P_POWER + 0] = 1.0;
    p[SS2O_P_POWER + 1] = 1.0;
    p[SS2O_P_POWER + 2] = 0.0;
    /* XYB opsin mixing matrix and bias (JPEG XL, ISO/IEC 18181-1). */
    static const double opsin[9] = {
        0.30, 0.622, 0.078,
        0.23, 0.692, 0.078,
        0.24342268924547819, 0.20476744424496821, 0.55180986650955360,
    };
    for (int i = 0; i < 9; ++i) p[SS2O_P_OPSIN + i] = opsin[i];
    for (int i = 0; i < 3; ++i) p[SS2O_P_BIAS + i] = 0.0037930732552754493;
    p[SS2O_P_AFFINE + 0] = 1.0;   /* sx  (placeholder) */
    p[SS2O_P_AFFINE + 1] = 0.0;   /* ox  */
    p[SS2O_P_AFFINE + 2] = 0.0;   /* oy  */
    p[SS2O_P_AFFINE + 3] = 1.0;   /* sb  */
    p[SS2O_P_AFFINE + 4] = 0.0;   /* ob  */
    p[SS2O_P_C2] = 0.0009;        /* (0.03 * 1)^2, textbook SSIM C2 */
}

/* ------------------------------------------------------------------------ */
/* Geometry                                                                  */
/* ------------------------------------------------------------------------ */

static int chroma_shift(int chroma, int *sx, int *sy)
{
    switch (chroma) {
    case 420: *sx = 1; *sy = 1; return 0;
    case 422: *sx = 1; *sy = 0; return 0;
    case 444: *sx = 0; *sy = 0; return 0;
    default: return EINVAL_RC;
    }
}

/* Same acceptance rule as the library: w, h >= 8, depth 8..16, chroma in
 * {420, 422, 444}, and an even width for subsampled chroma (the page's
 * fixtures note that the CLI rejects odd widths for 4:2:0).                 */
static int check_geometry(int w, int h, int depth, int chroma)
{
    int sx = 0, sy = 0;
    if (w < 8 || h < 8 || w > 65536 || h > 65536) return EINVAL_RC;
    if (depth < 8 || depth > 16) return EINVAL_RC;
    if (chroma_shift(chroma, &sx, &sy)) return EINVAL_RC;
    if (sx && (w & 1)) return EINVAL_RC;
    return 0;
}

size_t ss2o_frame_bytes(int w, int h, int depth, int chroma)
{
    int sx = 0, sy = 0;
    chroma_shift(chroma, &sx, &sy);
    size_t cw = (size_t)((w + sx) >> sx), ch = (size_t)((h + sy) >> sy);
    size_t bps = depth > 8 ? 2 : 1;
    return ((size_t)w * (size_t)h + 2 * cw * ch) * bps;
}

/* Scale s has dims ceil(w/2^s) x ceil(h/2^s); a scale is computed only while
 * both dims are >= 8, at most 6 scales.                                     */
int ss2o_scale_dims(int w, int h, int *ws, int *hs)
{
    int n = 0;
    while (n < SS2O_NSCALES && w >= 8 && h >= 8) {
        ws[n] = w; hs[n] = h; ++n;
        w = (w + 1) / 2; h = (h + 1) / 2;
    }
    return n;
}

/* ------------------------------------------------------------------------ */
/* Correctly rounded cube root                                               */
/* ------------------------------------------------------------------------ */

/* A positive finite float as X * 2^e with X an integer < 2^24. */
static void float_parts(float v, uint32_t *X, int *e)
{
    uint32_t bits;
    memcpy(&bits, &v, 4);
    uint32_t be = (bits >> 23) & 0xff, m = bits & 0x7fffff;
    if (be == 0) { *X = m; *e = -149; }
    else { *X = m | 0x800000u; *e = (int)be - 150; }
}

/* Sign of (M * 2^f)^3 - x, exact.  M < 2^26, x positive finite. */
static int cube_cmp(uint64_t M, int f, float x)
{
    uint32_t X; int g;
    float_parts(x, &X, &g);
    unsigned __int128 c = (unsigned __int128)M * M * M;     /* < 2^78 */
    int d = 3 * f - g;               /* compare c * 2^d with X */
    if (d >= 0) {
        if (d >= 24) return 1;       /* c >= 1 and X < 2^24 */
        unsigned __int128 lhs = c << d, rhs = X;
        return lhs > rhs ? 1 : (lhs < rhs ? -1 : 0);
    } else {
        if (-d >= 100) return X ? -1 : 1;   /* c < 2^78 */
        unsigned __int128 rhs = (unsigned __int128)X << (-d);
        return c > rhs ? 1 : (c < rhs ? -1 : 0);
    }
}

/* cbrt(x) rounded to nearest float.  Start from the double cube root and
 * move one float at a time until x lies strictly between the cubes of the
 * two midpoints around the candidate (no ties exist: an odd 25+-bit
 * midpoint cubed has no 24-bit representation).                            */
float ss2o_cbrtf_cr(float x)
{
    if (x == 0.0f || isnan(x) || isinf(x)) return x;
    if (x < 0.0f) return -ss2o_cbrtf_cr(-x);
    float y = (float)cbrt((double)x);
    for (int it = 0; it < 8; ++it) {
        uint32_t Y; int e;
        float_parts(y, &Y, &e);
        /* upper midpoint (2Y+1) 2^(e-1) */
        if (cube_cmp(2 * (uint64_t)Y + 1, e - 1, x) < 0) {
            y = nextafterf(y, INFINITY);
            continue;
        }
        /* lower midpoint: below a power of two the spacing halves */
        int at_binade_floor = (Y == 0x800000u) && (e > -149);
        uint64_t Ml = at_binade_floor ? 4 * (uint64_t)Y - 1 : 2 * (uint64_t)Y - 1;
        int fl = at_binade_floor ? e - 2 : e - 1;
        if (cube_cmp(Ml, fl, x) > 0) {
            y = nextafterf(y, 0.0f);
            continue;
        }
        break;
    }
    return y;
}

void ss2o_cbrtf_cr_array(const float *x, float *y, long long n)
{
    for (long long i = 0; i < n; ++i) y[i] = ss2o_cbrtf_cr(x[i]);
}

/* ------------------------------------------------------------------------ */
/* sRGB EOTF table                                                           */
/* ------------------------------------------------------------------------ */

/* IEC 61966-2-1 sRGB decoding: V <= 0.04045 -> V / 12.92, else
 * ((V + 0.055) / 1.055)^2.4, evaluated in fp64.                             */
static double srgb_eotf(double v)
{
    if (v <= 0.04045) return v / 12.92;
    return pow((v + 0.055) / 1.055, 2.4);
}

/* Reading: a table on a uniform grid of 4096 intervals over [0, 1], each
 * entry the fp64 EOTF rounded to float.                                     */
void ss2o_eotf_table(float *T)
{
    for (int i = 0; i <= SS2O_EOTF_N; ++i)
        T[i] = (float)srgb_eotf((double)i / (double)SS2O_EOTF_N);
}

/* Linear interpolation in the table for v in [0, 1]. */
float ss2o_eotf_lookup(const float *T, float v)
{
    float t = v * (float)SS2O_EOTF_N;
    int i = (int)t;
    if (i > SS2O_EOTF_N - 1) i = SS2O_EOTF_N - 1;
    float f = t - (float)i;
    float slope = T[i + 1] - T[i];
    return fmaf(f, slope, T[i]);
}

/* ------------------------------------------------------------------------ */
/* YUV -> R'G'B'                                                             */
/* ------------------------------------------------------------------------ */

/* BT.709: Kr = 0.2126, Kb = 0.0722.  R' = Y + 2(1-Kr) Cr, B' = Y + 2(1-Kb) Cb,
 * G' = Y - 2Kb(1-Kb)/Kg Cb - 2Kr(1-Kr)/Kg Cr.  Coefficients formed in fp64
 * and rounded once to float: {cr_r, cb_g, cr_g, cb_b} (signs positive).     */
void ss2o_yuv_coeffs(float *k)
{
    const double kr = 0.2126, kb = 0.0722, kg = 1.0 - kr - kb;
    k[0] = (float)(2.0 * (1.0 - kr));
    k[1] = (float)(2.0 * kb * (1.0 - kb) / kg);
    k[2] = (float)(2.0 * kr * (1.0 - kr) / kg);
    k[3] = (float)(2.0 * (1.0 - kb));
}

static float clamp01(float v)
{
    if (v < 0.0f) return 0.0f;
    if (v > 1.0f) return 1.0f;
    return v;
}

static int read_sample(const uint8_t *base, size_t idx, int bps)
{
    if (bps == 1) return base[idx];
    return (int)base[2 * idx] | ((int)base[2 * idx + 1] << 8);
}

/* One frame to linear RGB planes (w*h each).  Reading: limited range with
 * k = 2^(depth-8): Y' = (Y - 16k) / 219k, Cb = (U - 128k) / 224k, Cr alike,
 * each a correctly rounded float division; nearest chroma siting
 * U[(y >> sy) * cw + (x >> sx)]; fma in the matrix as listed by Finding 2;
 * clamp to [0, 1]; then the EOTF table.                                     */
static void frame_to_linear(const void *frame, int w, int h, int depth,
                            int chroma, const float *T, float *R, float *G,
                            float *B)
{
    int sx = 0, sy = 0;
    chroma_shift(chroma, &sx, &sy);
    const int cw = (w + sx) >> sx, ch = (h + sy) >> sy;
    const int bps = depth > 8 ? 2 : 1;
    const uint8_t *py = (const uint8_t *)frame;
    const uint8_t *pu = py + (size_t)w * h * bps;
    const uint8_t *pv = pu + (size_t)cw * ch * bps;
    const int k = 1 << (depth - 8);
    const float dy = (float)(219 * k), dc = (float)(224 * k);
    float c[4];
    ss2o_yuv_coeffs(c);
    for (int y = 0; y < h; ++y) {
        for (int x = 0; x < w; ++x) {
            size_t ci = (size_t)(y >> sy) * cw + (size_t)(x >> sx);
            int Ys = read_sample(py, (size_t)y * w + x, bps);
            int Us = read_sample(pu, ci, bps);
            int Vs = read_sample(pv, ci, bps);
            float yn = (float)(Ys - 16 * k) / dy;
            float cb = (float)(Us - 128 * k) / dc;
            float cr = (float)(Vs - 128 * k) / dc;
            float r = fmaf(c[0], cr, yn);
            float g = fmaf(-c[2], cr, fmaf(-c[1], cb, yn));
            float b = fmaf(c[3], cb, yn);
            size_t o = (size_t)y * w + x;
            R[o] = ss2o_eotf_lookup(T, clamp01(r));
            G[o] = ss2o_eotf_lookup(T, clamp01(g));
            B[o] = ss2o_eotf_lookup(T, clamp01(b));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Linear RGB -> XYB                                                         */
/* ------------------------------------------------------------------------ */

typedef struct {
    float m[9], bias[3], cbrt_bias[3];
    float sx, ox, oy, sb, ob;
    float c2;
} pix_params;

static void load_pix_params(const double *p, pix_params *pp)
{
    for (int i = 0; i < 9; ++i) pp->m[i] = (float)p[SS2O_P_OPSIN + i];
    for (int i = 0; i < 3; ++i) {
        pp->bias[i] = (float)p[SS2O_P_BIAS + i];
        pp->cbrt_bias[i] = ss2o_cbrtf_cr(pp->bias[i]);
    }
    pp->sx = (float)p[SS2O_P_AFFINE + 0];
    pp->ox = (float)p[SS2O_P_AFFINE + 1];
    pp->oy = (float)p[SS2O_P_AFFINE + 2];
    pp->sb = (float)p[SS2O_P_AFFINE + 3];
    pp->ob = (float)p[SS2O_P_AFFINE + 4];
    pp->c2 = (float)p[SS2O_P_C2];
}

/* Opsin mix m_i = ((a_i0 r + a_i1 g) + a_i2 b) + bias_i (products rounded
 * one by one), clamp at 0, c_i = cbrt(m_i) - cbrt(bias_i), X = (c0 - c1)/2,
 * Y = (c0 + c1)/2, B = c2; then the make-positive affine
 * X' = sx X + ox, Y' = Y + oy, B' = (B - Y) sb + ob.                        */
static void pixel_xyb(const pix_params *pp, float r, float g, float b,
                      float *X, float *Y, float *B)
{
    float c[3];
    for (int i = 0; i < 3; ++i) {
        float t0 = pp->m[3 * i + 0] * r;
        float t1 = pp->m[3 * i + 1] * g;
        float t2 = pp->m[3 * i + 2] * b;
        float s = (t0 + t1) + t2;
        s = s + pp->bias[i];
        if (s < 0.0f) s = 0.0f;
        c[i] = ss2o_cbrtf_cr(s) - pp->cbrt_bias[i];
    }
    float x = 0.5f * (c[0] - c[1]);
    float y = 0.5f * (c[0] + c[1]);
    float bb = c[2];
    float xs = x * pp->sx;
    *X = xs + pp->ox;
    *Y = y + pp->oy;
    float bmy = bb - y;
    float bs = bmy * pp->sb;
    *B = bs + pp->ob;
}

void ss2o_xyb_pixel(const double *params, float r, float g, float b, float *xyb)
{
    pix_params pp;
    load_pix_params(params, &pp);
    pixel_xyb(&pp, r, g, b, &xyb[0], &xyb[1], &xyb[2]);
}

/* ------------------------------------------------------------------------ */
/* Recursive Gaussian                                                        */
/* ------------------------------------------------------------------------ */

/* Reading of "fast_gaussian_1d": the kernel is a sum of three odd cosine
 * harmonics h[m] = sum_k a_k cos(w_k m), w_k = k pi / (2 (R+1)), k = 1, 3, 5,
 * on |m| <= R = 4.  Each harmonic vanishes at m = +-(R+1), so the windowed
 * sum Y_k[n] = a_k sum_{|m|<=R} cos(w_k m) x[n+m] obeys the two-tap resonator
 *   Y_k[n+1] = 2 cos(w_k) Y_k[n] - Y_k[n-1]
 *              + a_k cos(w_k R) (x[n+R+1] + x[n-R-1]).
 * The a_k minimise sum_m (h[m] - G[m])^2 subject to sum_m h[m] = 1, with
 * G[m] = exp(-m^2 / (2 sigma^2)) / (sigma sqrt(2 pi)), sigma = 1.5: a 4x4
 * KKT system solved in fp64 by Gaussian elimination with partial pivoting.
 * The recursion coefficients 2 cos(w_k) and a_k cos(w_k R) are rounded to
 * float.                                                                    */
void ss2o_iir_coeffs(double *a, float *c2, float *g)
{
    const int R = SS2O_IIR_R, L = SS2O_IIR_R + 1;
    const double sigma = 1.5, pi = 3.14159265358979323846;
    double w[3], M[4][5];
    for (int k = 0; k < 3; ++k) w[k] = (double)(2 * k + 1) * pi / (2.0 * L);
    memset(M, 0, sizeof(M));
    for (int m = -R; m <= R; ++m) {
        double G = exp(-(double)(m * m) / (2.0 * sigma * sigma)) /
                   (sigma * sqrt(2.0 * pi));
        double cm[3];
        for (int k = 0; k < 3; ++k) cm[k] = cos(w[k] * m);
        for (int i = 0; i < 3; ++i) {
            for (int j = 0; j < 3; ++j) M[i][j] += cm[i] * cm[j];
            M[i][3] += cm[i];          /* constraint column */
            M[i][4] += cm[i] * G;      /* right-hand side */
        }
    }
    for (int j = 0; j < 3; ++j) M[3][j] = M[j][3];
    M[3][3] = 0.0;
    M[3][4] = 1.0;
    /* elimination with partial pivoting */
    for (int col = 0; col < 4; ++col) {
        int piv = col;
        for (int r = col + 1; r < 4; ++r)
            if (fabs(M[r][col]) > fabs(M[piv][col])) piv = r;
        if (piv != col)
            for (int j = 0; j < 5; ++j) {
                double t = M[col][j]; M[col][j] = M[piv][j]; M[piv][j] = t;
            }
        for (int r = col + 1; r < 4; ++r) {
            double f = M[r][col] / M[col][col];
            for (int j = col; j < 5; ++j) M[r][j] -= f * M[col][j];
        }
    }
    double sol[4];
    for (int r = 3; r >= 0; --r) {
        double s = M[r][4];
        for (int j = r + 1; j < 4; ++j) s -= M[r][j] * sol[j];
        sol[r] = s / M[r][r];
    }
    for (int k = 0; k < 3; ++k) {
        a[k] = sol[k];
        c2[k] = (float)(2.0 * cos(w[k]));
        g[k] = (float)(sol[k] * cos(w[k] * R));
    }
}

typedef struct { float c2[3], g[3]; } iir_t;

/* One line, zero-extended at both ends, walked in order.  With reach
 * N = R + 1: Y[-N] = Y[-N-1] = 0; for i = -N .. n-2 the step forms
 * Y[i+1] from Y[i], Y[i-1] and in = x[i+N] + x[i-N] as
 *   u = fma(g_k, in, -Y_k[i-1]);  Y_k[i+1] = fma(c2_k, Y_k[i], u),
 * and out[i+1] = (Y_1 + Y_3) + Y_5 once i+1 >= 0.                           */
static void blur_line(const iir_t *c, const float *in, ptrdiff_t istride,
                      int n, float *out, ptrdiff_t ostride)
{
    const int N = SS2O_IIR_R + 1;
    float prev[3] = {0.0f, 0.0f, 0.0f}, cur[3] = {0.0f, 0.0f, 0.0f};
    for (int i = -N; i <= n - 2; ++i) {
        float xa = (i + N < n) ? in[(ptrdiff_t)(i + N) * istride] : 0.0f;
        float xb = (i - N >= 0) ? in[(ptrdiff_t)(i - N) * istride] : 0.0f;
        float s = xa + xb;
        for (int k = 0; k < 3; ++k) {
            float u = fmaf(c->g[k], s, -prev[k]);
            float nxt = fmaf(c->c2[k], cur[k], u);
            prev[k] = cur[k];
            cur[k] = nxt;
        }
        if (i + 1 >= 0) {
            float t = cur[0] + cur[1];
            out[(ptrdiff_t)(i + 1) * ostride] = t + cur[2];
        }
    }
}

static void get_iir(iir_t *c)
{
    double a[3];
    ss2o_iir_coeffs(a, c->c2, c->g);
}

void ss2o_blur_line(const float *in, int n, float *out)
{
    iir_t c;
    get_iir(&c);
    blur_line(&c, in, 1, n, out, 1);
}

/* Horizontal pass over every row, then vertical pass over every column. */
static void blur_plane(const iir_t *c, const float *in, int w, int h,
                       float *tmp, float *out)
{
    for (int y = 0; y < h; ++y)
        blur_line(c, in + (size_t)y * w, 1, w, tmp + (size_t)y * w, 1);
    for (int x = 0; x < w; ++x)
        blur_line(c, tmp + x, w, h, out + x, w);
}

/* ------------------------------------------------------------------------ */
/* Downsample                                                                */
/* ------------------------------------------------------------------------ */

/* Reading: output dims ceil(w/2) x ceil(h/2); sources beyond the last
 * row/column are clamped to it; ((p00 + p01) + p10) + p11, then * 0.25.    */
void ss2o_downsample(const float *in, int w, int h, float *out)
{
    int ow = (w + 1) / 2, oh = (h + 1) / 2;
    for (int y = 0; y < oh; ++y) {
        int y0 = 2 * y, y1 = 2 * y + 1 < h ? 2 * y + 1 : h - 1;
        for (int x = 0; x < ow; ++x) {
            int x0 = 2 * x, x1 = 2 * x + 1 < w ? 2 * x + 1 : w - 1;
            float s = in[(size_t)y0 * w + x0] + in[(size_t)y0 * w + x1];
            s = s + in[(size_t)y1 * w + x0];
            s = s + in[(size_t)y1 * w + x1];
            out[(size_t)y * ow + x] = s * 0.25f;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Per-pixel maps                                                            */
/* ------------------------------------------------------------------------ */

/* ssim_map term (Finding 4).  fp32: dm = mu1 - mu2, num_m = 1 - dm^2,
 * num_s = 2 (s12 - mu1 mu2) + C2, den_s = (s11 - mu1^2) + (s22 - mu2^2) + C2.
 * fp64: q = (num_m * num_s) / den_s, d = 1 - q, clamped at 0 (reading).   */
static double ssim_term(float mu1, float mu2, float s11, float s22, float s12,
                        float c2)
{
    float dm = mu1 - mu2;
    float dm2 = dm * dm;
    float num_m = 1.0f - dm2;
    float m12 = mu1 * mu2;
    float cov = s12 - m12;
    float cov2 = 2.0f * cov;
    float num_s = cov2 + c2;
    float m11 = mu1 * mu1;
    float v1 = s11 - m11;
    float m22 = mu2 * mu2;
    float v2 = s22 - m22;
    float vs = v1 + v2;
    float den_s = vs + c2;
    double num = (double)num_m * (double)num_s;
    double q = num / (double)den_s;
    double d = 1.0 - q;
    return d > 0.0 ? d : 0.0;
}

/* edge_diff_map term (Finding 4): r = (1 + |x2 - mu2|) / (1 + |x1 - mu1|) - 1
 * in fp64 from fp32 absolute differences; artifact = max(r, 0),
 * detail lost = max(-r, 0).                                                 */
static double edge_term(float x1, float mu1, float x2, float mu2)
{
    float a2 = fabsf(x2 - mu2);
    float a1 = fabsf(x1 - mu1);
    double num = 1.0 + (double)a2;
    double den = 1.0 + (double)a1;
    return num / den - 1.0;
}

static double pow4(double v)
{
    double v2 = v * v;
    return v2 * v2;
}

/* ------------------------------------------------------------------------ */
/* The frame pipeline                                                        */
/* ------------------------------------------------------------------------ */

int ss2o_score(const void *ref, const void *dis, int w, int h, int depth,
               int chroma, const double *params, double *score_out,
               double *values_out, const ss2o_dump *dump)
{
    int rc = check_geometry(w, h, depth, chroma);
    if (rc) return rc;
    int ws[SS2O_NSCALES], hs[SS2O_NSCALES];
    int nscales = ss2o_scale_dims(w, h, ws, hs);

    pix_params pp;
    load_pix_params(params, &pp);
    iir_t iir;
    get_iir(&iir);
    float T[SS2O_EOTF_N + 1];
    ss2o_eotf_table(T);

    const size_t n0 = (size_t)w * h;
    /* lin: 6 planes (ref RGB, dis RGB) at the current scale */
    float *lin = malloc(sizeof(float) * 6 * n0);
    float *nxt = malloc(sizeof(float) * 6 * n0);
    float *xyb = malloc(sizeof(float) * 6 * n0);
    float *prod = malloc(sizeof(float) * NQ * n0);
    float *tmp = malloc(sizeof(float) * n0);
    float *blur = malloc(sizeof(float) * NQ * n0);
    if (!lin || !nxt || !xyb || !prod || !tmp || !blur) {
        free(lin); free(nxt); free(xyb); free(prod); free(tmp); free(blur);
        return -12;
    }
    frame_to_linear(ref, w, h, depth, chroma, T, lin, lin + n0, lin + 2 * n0);
    frame_to_linear(dis, w, h, depth, chroma, T, lin + 3 * n0, lin + 4 * n0,
                    lin + 5 * n0);

    double values[SS2O_NVALUES];
    memset(values, 0, sizeof(values));

    for (int s = 0; s < nscales; ++s) {
        const int sw = ws[s], sh = hs[s];
        const size_t ns = (size_t)sw * sh;
        const int dumping = dump && dump->scale == s;
        if (s > 0) {
            for (int p = 0; p < 6; ++p)
                ss2o_downsample(lin + (size_t)p * (ws[s - 1] * (size_t)hs[s - 1]),
                                ws[s - 1], hs[s - 1], nxt + (size_t)p * ns);
            memcpy(lin, nxt, sizeof(float) * 6 * ns);
        }
        /* planes at this scale are packed with stride ns */
        for (int img = 0; img < 2; ++img) {
            const float *R = lin + (size_t)(3 * img) * ns;
            const float *G = R + ns, *B = G + ns;
            float *X = xyb + (size_t)(3 * img) * ns, *Y = X + ns, *Bo = Y + ns;
            for (size_t i = 0; i < ns; ++i)
                pixel_xyb(&pp, R[i], G[i], B[i], &X[i], &Y[i], &Bo[i]);
        }
        if (dumping && dump->lin) memcpy(dump->lin, lin, sizeof(float) * 6 * ns);
        if (dumping && dump->xyb) memcpy(dump->xyb, xyb, sizeof(float) * 6 * ns);

        for (int c = 0; c < 3; ++c) {
            const float *x1 = xyb + (size_t)c * ns;
            const float *x2 = xyb + (size_t)(3 + c) * ns;
            /* multiply_3plane: the three products, one rounding each */
            memcpy(prod, x1, sizeof(float) * ns);
            memcpy(prod + ns, x2, sizeof(float) * ns);
            for (size_t i = 0; i < ns; ++i) {
                prod[2 * ns + i] = x1[i] * x1[i];
                prod[3 * ns + i] = x2[i] * x2[i];
                prod[4 * ns + i] = x1[i] * x2[i];
            }
            for (int q = 0; q < NQ; ++q) {
                blur_plane(&iir, prod + (size_t)q * ns, sw, sh, tmp,
                           blur + (size_t)q * ns);
                if (dumping && dump->hblur)
                    memcpy(dump->hblur + (size_t)(c * NQ + q) * ns, tmp,
                           sizeof(float) * ns);
            }
            if (dumping && dump->blur)
                memcpy(dump->blur + (size_t)c * NQ * ns, blur,
                       sizeof(float) * NQ * ns);
            const float *mu1 = blur, *mu2 = blur + ns, *s11 = blur + 2 * ns,
                        *s22 = blur + 3 * ns, *s12 = blur + 4 * ns;
            double sum[NSUM] = {0, 0, 0, 0, 0, 0};
            for (size_t i = 0; i < ns; ++i) {
                double d = ssim_term(mu1[i], mu2[i], s11[i], s22[i], s12[i],
                                     pp.c2);
                double r = edge_term(x1[i], mu1[i], x2[i], mu2[i]);
                double art = r > 0.0 ? r : 0.0;
                double det = r < 0.0 ? -r : 0.0;
                double t[NSUM] = {d, pow4(d), art, pow4(art), det, pow4(det)};
                for (int k = 0; k < NSUM; ++k) sum[k] += t[k];
                if (dumping && dump->terms)
                    for (int k = 0; k < NSUM; ++k)
                        dump->terms[(size_t)(c * NSUM + k) * ns + i] = t[k];
            }
            if (dumping && dump->sums)
                for (int k = 0; k < NSUM; ++k) dump->sums[c * NSUM + k] = sum[k];
            /* 1-norm = mean, 4-norm = fourth root of the mean fourth power */
            for (int kind = 0; kind < 3; ++kind) {
                double avg1 = sum[2 * kind] / (double)ns;
                double avg4 = sqrt(sqrt(sum[2 * kind + 1] / (double)ns));
                values[((c * 6 + s) * 2 + 0) * 3 + kind] = avg1;
                values[((c * 6 + s) * 2 + 1) * 3 + kind] = avg4;
            }
        }
    }
    free(lin); free(nxt); free(xyb); free(prod); free(tmp); free(blur);

    /* pool_score: P = sum_i w_i |v_i| in index order, then the map. */
    double P = 0.0;
    for (int i = 0; i < SS2O_NVALUES; ++i) {
        double t = params[SS2O_P_WEIGHTS + i] * fabs(values[i]);
        P = P + t;
    }
    const double *pc = params + SS2O_P_POLY;
    double sc = pc[3] * P;
    sc = sc + pc[2];
    sc = sc * P;
    sc = sc + pc[1];
    sc = sc * P;
    sc = sc + pc[0];
    const double *pw = params + SS2O_P_POWER;
    if (sc > 0.0) {
        double t = pw[1] == 1.0 ? sc : pow(sc, pw[1]);
        t = pw[0] * t;
        sc = t + pw[2];
    }
    if (score_out) *score_out = sc;
    if (values_out) memcpy(values_out, values, sizeof(values));
    return 0;
}

int ss2o_score_frames(const void *ref, const void *dis, int n, int w, int h,
                      int depth, int chroma, const double *params,
                      double *scores, double *values)
{
    size_t fb = ss2o_frame_bytes(w, h, depth, chroma);
    for (int f = 0; f < n; ++f) {
        int rc = ss2o_score((const uint8_t *)ref + fb * f,
                            (const uint8_t *)dis + fb * f, w, h, depth, chroma,
                            params, scores ? scores + f : NULL,
                            values ? values + (size_t)SS2O_NVALUES * f : NULL,
                            NULL);
        if (rc) return rc;
    }
    return 0;
}
