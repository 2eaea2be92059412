/*
 * ss2_oracle.h — plain, slow, single-threaded CPU reference of the per-frame
 * SSIMULACRA2 scoring pipeline.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this code.  The CUDA library never
 * links, includes or calls it, and it shares no code with the CUDA library.
 *
 * Source of the method: "Research-1363: Device-resident ssimulacra2 and a
 * single-wait MS-SSIM on SYCL" (vmafx documentation), sections "Sources"
 * (the list of CPU pipeline steps) and "Findings" 2-4 (contraction-off fp32
 * pipeline, fp64 per-pixel terms summed in sequential order, six sums per
 * channel).  Where the page is silent the plainest reading is taken; every
 * such reading is listed in the repository's design notes and restated at
 * the function that takes it.
 *
 * Parity pins: every function here is pinned by a CPU test against something
 * other than itself (closed forms, exact integer arithmetic, brute force,
 * invariants); the one exception is the absolute SSIMULACRA2 score scale,
 * which depends on tuned constants the pages do not give — parity unpinned
 * for the absolute score values (GPU-vs-oracle parity does not depend on them).
 *
 * Build: any C99 compiler with contraction OFF (-ffp-contract=off), no
 * fast-math.  Products are kept in named temporaries so each rounding is the
 * one written.
 */
#ifndef SS2_ORACLE_H
#define SS2_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Parameter vector layout (doubles).  Values used in the fp32 pipeline are
 * rounded to float once, at the start of a call.                            */
#define SS2O_P_WEIGHTS 0    /* 108 pooling weights, index ((c*6+s)*2+n)*3+k */
#define SS2O_P_POLY 108     /* p0..p3: score = p0 + p1 P + p2 P^2 + p3 P^3  */
#define SS2O_P_POWER 112    /* alpha, beta, gamma: s > 0 -> alpha s^beta + gamma */
#define SS2O_P_OPSIN 115    /* 3x3 opsin mixing matrix, row-major            */
#define SS2O_P_BIAS 124     /* 3 opsin biases                                */
#define SS2O_P_AFFINE 127   /* sx, ox, oy, sb, ob                            */
#define SS2O_P_C2 132       /* SSIM stabiliser C2                            */
#define SS2O_NPARAMS 133

#define SS2O_NVALUES 108
#define SS2O_NSCALES 6
#define SS2O_EOTF_N 4096    /* table has SS2O_EOTF_N + 1 entries            */
#define SS2O_IIR_R 4        /* kernel support |m| <= R; zeros at +-(R+1)    */

/* Optional stage dump of one scale (any pointer may be NULL).               */
typedef struct {
    int scale;      /* scale to dump; a scale that is not computed dumps nothing */
    float *lin;     /* 6 planes w_s*h_s: ref R,G,B then dis R,G,B (linear)   */
    float *xyb;     /* 6 planes: ref X,Y,B then dis X,Y,B (after the affine) */
    float *hblur;   /* 15 planes: per channel c, (mu1, mu2, s11, s22, s12)
                       after the horizontal pass only                         */
    float *blur;    /* 15 planes, same order, after both passes              */
    double *terms;  /* 18 planes: per channel, d, d^4, art, art^4, det, det^4 */
    double *sums;   /* 18 sequential sums, same order                        */
} ss2o_dump;

/* Writes the default parameter vector (placeholders for the tuned pooling
 * weights, map and make-positive affine; see the header of the .c file).   */
void ss2o_default_params(double *params);

/* Scores one frame pair.  ref/dis: one packed planar frame each
 * (Y, then U, then V; uint8 for depth 8, little-endian uint16 otherwise).
 * values (108 doubles) and dump may be NULL.  Returns 0, or -22 (EINVAL)
 * for a geometry the pipeline rejects.                                       */
int ss2o_score(const void *ref, const void *dis, int width, int height,
               int bitdepth, int chroma, const double *params,
               double *score, double *values, const ss2o_dump *dump);

/* Scores n packed frames (each frame_bytes long) one after another.         */
int ss2o_score_frames(const void *ref, const void *dis, int n_frames,
                      int width, int height, int bitdepth, int chroma,
                      const double *params, double *scores, double *values);

/* Building blocks, exported for the pins. */
size_t ss2o_frame_bytes(int width, int height, int bitdepth, int chroma);
int ss2o_scale_dims(int width, int height, int *ws, int *hs); /* -> #scales */
float ss2o_cbrtf_cr(float x);
void ss2o_cbrtf_cr_array(const float *x, float *y, long long n);
void ss2o_eotf_table(float *table);            /* SS2O_EOTF_N + 1 floats */
float ss2o_eotf_lookup(const float *table, float v);
void ss2o_yuv_coeffs(float *coeffs);           /* cr_r, cb_g, cr_g, cb_b */
void ss2o_xyb_pixel(const double *params, float r, float g, float b,
                    float *xyb);                /* linear RGB -> X, Y, B */
void ss2o_iir_coeffs(double *a, float *c2, float *g); /* 3 each */
void ss2o_blur_line(const float *in, int n, float *out);
void ss2o_downsample(const float *in, int w, int h, float *out);

/* float_ssim with decimation (fssim_oracle.c): factor, decimated dims,
 * one decimated luma plane (frame = packed YUV, luma first; samples in the
 * 8-bit range, raw / 2^(depth - 8)), and the score of a pair (dec_ref /
 * dec_dis may be NULL).  -22 bad arguments, -95 a decimated plane below
 * 11x11 or a factor above 128.                                             */
int ss2o_fssim_scale(int width, int height);
int ss2o_fssim_dims(int width, int height, int *wd, int *hd); /* -> factor */
int ss2o_fssim_decimate(const void *frame, int width, int height, int bitdepth,
                        float *out);
int ss2o_fssim(const void *ref, const void *dis, int width, int height,
               int bitdepth, double *score, float *dec_ref, float *dec_dis);

/* MS-SSIM of the luma plane (msssim_oracle.c): per-scale dims (w, h pairs,
 * 5 scales), the 5-level pyramid of one frame (levels concatenated, fp64,
 * samples in the 8-bit range), and the score of a pair with the per-scale
 * means values[5][5] = (l, c, s, cs, l cs) per scale (may be NULL).
 * -22 bad arguments, -95 a scale-5 plane below 11x11.                      */
/* CAMBI c-values and top-K pool (cambi_oracle.c).  levels: w x h 10-bit
 * levels (< 1024); mask: w x h bytes, nonzero = counted, or NULL; window
 * odd with window^2 <= 4225; ndiff 1..4 (d >= 1, w in 1..9); out: w x h
 * floats.  topk: the exact top-k sum of c in units of 2^-24 (128 bits as
 * lo, hi), the k-th largest value and the mean.  -22 bad arguments.       */
float ss2o_cambi_recip(int n);
int ss2o_cambi_cvalues(const uint16_t *levels, const uint8_t *mask, int w, int h,
                       int window, int ndiff, const int *diffs, const int *weights,
                       float *out);
int ss2o_cambi_cvalue_at(const uint16_t *levels, const uint8_t *mask, int w, int h,
                         int window, int ndiff, const int *diffs, const int *weights,
                         int x, int y, float *out);
int ss2o_cambi_topk(const float *c, long n, long k, uint64_t *sum_lo,
                    uint64_t *sum_hi, float *threshold, double *mean);

void ss2o_msssim_dims(int width, int height, int *dims);
size_t ss2o_msssim_pyramid_len(int width, int height);
int ss2o_msssim_pyramid(const void *frame, int width, int height, int bitdepth,
                        double *levels);
int ss2o_msssim(const void *ref, const void *dis, int width, int height,
                int bitdepth, double *score, double *values);
/* MS-SSIM per plane of a packed frame pair (Y, then Cb and Cr at chroma
 * resolution when nplanes = 3): scores[nplanes], values[nplanes][5][5]. */
int ss2o_msssim_planes(const void *ref, const void *dis, int width, int height,
                       int bitdepth, int chroma, int nplanes, double *scores,
                       double *values);

#ifdef __cplusplus
}
#endif
#endif
