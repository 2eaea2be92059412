"""Planted mistakes in the oracle must fail its pins (CPU).

Each case copies the oracle's sources, plants one plausible slip in one of
them (a dropped term, a wrong sign, index or operand, a missed clamp), builds
the copy with the oracle's own flags and runs that source's pin suite against
it in a child process.  A pin suite that still passes would not have caught
that mistake in the real oracle.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "iir_drops_trailing_tap": ("float s = xa + xb;", "float s = xa;"),
    "iir_recursion_sign": ("float u = fmaf(c->g[k], s, -prev[k]);",
                           "float u = fmaf(c->g[k], s, prev[k]);"),
    "iir_drops_a_harmonic": ("out[(ptrdiff_t)(i + 1) * ostride] = t + cur[2];",
                             "out[(ptrdiff_t)(i + 1) * ostride] = t;"),
    "iir_fit_wrong_sigma": ("const double sigma = 1.5, pi", "const double sigma = 1.4, pi"),
    "edge_ratio_inverted": ("return num / den - 1.0;", "return den / num - 1.0;"),
    "ssim_den_without_c2": ("float den_s = vs + c2;", "float den_s = vs;"),
    "ssim_cov_sign": ("float cov = s12 - m12;", "float cov = s12 + m12;"),
    "fourth_power_is_square": ("double t[NSUM] = {d, pow4(d), art, pow4(art), det, pow4(det)};",
                               "double t[NSUM] = {d, d * d, art, pow4(art), det, pow4(det)};"),
    "chroma_column_uses_row_shift": ("(size_t)(y >> sy) * cw + (size_t)(x >> sx);",
                                     "(size_t)(y >> sy) * cw + (size_t)(x >> sy);"),
    "downsample_wrong_clamp": ("int x0 = 2 * x, x1 = 2 * x + 1 < w ? 2 * x + 1 : w - 1;",
                               "int x0 = 2 * x, x1 = 2 * x + 1 < w ? 2 * x + 1 : w - 2;"),
    "xyb_x_uses_s_cone": ("float x = 0.5f * (c[0] - c[1]);", "float x = 0.5f * (c[0] - c[2]);"),
    "eotf_no_interpolation": ("return fmaf(f, slope, T[i]);", "return T[i];"),
    "chroma_offset_16": ("float cb = (float)(Us - 128 * k) / dc;",
                         "float cb = (float)(Us - 16 * k) / dc;"),
    "matrix_red_from_cb": ("float r = fmaf(c[0], cr, yn);", "float r = fmaf(c[0], cb, yn);"),
    "cbrt_not_correctly_rounded": ("float y = (float)cbrt((double)x);",
                                   "return cbrtf(x);\n    float y = (float)cbrt((double)x);"),
    "avg4_square_root_once": ("double avg4 = sqrt(sqrt(sum[2 * kind + 1] / (double)ns));",
                              "double avg4 = sqrt(sum[2 * kind + 1] / (double)ns);"),
    "pool_weight_misindexed": ("double t = params[SS2O_P_WEIGHTS + i] * fabs(values[i]);",
                               "double t = params[SS2O_P_WEIGHTS + (i + 1) % 108] * fabs(values[i]);"),
    "scale_stop_at_9": ("while (n < SS2O_NSCALES && w >= 8 && h >= 8) {",
                        "while (n < SS2O_NSCALES && w >= 9 && h >= 9) {"),
    "norm_limited_range_219_as_220": ("const float dy = (float)(219 * k), dc = (float)(224 * k);",
                                      "const float dy = (float)(220 * k), dc = (float)(224 * k);"),
    "default_c2_0_003": ("p[SS2O_P_C2] = 0.0009;", "p[SS2O_P_C2] = 0.003;"),
    "default_c2_0_0005": ("p[SS2O_P_C2] = 0.0009;", "p[SS2O_P_C2] = 0.0005;"),
    "default_c2_0_0015": ("p[SS2O_P_C2] = 0.0009;", "p[SS2O_P_C2] = 0.0015;"),
}


# Planted slips in the float_ssim oracle, caught by tests/test_fssim_pins.py.
FSSIM_MUTATIONS = {
    "fssim_scale_truncates": ("int s = (int)lround((double)m / 256.0);",
                              "int s = (int)((double)m / 256.0);"),
    "fssim_window_not_centred": ("const int lo = -(s / 2), hi = s - 1 - s / 2;",
                                 "const int lo = 0, hi = s - 1;"),
    "fssim_mirror_without_edge_repeat": ("if (i < 0) i = -1 - i;", "if (i < 0) i = -i;"),
    "fssim_tap_in_double": ("float tap = sample8(f, w, xx, yy, bps, norm) * wt;",
                            "double tap = (double)sample8(f, w, xx, yy, bps, norm) / (s * s);"),
    "fssim_c2_with_k1": ("C2 = (0.03 * L) * (0.03 * L);", "C2 = (0.01 * L) * (0.01 * L);"),
    "fssim_cov_sign": ("cv = s12 - m1 * m2;", "cv = s12 + m1 * m2;"),
    "fssim_window_sigma": ("g[i] = exp(-t * t / (2.0 * 1.5 * 1.5));",
                           "g[i] = exp(-t * t / (2.0 * 1.0 * 1.0));"),
    "fssim_raw_samples_above_8_bits": ("const float norm = 1.0f / (float)(1 << (depth - 8));",
                                       "const float norm = 1.0f;"),
    "fssim_dynamic_range_256": ("*score = ssim_planes(a, b, wd, hd, 255.0);",
                                "*score = ssim_planes(a, b, wd, hd, 256.0);"),
    "fssim_drops_last_window_row": ("for (int y = 0; y + WIN <= h; ++y) {",
                                    "for (int y = 0; y + WIN < h; ++y) {"),
}

# Planted slips in the MS-SSIM oracle, caught by tests/test_msssim_pins.py.
MSSSIM_MUTATIONS = {
    "msssim_betas_swapped": ("{0.0448, 0.2856, 0.3001, 0.2363, 0.1333}",
                             "{0.2856, 0.0448, 0.3001, 0.2363, 0.1333}"),
    "msssim_beta4_as_beta3": ("{0.0448, 0.2856, 0.3001, 0.2363, 0.1333}",
                              "{0.0448, 0.2856, 0.3001, 0.3001, 0.1333}"),
    "msssim_subsample_without_average": (
        "out[(size_t)y * wo + x] = (in[(size_t)y0 * w + x0] + in[(size_t)y0 * w + x1] +",
        "out[(size_t)y * wo + x] = 4.0 * in[(size_t)y0 * w + x0] / 4.0 + 0.0 * (in[(size_t)y0 * w + x1] +"),
    "msssim_edge_clamp_off_by_one": ("const int x0 = 2 * x, x1 = 2 * x + 1 < w ? 2 * x + 1 : w - 1;",
                                     "const int x0 = 2 * x, x1 = 2 * x + 1 < w ? 2 * x + 1 : w - 2;"),
    "msssim_c3_equals_c2": ("C3 = C2 / 2.0;", "C3 = C2;"),
    "msssim_last_scale_cs_only": ("ms *= pow(m[NSCALE - 1][4], kBeta[NSCALE - 1]);",
                                  "ms *= pow(m[NSCALE - 1][3], kBeta[NSCALE - 1]);"),
    "msssim_contrast_without_root": ("const double c = (2.0 * sd1 * sd2 + C2) / (v1 + v2 + C2);",
                                     "const double c = (2.0 * v1 * v2 + C2) / (v1 + v2 + C2);"),
    "msssim_no_depth_normalisation": ("const double norm = 1.0 / (double)(1 << (depth - 8));",
                                      "const double norm = 1.0;"),
    "msssim_product_skips_scale_4": ("for (int j = 0; j < NSCALE - 1; ++j) ms *= pow(m[j][3], kBeta[j]);",
                                     "for (int j = 0; j < NSCALE - 2; ++j) ms *= pow(m[j][3], kBeta[j]);"),
    "msssim_cr_reads_cb": ("(size_t)w * h + (size_t)(p - 1) * cw * ch;",
                           "(size_t)w * h + (size_t)0 * cw * ch;"),
    "msssim_chroma_width_uses_sy": ("const int cw = (w + sx) >> sx, ch = (h + sy) >> sy;",
                                    "const int cw = (w + sy) >> sy, ch = (h + sy) >> sy;"),
}

# Planted slips in the CAMBI oracle, caught by tests/test_cambi_pins.py.
CAMBI_MUTATIONS = {
    "cambi_window_radius_short": ("const int r = window / 2;", "const int r = window / 2 - 1;"),
    "cambi_diff_downwards": ("if (v == L + diffs[i]) ++pm[i];", "if (v == L - diffs[i]) ++pm[i];"),
    "cambi_weight_ignored": ("const long num = (long)weights[i] * p0 * pm[i];",
                             "const long num = (long)p0 * pm[i];"),
    "cambi_reciprocal_off_by_one": ("ss2o_cambi_recip((int)(p0 + pm[i]));",
                                    "ss2o_cambi_recip((int)(p0 + pm[i] + 1));"),
    "cambi_mask_not_applied_to_counts": ("if (mask && !mask[j]) continue;", "(void)j;"),
    "cambi_ties_counted_as_above": ("if (c[i] > T) {", "if (c[i] >= T) {"),
    "cambi_recip_in_double": ("return 1.0f / (float)n;   /* IEEE division: correctly rounded */",
                              "return (float)(1.0 / (double)n + 1e-12);"),
}

CASES = {**{n: ("ss2_oracle.c", "test_oracle_pins.py") for n in MUTATIONS},
         **{n: ("cambi_oracle.c", "test_cambi_pins.py") for n in CAMBI_MUTATIONS},
         **{n: ("fssim_oracle.c", "test_fssim_pins.py") for n in FSSIM_MUTATIONS},
         **{n: ("msssim_oracle.c", "test_msssim_pins.py") for n in MSSSIM_MUTATIONS}}


@pytest.mark.parametrize("name", sorted(CASES))
def test_planted_mistake_fails_the_pins(name, tmp_path):
    target, pins = CASES[name]
    old, new = {**MUTATIONS, **FSSIM_MUTATIONS, **MSSSIM_MUTATIONS, **CAMBI_MUTATIONS}[name]
    srcs = []
    for path in oracle.SOURCES:
        text = open(path).read()
        if os.path.basename(path) == target:
            assert text.count(old) == 1, f"mutation site not found exactly once: {old!r}"
            text = text.replace(old, new)
        dst = tmp_path / os.path.basename(path)
        dst.write_text(text)
        srcs.append(str(dst))
    (tmp_path / "ss2_oracle.h").write_text(open(os.path.join(oracle.HERE, "ss2_oracle.h")).read())
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-shared", "-o", str(so), *srcs, "-lm"], check=True)
    env = dict(os.environ, **{oracle.SO_OVERRIDE_ENV: str(so)})
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", pins)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"the pins did not catch '{name}':\n{r.stdout[-2000:]}"
