"""The float_ssim oracle pinned to the page and to closed forms (CPU).

Decimation: the factors printed on "ADR-1405: float_ssim_hip decimates on
the device, bit-identical to the CPU" (Context); the window sum against
exact integer arithmetic in the page's 2^-52 units (Decision 1) with numpy's
own symmetric padding; a constant plane.  SSIM: identity, symmetry, two flat
frames, and one bright pixel on a flat frame, each in closed form from the
definition (Wang et al. 2004) and an 11-tap sigma-1.5 Gaussian written out
here.  Samples are in the 8-bit range (raw / 2^(depth - 8)) with L = 255.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
K1, K2 = 0.01, 0.03


def _luma_frame(Y, chroma=444, depth=8):
    h, w = Y.shape
    cw, ch = (w, h) if chroma == 444 else ((w + 1) // 2, (h + 1) // 2)
    dt = np.uint8 if depth == 8 else np.uint16
    mid = 1 << (depth - 1)
    return np.concatenate([Y.astype(dt).ravel(), np.full(2 * cw * ch, mid, dt)])


def test_factors_printed_on_the_page():
    rows = [tuple(map(int, ln.split())) for ln in open(os.path.join(HERE, "golden",
            "fssim_scale_factors.txt")) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 4
    for w, h, f in rows:
        assert oracle.fssim_scale(w, h) == f, (w, h)


def test_factor_is_rounded_not_truncated():
    """The printed formula rounds min(w, h) / 256 to the nearest integer."""
    assert [oracle.fssim_scale(700, 900), oracle.fssim_scale(900, 700)] == [3, 3]   # 2.73
    assert oracle.fssim_scale(1000, 4000) == 4                                     # 3.91
    assert oracle.fssim_scale(1100, 1100) == 4                                     # 4.30


def _f32_of_units(units: int, k: int) -> np.float32:
    """units * 2^-k rounded once to fp32 (nearest, ties to even)."""
    if units == 0:
        return np.float32(0.0)
    shift = units.bit_length() - 24
    if shift > 0:
        q, r = divmod(units, 1 << shift)
        half = 1 << (shift - 1)
        if r > half or (r == half and q & 1):
            q += 1
        return np.float32(math.ldexp(q, shift - k))      # q <= 2^24: exact
    return np.float32(math.ldexp(units, -k))


@pytest.mark.parametrize("size,depth", [(512, 8), (768, 8), (1280, 16), (853, 10), (700, 12)])
def test_decimation_is_the_exact_window_sum(size, depth):
    """Every output is the sum of the fp32 taps sample * RN(1/s^2) over the
    s x s window at (x s, y s) with offsets -s/2 .. s-1-s/2 and symmetric
    edges, sample = raw / 2^(depth - 8), counted exactly in 2^-52 units
    (Python integers) and rounded once to float."""
    w, h = size, size - 3 if size == 853 else size
    rng = np.random.default_rng(size)
    Y = rng.integers(0, 1 << depth, (h, w))
    s, wd, hd = oracle.fssim_dims(w, h)
    assert s >= 2
    got = oracle.fssim_decimate(_luma_frame(Y, depth=depth), w, h, depth)
    assert got.shape == (hd, wd) and wd == -(-w // s) and hd == -(-h // s)
    wt = np.float32(1.0) / np.float32(s * s)
    norm = np.float32(2.0 ** (8 - depth))
    lo = s // 2
    pad = np.pad(Y, ((lo, 2 * s), (lo, 2 * s)), mode="symmetric")
    pts = [(0, 0), (0, wd - 1), (hd - 1, 0), (hd - 1, wd - 1)]
    pts += [(int(a), int(b)) for a, b in zip(rng.integers(0, hd, 200), rng.integers(0, wd, 200))]
    for (y, x) in pts:
        win = pad[y * s:y * s + s, x * s:x * s + s].astype(np.float32) * norm   # exact
        taps = (win * wt).astype(np.float32)            # one fp32 product per tap
        tl = [float(t) * 2.0 ** 52 for t in taps.ravel().tolist()]
        assert all(t.is_integer() and t < 2.0 ** 61 for t in tl)   # 2^-52 units fit int64
        want = _f32_of_units(sum(int(t) for t in tl), 52)
        assert got[y, x] == want, (y, x, got[y, x], want)


def test_decimating_a_constant_plane_at_a_power_of_two():
    Y = np.full((1024, 1024), 77)
    s, wd, hd = oracle.fssim_dims(1024, 1024)
    assert s == 4
    assert np.all(oracle.fssim_decimate(_luma_frame(Y), 1024, 1024, 8) == 77.0)


def _gauss():
    g = np.exp(-((np.arange(11) - 5.0) ** 2) / (2 * 1.5 ** 2))
    return g / g.sum()


def test_identical_and_swapped_pairs():
    rng = np.random.default_rng(3)
    a = _luma_frame(rng.integers(0, 256, (60, 80)))
    b = _luma_frame(rng.integers(0, 256, (60, 80)))
    assert oracle.fssim(a, a, 80, 60, 8)[0] == 1.0
    # symmetric up to the order of two fp64 additions
    assert abs(oracle.fssim(a, b, 80, 60, 8)[0] - oracle.fssim(b, a, 80, 60, 8)[0]) <= 1e-15


@pytest.mark.parametrize("depth", [8, 10, 16])
def test_two_flat_frames(depth):
    """Means c1, c2 in the 8-bit range, no variance: SSIM is the luminance
    term (2 c1 c2 + C1) / (c1^2 + c2^2 + C1), C1 = (0.01 * 255)^2."""
    L = 255.0
    C1 = (K1 * L) ** 2
    k = 1 << (depth - 8)
    for r1, r2 in ((40 * k, 200 * k + 1), (128 * k, 130 * k), (0, 255 * k + k - 1)):
        a = _luma_frame(np.full((48, 64), r1), depth=depth)
        b = _luma_frame(np.full((48, 64), r2), depth=depth)
        c1, c2 = r1 / k, r2 / k
        want = (2 * c1 * c2 + C1) / (c1 * c1 + c2 * c2 + C1)
        assert abs(oracle.fssim(a, b, 64, 48, depth)[0] - want) <= 1e-12


def test_one_bright_pixel_on_a_flat_frame():
    """Windows holding the pixel at tap (i, j) see weight w = g_i g_j:
    mu1 = c, mu2 = c + w d, var2 = w (1 - w) d^2, var1 = cov = 0."""
    c, d, W, H = 100.0, 60.0, 40, 36
    L = 255.0
    C1, C2 = (K1 * L) ** 2, (K2 * L) ** 2
    Y = np.full((H, W), int(c))
    Y[17, 19] += int(d)
    s, _, _ = oracle.fssim(_luma_frame(np.full((H, W), int(c))), _luma_frame(Y), W, H, 8)
    g = _gauss()
    n_valid = (W - 10) * (H - 10)
    total = n_valid - 121.0
    for i in range(11):
        for j in range(11):
            w = g[i] * g[j]
            mu2 = c + w * d
            num = (2 * c * mu2 + C1) * C2
            den = (c * c + mu2 * mu2 + C1) * (w * (1 - w) * d * d + C2)
            total += num / den
    assert abs(s - total / n_valid) <= 1e-12


def test_planes_below_the_window_are_refused():
    f = _luma_frame(np.zeros((10, 10), np.int64))
    with pytest.raises(ValueError):
        oracle.fssim(f, f, 10, 10, 8)
    assert math.isfinite(oracle.fssim(_luma_frame(np.zeros((11, 11), np.int64)),
                                      _luma_frame(np.zeros((11, 11), np.int64)), 11, 11, 8)[0])
