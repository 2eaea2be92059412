"""The MS-SSIM oracle pinned to closed forms (CPU).

The pages ("Research-1363: Device-resident ssimulacra2 and a single-wait
MS-SSIM on SYCL", Findings 6 and 9) name the feature but print no formula;
the oracle restates Wang, Simoncelli and Bovik (2003).  These pins hold it to
results that follow from that definition by a different route:
  - the pyramid against numpy's own edge padding and block means;
  - identical frames, swapped frames, a bit depth change of the same content;
  - flat frames: only the scale-5 luminance term is below 1;
  - a +-a block pattern of block size 2^(k-1) on a flat frame: it survives
    k - 1 halvings, vanishes at scale k + 1, and within a window it has the
    variance a^2 (1 - Q^2), Q its Gaussian-weighted mean pattern, so the
    score is prod_{j<=k} mean(cs_j)^beta_j, with mean(cs_j) counted over the
    window phases (pins beta_1 .. beta_4, the window and the pyramid);
  - a pattern against its negative: the structure term (cov + C3) /
    (s1 s2 + C3) with cov = -s^2 (pins C3 = C2 / 2);
  - with the chroma planes (enable_chroma): the block pattern placed in the
    Cb or the Cr plane alone, at chroma resolution, gives that plane the
    closed-form score and the other two planes exactly 1, at 4:2:0, 4:2:2
    and 4:4:4 (pins each plane's offset, size and order).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

L = 255.0
C1, C2 = (0.01 * L) ** 2, (0.03 * L) ** 2
C3 = C2 / 2
BETA = (0.0448, 0.2856, 0.3001, 0.2363, 0.1333)


def _gauss():
    g = np.exp(-((np.arange(11) - 5.0) ** 2) / (2 * 1.5 ** 2))
    return g / g.sum()


def _frame(Y, depth=8):
    h, w = Y.shape
    dt = np.uint8 if depth == 8 else np.uint16
    mid = 1 << (depth - 1)
    cw, ch = (w + 1) // 2, (h + 1) // 2
    return np.concatenate([Y.astype(dt).ravel(), np.full(2 * cw * ch, mid, dt)])


def test_scale_dims():
    assert oracle.msssim_dims(3840, 2160) == [(3840, 2160), (1920, 1080), (960, 540),
                                              (480, 270), (240, 135)]
    assert oracle.msssim_dims(853, 481) == [(853, 481), (427, 241), (214, 121), (107, 61),
                                            (54, 31)]


@pytest.mark.parametrize("w,h,depth", [(200, 170, 8), (333, 181, 10), (256, 256, 16)])
def test_pyramid_is_the_edge_padded_block_mean(w, h, depth):
    rng = np.random.default_rng(w)
    Y = rng.integers(0, 1 << depth, (h, w))
    lv = oracle.msssim_pyramid(_frame(Y, depth), w, h, depth)
    cur = Y / float(1 << (depth - 8))
    assert np.array_equal(lv[0], cur)
    for j in range(1, 5):
        ph, pw = cur.shape
        p = np.pad(cur, ((0, ph % 2), (0, pw % 2)), mode="edge")
        cur = p.reshape(p.shape[0] // 2, 2, p.shape[1] // 2, 2).mean(axis=(1, 3))
        assert lv[j].shape == cur.shape
        assert np.max(np.abs(lv[j] - cur)) <= 1e-12
        # every level is exact in fp32: a multiple of 2^-(depth - 8) / 4^j below 256
        assert np.array_equal(lv[j].astype(np.float32).astype(np.float64), lv[j])


def test_identical_swapped_and_rescaled():
    rng = np.random.default_rng(7)
    a = rng.integers(0, 256, (180, 200))
    b = np.clip(a + rng.integers(-9, 10, a.shape), 0, 255)
    s, v = oracle.msssim(_frame(a), _frame(a), 200, 180, 8)
    assert s == 1.0 and np.all(v == 1.0)
    s1, v1 = oracle.msssim(_frame(a), _frame(b), 200, 180, 8)
    s2, v2 = oracle.msssim(_frame(b), _frame(a), 200, 180, 8)
    assert abs(s1 - s2) <= 1e-14 and 0.5 < s1 < 1.0
    # the same content at 10 and 16 bits: samples in the 8-bit range, L = 255
    for d in (10, 16):
        k = 1 << (d - 8)
        s3, _ = oracle.msssim(_frame(a * k, d), _frame(b * k, d), 200, 180, d)
        assert abs(s3 - s1) <= 1e-14


@pytest.mark.parametrize("c1,c2", [(40, 200), (128, 131), (0, 255)])
def test_flat_frames(c1, c2):
    s, v = oracle.msssim(_frame(np.full((176, 192), c1)), _frame(np.full((176, 192), c2)),
                         192, 176, 8)
    lum = (2 * c1 * c2 + C1) / (c1 * c1 + c2 * c2 + C1)
    # variances are E[x^2] - mu^2 in fp64: zero up to ~1e-11 at x^2 ~ 4e4
    assert np.allclose(v[:, 0], lum, rtol=0, atol=1e-12)
    assert np.allclose(v[:, 1:4], 1.0, rtol=0, atol=1e-11)
    assert abs(s - lum ** BETA[4]) <= 1e-11


def _pattern(n, b):
    """+1 / -1 in blocks of b samples: q(x) = (-1)^floor(x / b)."""
    return np.where((np.arange(n) // b) % 2 == 0, 1.0, -1.0)


def _mean_cs_of_pattern(W, H, b, a):
    """Mean over the 11x11 windows of cs for a flat frame against
    flat + a qx(x) qy(y): per window Q = (sum g qx)(sum g qy), var = a^2 (1 - Q^2),
    cov = 0, so cs = C2 / (var + C2)."""
    g = _gauss()
    qx, qy = _pattern(W, b), _pattern(H, b)
    Qx = np.array([g @ qx[x:x + 11] for x in range(W - 10)])
    Qy = np.array([g @ qy[y:y + 11] for y in range(H - 10)])
    Q = np.outer(Qy, Qx)
    return np.mean(C2 / (a * a * (1 - Q * Q) + C2))


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_block_pattern_survives_k_scales(k):
    W, H, a, c0 = 352, 192, 20.0, 128.0
    b = 1 << (k - 1)
    Y = c0 + a * np.outer(_pattern(H, b), _pattern(W, b))
    s, v = oracle.msssim(_frame(np.full((H, W), c0)), _frame(Y), W, H, 8)
    want = 1.0
    for j in range(1, k + 1):
        bj = 1 << (k - j)                      # block size at scale j
        mcs = _mean_cs_of_pattern(W >> (j - 1), H >> (j - 1), bj, a)
        assert abs(v[j - 1, 3] - mcs) <= 1e-12, (j, v[j - 1, 3], mcs)
        want *= mcs ** BETA[j - 1]
    assert np.allclose(v[k:, :], 1.0, rtol=0, atol=1e-12)
    assert abs(s - want) <= 1e-12


def test_pattern_against_its_negative():
    """cov = -var, s1 = s2 = s: the structure term (C3 - s^2) / (s^2 + C3),
    contrast 1, cs = (C2 - 2 s^2) / (2 s^2 + C2)."""
    W, H, a, c0 = 352, 192, 2.0, 128.0
    cb = np.outer(_pattern(H, 1), _pattern(W, 1))
    s, v = oracle.msssim(_frame(c0 + a * cb), _frame(c0 - a * cb), W, H, 8)
    g = _gauss()
    P = (g @ _pattern(11, 1)) ** 2
    var = a * a * (1 - P * P)
    assert abs(v[0, 1] - 1.0) <= 1e-12
    assert abs(v[0, 2] - (C3 - var) / (var + C3)) <= 1e-12
    cs = (C2 - 2 * var) / (2 * var + C2)
    assert abs(v[0, 3] - cs) <= 1e-12
    assert abs(s - cs ** BETA[0]) <= 1e-12


def test_smallest_frame():
    f = _frame(np.zeros((161, 161), np.int64))
    assert oracle.msssim(f, f, 161, 161, 8)[0] == 1.0
    g = _frame(np.zeros((160, 161), np.int64))
    with pytest.raises(ValueError):
        oracle.msssim(g, g, 161, 160, 8)


@pytest.mark.parametrize("chroma", [420, 422, 444])
@pytest.mark.parametrize("plane", [1, 2])
def test_chroma_planes_carry_their_own_pattern(chroma, plane):
    W, H, a, c0, k = 704, 384, 20.0, 128.0, 2
    sx, sy = {420: (1, 1), 422: (1, 0), 444: (0, 0)}[chroma]
    cw, ch = (W + sx) >> sx, (H + sy) >> sy
    b = 1 << (k - 1)
    flat_y = np.full(W * H, 100, np.uint8)
    flat_c = np.full(cw * ch, int(c0), np.uint8)
    pat = (c0 + a * np.outer(_pattern(ch, b), _pattern(cw, b))).astype(np.uint8).ravel()
    ref = np.concatenate([flat_y, flat_c, flat_c])
    dis = np.concatenate([flat_y, pat if plane == 1 else flat_c, pat if plane == 2 else flat_c])
    sc, v = oracle.msssim_planes(ref, dis, W, H, 8, chroma)
    want = 1.0
    for j in range(1, k + 1):
        mcs = _mean_cs_of_pattern(cw >> (j - 1), ch >> (j - 1), 1 << (k - j), a)
        assert abs(v[plane, j - 1, 3] - mcs) <= 1e-12, (j, v[plane, j - 1, 3], mcs)
        want *= mcs ** BETA[j - 1]
    assert abs(sc[plane] - want) <= 1e-12 and want < 0.99
    other = 3 - plane
    assert sc[0] == 1.0 and sc[other] == 1.0


def test_identical_chroma_scores_one_with_distorted_luma():
    rng = np.random.default_rng(3)
    W, H = 400, 352
    a = rng.integers(0, 256, W * H + 2 * (W // 2) * (H // 2)).astype(np.uint8)
    b = a.copy()
    b[:W * H] = np.clip(a[:W * H].astype(int) + rng.integers(-20, 21, W * H), 0, 255)
    sc, v = oracle.msssim_planes(a, b, W, H, 8, 420)
    assert sc[0] < 0.99 and sc[1] == 1.0 and sc[2] == 1.0
    assert np.all(v[1:] == 1.0)
    luma, _ = oracle.msssim(a, b, W, H, 8)
    assert sc[0] == luma
