"""The oracle pinned to things other than itself (CPU only).

Each pin comes from the mathematics or from a property the method must have:
closed forms, exact rational arithmetic, brute force on tiny inputs and
invariants.  Together they are meant to fail on any plausible slip in the
oracle: a dropped term, a wrong sign, index or operand, a missed clamp.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

SIGMA = 1.5


def _frame(y, u, v):
    return np.concatenate([np.asarray(p).ravel() for p in (y, u, v)])


def _const_frame(w, h, depth, chroma, Y, U, V):
    cw, ch = synth.chroma_dims(w, h, chroma)
    dt = np.uint8 if depth == 8 else np.uint16
    return _frame(np.full((h, w), Y, dt), np.full((ch, cw), U, dt), np.full((ch, cw), V, dt))


# ---------------------------------------------------------------------------
# 1. identical pair -> exactly 100
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("geom", [(64, 48, 8, 420), (33, 20, 12, 444), (40, 17, 10, 422),
                                  (8, 8, 16, 444)])
def test_identical_pair_scores_exactly_100(geom):
    w, h, d, c = geom
    wl = synth.custom(w, h, d, c, 1, seed=7)
    s, v, _ = oracle.score(wl.ref[0], wl.ref[0], w, h, d, c)
    assert s == 100.0
    assert np.all(v == 0.0)


def test_identical_frame_of_odd_size_workload_scores_100():
    wl = synth.make("c1_853x481_8b_444", [0])
    s, _, _ = oracle.score(wl.ref[0], wl.dis[0], 853, 481, 8, 444)
    assert s == 100.0


# ---------------------------------------------------------------------------
# 2. recursive Gaussian vs the closed-form Gaussian, and vs a direct FIR
# ---------------------------------------------------------------------------

def _impulse(n=41):
    x = np.zeros(n, np.float32)
    x[n // 2] = 1.0
    return oracle.blur_line(x)


def test_blur_impulse_response_is_gaussian_sigma_1_5():
    r = _impulse().astype(np.float64)
    m = np.arange(41) - 20
    g = np.exp(-m * m / (2 * SIGMA ** 2)) / (SIGMA * math.sqrt(2 * math.pi))
    err = np.abs(r - g).max()
    # stated bound: three cosine harmonics on |m| <= 4 fit the sigma = 1.5
    # Gaussian to 3.9e-3 of its peak (least squares with unit sum)
    assert err <= 4e-3 * g.max(), err
    assert abs(r.sum() - 1.0) <= 1e-6
    # symmetric about the impulse, up to fp32 rounding of the recursion
    assert np.abs(r - r[::-1]).max() <= 1e-6
    # support: |m| <= 4 carries the kernel; beyond it only rounding residue
    assert np.abs(r[np.abs(m) > 4]).max() <= 1e-6
    assert np.all(r[np.abs(m) <= 4] > 0)


def test_blur_recursion_matches_direct_fir():
    """Linearity and zero-extended borders: the recursion over a random line
    equals the direct convolution with its own impulse response."""
    taps = _impulse().astype(np.float64)[16:25]      # m = -4..4
    rng = np.random.default_rng(0)
    for n in (3840, 17, 9, 5, 1):
        x = rng.uniform(-1, 1, n).astype(np.float32)
        got = oracle.blur_line(x).astype(np.float64)
        want = np.convolve(x.astype(np.float64), taps, mode="full")[4:4 + n]
        bound = 2e-5 * np.abs(x).sum() / max(1, n) * 9 + 1e-6
        assert np.abs(got - want).max() <= bound, (n, np.abs(got - want).max())


def test_blur_edge_response_is_truncated_kernel():
    """An impulse at the first sample sees only the right half of the kernel."""
    x = np.zeros(20, np.float32)
    x[0] = 1.0
    got = oracle.blur_line(x)
    full = _impulse()
    assert np.abs(got[:5] - full[20:25]).max() <= 1e-6


def test_iir_coefficients_describe_cosine_resonators():
    """2 cos(w_k) for w_k = (2k+1) pi / 10 (zeros at +-5), so the resonator
    frequencies are the ones a radius-4 window needs."""
    a, c2, g = oracle.iir_coeffs()
    for k, wk in enumerate([math.pi / 10, 3 * math.pi / 10, 5 * math.pi / 10]):
        assert abs(float(c2[k]) - 2 * math.cos(wk)) <= 2.5e-7
    assert abs(sum(float(x) for x in a) * 1 - a.sum()) < 1e-15


# ---------------------------------------------------------------------------
# 3. neutral gray -> X = 0
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("depth", [8, 10])
def test_neutral_gray_maps_to_x_zero(depth):
    k = 1 << (depth - 8)
    w, h = 16, 14
    ys = np.linspace(16 * k, 235 * k, w * h).round().astype(np.int64).reshape(h, w)
    cw, ch = synth.chroma_dims(w, h, 420)
    dt = np.uint8 if depth == 8 else np.uint16
    f = _frame(ys.astype(dt), np.full((ch, cw), 128 * k, dt), np.full((ch, cw), 128 * k, dt))
    _, _, d = oracle.score(f, f, w, h, depth, 420, dump_scale=0)
    lin, xyb = d["lin"], d["xyb"]
    assert np.array_equal(lin[0], lin[1]) and np.array_equal(lin[1], lin[2])
    assert np.abs(xyb[0]).max() <= 1e-7
    yv = xyb[1].ravel()
    order = np.argsort(ys.ravel(), kind="stable")
    assert np.all(np.diff(yv[order]) >= 0)


def test_xyb_channels_on_the_primaries():
    """The opsin rows L and M share their blue weight, so pure blue has X = 0;
    red drives L above M (X > 0), green drives M above L (X < 0); black is
    the origin; Y grows with every primary; B - Y is largest for blue."""
    z = oracle.xyb_pixel(0.0, 0.0, 0.0)
    assert np.array_equal(z, np.zeros(3, np.float32))
    r = oracle.xyb_pixel(1.0, 0.0, 0.0)
    g = oracle.xyb_pixel(0.0, 1.0, 0.0)
    b = oracle.xyb_pixel(0.0, 0.0, 1.0)
    assert b[0] == 0.0 and r[0] > 1e-3 and g[0] < -1e-3
    assert r[1] > 0 and g[1] > 0 and b[1] > 0
    assert b[2] > r[2] and b[2] > g[2] and b[2] > 0
    w = oracle.xyb_pixel(1.0, 1.0, 1.0)
    assert abs(w[0]) <= 1e-7 and abs(w[2]) <= 1e-6


def test_bt709_round_trip_of_coloured_pixels():
    """Encode R'G'B' with the forward BT.709 transform (Kr = 0.2126,
    Kb = 0.0722) at 10 bits; the oracle's decoding must return the colour
    (through the EOTF) within the quantisation error."""
    kr, kb = 0.2126, 0.0722
    kg = 1 - kr - kb
    cols = [(0.8, 0.3, 0.5), (0.1, 0.9, 0.2), (0.6, 0.2, 0.95), (0.5, 0.5, 0.1)]
    w, h = 8, 8
    ys, us, vs = [], [], []
    for (R, G, B) in cols:
        Yp = kr * R + kg * G + kb * B
        cb = (B - Yp) / (2 * (1 - kb))
        cr = (R - Yp) / (2 * (1 - kr))
        ys.append(round(64 + 876 * Yp))
        us.append(round(512 + 896 * cb))
        vs.append(round(512 + 896 * cr))
    Y = np.repeat(np.array(ys, np.uint16), 16).reshape(h, w)
    U = np.repeat(np.array(us, np.uint16), 16).reshape(h, w)
    V = np.repeat(np.array(vs, np.uint16), 16).reshape(h, w)
    f = _frame(Y, U, V)
    _, _, d = oracle.score(f, f, w, h, 10, 444, dump_scale=0)
    lin = d["lin"][:3].reshape(3, -1)
    eotf = lambda v: v / 12.92 if v <= 0.04045 else ((v + 0.055) / 1.055) ** 2.4  # noqa: E731
    for i, (R, G, B) in enumerate(cols):
        got = lin[:, 16 * i]
        want = np.array([eotf(R), eotf(G), eotf(B)])
        assert np.abs(got - want).max() <= 4e-3, (i, got, want)


# ---------------------------------------------------------------------------
# 4. 8x8 sums vs exact sums
# ---------------------------------------------------------------------------

def test_8x8_sums_equal_exact_sums():
    wl = synth.custom(8, 8, 8, 444, 1, seed=99, noise=12.0)
    _, v, d = oracle.score(wl.ref[0], wl.dis[0], 8, 8, 8, 444, dump_scale=0)
    terms, sums = d["terms"], d["sums"]
    for j in range(18):
        t = terms[j].ravel()
        exact = math.fsum(t.tolist())
        assert abs(sums[j] - exact) <= 64 * 2.0 ** -53 * np.abs(t).sum(), j
        assert np.all(t >= 0)
    # the values are the 1-norms and 4-norms of these sums
    for c in range(3):
        for kind in range(3):
            s1, s4 = sums[c * 6 + 2 * kind], sums[c * 6 + 2 * kind + 1]
            assert v[((c * 6 + 0) * 2 + 0) * 3 + kind] == s1 / 64.0
            assert v[((c * 6 + 0) * 2 + 1) * 3 + kind] == math.sqrt(math.sqrt(s4 / 64.0))
    # fourth powers are the squares of the squares of the first-power terms
    for c in range(3):
        for kind in range(3):
            t1 = terms[c * 6 + 2 * kind].ravel()
            t4 = terms[c * 6 + 2 * kind + 1].ravel()
            assert np.array_equal(t4, (t1 * t1) * (t1 * t1))
    # artifact and detail-lost are the two signs of one ratio: never both > 0
    for c in range(3):
        art, det = terms[c * 6 + 2], terms[c * 6 + 4]
        assert np.all((art == 0) | (det == 0))
    assert np.any(terms[[2, 8, 14]] > 0) and np.any(terms[[4, 10, 16]] > 0)


def _flat(w, h, Y, U, V):
    cw, ch = synth.chroma_dims(w, h, 444)
    return _const_frame(w, h, 8, 444, Y, U, V)


def test_ssim_term_on_flat_frames_is_the_squared_mean_difference():
    """Two flat frames: away from the borders every window sees one value,
    so both variances and the covariance vanish, num_s = den_s = C2 and the
    SSIM term is 1 - (1 - (x1 - x2)^2) = (x1 - x2)^2 per channel."""
    w = h = 40
    a = _flat(w, h, 60, 100, 170)
    b = _flat(w, h, 180, 150, 90)
    _, _, d = oracle.score(a, b, w, h, 8, 444, dump_scale=0)
    xyb, terms = d["xyb"].astype(np.float64), d["terms"]
    inner = (slice(6, h - 6), slice(6, w - 6))
    for c in range(3):
        x1, x2 = xyb[c][inner].mean(), xyb[3 + c][inner].mean()
        want = (x1 - x2) ** 2
        got = terms[c * 6 + 0][inner]
        # fp32 rounding of the recursions leaves variances of ~1e-7 against
        # C2 = 9e-4, so the term carries ~1e-3 relative noise
        assert np.abs(got - want).max() <= 2e-5 + 2e-2 * want, (c, got.max(), want)
    assert (xyb[1][inner].mean() - xyb[4][inner].mean()) ** 2 > 1e-3


def test_ssim_and_edge_terms_around_an_impulse_pin_c2():
    """One bright luma pixel on a gray reference against the flat gray frame,
    with the affine set so that both frames' XYB planes are exactly zero but
    for the reference's Y value delta at the impulse.  Blurring is linear, so
    with h the pinned 1-D impulse response and H = h(dx) h(dy):
        mu1 = delta H, s11 = delta^2 H, mu2 = s22 = s12 = 0,
        d   = 1 - (1 - delta^2 H^2) C2 / (delta^2 H (1 - H) + C2),
        det = a / (1 + a), a = |x1 - mu1|, art = 0.
    Near the impulse delta^2 H is of the order of C2, so the SSIM term depends
    on C2 at first order: the textbook stabiliser C2 = (K2 L)^2 with K2 = 0.03
    and dynamic range L = 1 must be the default (a value 0.0005 or 0.0015
    moves the terms by over 40%).  Scales 0 and 1 (where the impulse is
    still large against the fp32 rounding of the variances)."""
    w = h = 128
    Yf, dY = 126, 60
    chroma = np.full(w * h, 128, np.uint8)
    luma = np.full((h, w), Yf, np.uint8)
    dis = np.concatenate([luma.ravel(), chroma, chroma])
    luma[64, 64] = Yf + dY
    ref = np.concatenate([luma.ravel(), chroma, chroma])
    p = oracle.default_params()
    _, _, d0 = oracle.score(ref, dis, w, h, 8, 444, p, dump_scale=0)
    y_flat = float(d0["xyb"][4, 0, 0])
    # X' = 0 X + 0, Y' = Y - Y(flat gray), B' = (B - Y) 0 + 0
    p[oracle.P_AFFINE:oracle.P_AFFINE + 5] = [0.0, 0.0, -y_flat, 0.0, 0.0]
    c2 = 0.03 ** 2
    n = 201
    e = np.zeros(n, np.float32)
    e[n // 2] = 1.0
    hl = oracle.blur_line(e).astype(np.float64)
    _, vals, _ = oracle.score(ref, dis, w, h, 8, 444, p)
    vals = vals.reshape(3, 6, 2, 3)
    for s in (0, 1):
        _, _, dump = oracle.score(ref, dis, w, h, 8, 444, p, dump_scale=s)
        xyb = dump["xyb"]
        py = px = 64 >> s
        delta = float(xyb[1, py, px])
        assert delta > 0.05
        rest = xyb.copy()
        rest[1, py, px] = 0.0
        assert not np.any(rest), "the XYB planes must vanish off the impulse"
        sh, sw = xyb.shape[1:]
        hy = hl[n // 2 - py:n // 2 - py + sh]
        hx = hl[n // 2 - px:n // 2 - px + sw]
        H = np.outer(hy, hx)
        dd = delta * delta
        d_want = 1.0 - (1.0 - dd * H * H) * c2 / (dd * H * (1.0 - H) + c2)
        x1 = np.zeros_like(H)
        x1[py, px] = delta
        a = np.abs(x1 - delta * H)
        det_want = a / (1.0 + a)
        supp = (slice(py - 4, py + 5), slice(px - 4, px + 5))
        terms = dump["terms"]
        d_got, art_got, det_got = terms[6], terms[8], terms[10]
        assert np.all(np.abs(d_got - d_want)[supp] <= 1e-4 * d_want[supp]), s
        assert np.all(np.abs(det_got - det_want)[supp] <= 1e-4 * det_want[supp]), s
        assert not np.any(art_got)
        # off the 9x9 support only rounding residue of the recursions is left
        off = np.ones_like(H, bool)
        off[supp] = False
        assert d_got[off].sum() <= 1e-3 and det_got[off].sum() <= 1e-4
        # the pooled 1-norms and 4-norms of the Y channel at this scale
        N = sh * sw
        assert abs(vals[1, s, 0, 0] - d_want[supp].sum() / N) <= 1e-4 * vals[1, s, 0, 0]
        assert abs(vals[1, s, 1, 0] - (np.sum(d_want[supp] ** 4) / N) ** 0.25) \
            <= 1e-4 * vals[1, s, 1, 0]
        assert abs(vals[1, s, 0, 2] - det_want.sum() / N) <= 1e-4 * vals[1, s, 0, 2]
        assert vals[1, s, 0, 1] == 0.0 and vals[1, s, 1, 1] == 0.0
    assert not np.any(vals[0]) and not np.any(vals[2])


def test_edge_terms_tell_lost_detail_from_artifacts():
    """A flat distorted frame against a textured reference loses detail
    (det >> art); a textured distorted frame against a flat reference has
    artifacts (art >> det)."""
    w, h = 48, 40
    tex = synth.custom(w, h, 8, 444, 1, seed=21, noise=0.0).ref[0]
    flat = _flat(w, h, 128, 128, 128)
    _, v1, _ = oracle.score(tex, flat, w, h, 8, 444)
    _, v2, _ = oracle.score(flat, tex, w, h, 8, 444)
    v1, v2 = v1.reshape(3, 6, 2, 3), v2.reshape(3, 6, 2, 3)
    # scale 0, 1-norm: kind 1 = artifact, 2 = detail lost; the flat frame's
    # borders (zero-extended blur) leave some of the other kind in Y
    for c in range(3):
        assert v1[c, 0, 0, 2] > 5 * v1[c, 0, 0, 1], c
        assert v2[c, 0, 0, 1] > 5 * v2[c, 0, 0, 2], c


# ---------------------------------------------------------------------------
# 5. correctly rounded cube root (exact rational arithmetic)
# ---------------------------------------------------------------------------

def _next(f, direction):
    return float(np.nextafter(np.float32(f), np.float32(direction), dtype=np.float32))


def _is_nearest(x: float, y: float) -> bool:
    """y is the float nearest to cbrt(x): x lies strictly between the cubes of
    the midpoints to the neighbouring floats (exact rationals)."""
    X, Y = Fraction(x), Fraction(y)
    up, dn = Fraction(_next(y, np.inf)), Fraction(_next(y, 0.0))
    hi, lo = (Y + up) / 2, (Y + dn) / 2
    return lo ** 3 < X < hi ** 3


def test_cbrt_perfect_cubes_exact():
    rng = np.random.default_rng(1)
    for _ in range(2000):
        m = int(rng.integers(1, 256))                 # 8-bit significand: cube fits 24 bits
        e = int(rng.integers(-12, 4))
        y = math.ldexp(m, e - 8)
        x = y ** 3
        assert float(np.float32(x)) == x
        assert oracle.cbrtf_cr(x) == float(np.float32(y))


def test_cbrt_nearest_on_random_sample():
    rng = np.random.default_rng(2)
    lo = np.float32(0.0037).view(np.uint32)
    hi = np.float32(1.01).view(np.uint32)
    bits = rng.integers(lo, hi, 3000, dtype=np.uint32)
    bits = np.concatenate([bits, rng.integers(1, 0x7f7fffff, 500, dtype=np.uint32)])
    xs = bits.view(np.float32)
    ys = oracle.cbrtf_cr_array(xs, threads=1)
    for x, y in zip(xs.tolist(), ys.tolist()):
        assert _is_nearest(x, y), (x, y)


def test_cbrt_rounding_boundaries():
    """For sampled results y: the first float above the lower midpoint cube
    and the last float below the upper one both give y; the floats just
    outside give the neighbours."""
    rng = np.random.default_rng(3)
    ylo = np.float32(0.155).view(np.uint32)
    yhi = np.float32(1.0).view(np.uint32)
    for yb in rng.integers(ylo, yhi, 400, dtype=np.uint32):
        y = float(yb.view(np.float32))
        Y = Fraction(y)
        hi_mid = ((Y + Fraction(_next(y, np.inf))) / 2) ** 3
        lo_mid = ((Y + Fraction(_next(y, 0.0))) / 2) ** 3
        a = float(np.float32(float(lo_mid)))
        while Fraction(a) <= lo_mid:
            a = _next(a, np.inf)
        b = float(np.float32(float(hi_mid)))
        while Fraction(b) >= hi_mid:
            b = _next(b, 0.0)
        assert oracle.cbrtf_cr(a) == y and oracle.cbrtf_cr(b) == y
        assert oracle.cbrtf_cr(_next(a, 0.0)) == _next(y, 0.0)
        assert oracle.cbrtf_cr(_next(b, np.inf)) == _next(y, np.inf)


# ---------------------------------------------------------------------------
# 6. sRGB EOTF table
# ---------------------------------------------------------------------------

def _srgb_encode(lin: np.ndarray) -> np.ndarray:
    """The sRGB OETF (the inverse of the decoding the table holds)."""
    lin = np.asarray(lin, np.float64)
    return np.where(lin <= 0.0031308, 12.92 * lin, 1.055 * np.power(lin, 1 / 2.4) - 0.055)


def test_eotf_table_inverts_the_oetf():
    T = oracle.eotf_table().astype(np.float64)
    assert T[0] == 0.0 and T[-1] == 1.0
    assert np.all(np.diff(T) > 0)
    grid = np.arange(T.size) / 4096.0
    assert np.abs(_srgb_encode(T) - grid).max() <= 2e-6
    # a published reference point: mid-grey code 0.5 decodes to 0.2140 linear
    assert abs(T[2048] - 0.21404114) <= 1e-7


def test_eotf_interpolation_error_bound():
    v = np.linspace(0, 1, 20001, dtype=np.float32)
    got = np.array([oracle.eotf_lookup(float(x)) for x in v[::20]])
    # decode by inverting the encoder with bisection-free closed form checks
    back = _srgb_encode(got)
    assert np.abs(back - v[::20].astype(np.float64)).max() <= 2e-5


# ---------------------------------------------------------------------------
# 7. YUV decoding special values and bit-depth invariance
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("depth", [8, 9, 10, 11, 12, 16])
def test_limited_range_black_and_white(depth):
    k = 1 << (depth - 8)
    for Y, want in ((16 * k, 0.0), (235 * k, 1.0)):
        f = _const_frame(16, 16, depth, 444, Y, 128 * k, 128 * k)
        _, _, d = oracle.score(f, f, 16, 16, depth, 444, dump_scale=0)
        assert np.all(d["lin"][:3] == want), (depth, Y)


@pytest.mark.parametrize("depth", [9, 10, 11, 12, 16])
def test_bit_depth_scaling_invariance(depth):
    """8-bit samples shifted to a deeper range decode to the same floats:
    (Y - 16) k / (219 k) rounds like (Y - 16) / 219."""
    wl = synth.custom(48, 32, 8, 420, 1, seed=4)
    k = 1 << (depth - 8)
    r16 = (wl.ref[0].astype(np.uint16) * k).astype(np.uint16)
    d16 = (wl.dis[0].astype(np.uint16) * k).astype(np.uint16)
    s8, v8, x8 = oracle.score(wl.ref[0], wl.dis[0], 48, 32, 8, 420, dump_scale=0)
    sd, vd, xd = oracle.score(r16, d16, 48, 32, depth, 420, dump_scale=0)
    assert np.array_equal(x8["xyb"], xd["xyb"])
    assert s8 == sd and np.array_equal(v8, vd)


def test_decoding_matrix_constants():
    """BT.709 with Kr = 0.2126, Kb = 0.0722: pure red/blue chroma reach the
    primaries' published luma shares."""
    k = oracle.yuv_coeffs().astype(np.float64)
    kr, kb = 0.2126, 0.0722
    kg = 1 - kr - kb
    # Y = kr R + kg G + kb B must hold for R' = Y + k0 Cr, G' = Y - k1 Cb - k2 Cr,
    # B' = Y + k3 Cb for every Cb, Cr: the Cb and Cr coefficients of Y vanish.
    assert abs(kg * -k[1] + kb * k[3]) <= 1e-7
    assert abs(kr * k[0] + kg * -k[2]) <= 1e-7
    # and the chroma scales: B' - Y = 2 (1 - Kb) Cb, R' - Y = 2 (1 - Kr) Cr
    assert abs(k[3] - 1.8556) <= 1e-7 and abs(k[0] - 1.5748) <= 1e-7


# ---------------------------------------------------------------------------
# 8. downsample
# ---------------------------------------------------------------------------

def test_downsample_constant_and_brute_force():
    c = np.full((9, 13), 0.3712, np.float32)
    assert np.all(oracle.downsample(c) == np.float32(0.3712))
    rng = np.random.default_rng(5)
    for (h, w) in ((8, 8), (9, 13), (1, 2), (2, 1), (7, 3)):
        p = rng.uniform(0, 1, (h, w)).astype(np.float32)
        got = oracle.downsample(p).astype(np.float64)
        ys = np.minimum(np.arange(2 * ((h + 1) // 2)), h - 1)
        xs = np.minimum(np.arange(2 * ((w + 1) // 2)), w - 1)
        q = p.astype(np.float64)[np.ix_(ys, xs)]
        want = q.reshape((h + 1) // 2, 2, (w + 1) // 2, 2).mean(axis=(1, 3))
        assert np.abs(got - want).max() <= 4 * 2.0 ** -24


def test_scale_stop_rule():
    assert oracle.scale_dims(8, 8) == [(8, 8)]
    assert oracle.scale_dims(17, 17) == [(17, 17), (9, 9)]
    d = oracle.scale_dims(3840, 2160)
    assert len(d) == 6 and d[-1] == (120, 68)
    assert oracle.scale_dims(853, 481)[-1] == (27, 16)
    wl = synth.custom(8, 8, 8, 444, 1, seed=8, noise=10.0)
    _, v, _ = oracle.score(wl.ref[0], wl.dis[0], 8, 8, 8, 444)
    v = v.reshape(3, 6, 2, 3)
    assert np.all(v[:, 1:] == 0) and np.any(v[:, 0] != 0)
    wl = synth.custom(17, 17, 8, 444, 1, seed=8, noise=10.0)
    _, v, _ = oracle.score(wl.ref[0], wl.dis[0], 17, 17, 8, 444)
    v = v.reshape(3, 6, 2, 3)
    assert np.all(v[:, 2:] == 0) and np.any(v[:, 1] != 0)


# ---------------------------------------------------------------------------
# 9. symmetry, pooling order, chroma siting, frame layout
# ---------------------------------------------------------------------------

def test_ssim_values_invariant_under_swap():
    wl = synth.custom(40, 30, 8, 420, 1, seed=6, noise=8.0)
    _, a, _ = oracle.score(wl.ref[0], wl.dis[0], 40, 30, 8, 420)
    _, b, _ = oracle.score(wl.dis[0], wl.ref[0], 40, 30, 8, 420)
    a, b = a.reshape(3, 6, 2, 3), b.reshape(3, 6, 2, 3)
    assert np.array_equal(a[..., 0], b[..., 0])
    assert not np.array_equal(a[..., 1], b[..., 1])


def test_one_hot_weights_recover_each_value():
    wl = synth.custom(24, 20, 8, 444, 1, seed=12, noise=6.0)
    _, v, _ = oracle.score(wl.ref[0], wl.dis[0], 24, 20, 8, 444)
    p = oracle.default_params()
    p[108:112] = [0.0, 1.0, 0.0, 0.0]
    p[112:115] = [1.0, 1.0, 0.0]
    for i in range(108):
        p[0:108] = 0.0
        p[i] = 1.0
        s, _, _ = oracle.score(wl.ref[0], wl.dis[0], 24, 20, 8, 444, p)
        assert s == abs(v[i]), i


def test_polynomial_and_power_map():
    wl = synth.custom(24, 20, 8, 444, 1, seed=12, noise=6.0)
    p = oracle.default_params()
    _, v, _ = oracle.score(wl.ref[0], wl.dis[0], 24, 20, 8, 444, p)
    P = math.fsum(abs(x) / 108.0 for x in v)
    p[108:112] = [50.0, -20.0, 3.0, -0.5]
    p[112:115] = [2.0, 0.5, -1.0]
    s, _, _ = oracle.score(wl.ref[0], wl.dis[0], 24, 20, 8, 444, p)
    poly = 50.0 - 20.0 * P + 3.0 * P * P - 0.5 * P ** 3
    assert abs(s - (2.0 * math.sqrt(poly) - 1.0)) <= 1e-12


@pytest.mark.parametrize("chroma", [420, 422])
def test_subsampled_chroma_equals_replicated_444(chroma):
    """Nearest chroma siting: a subsampled frame scores exactly like the
    4:4:4 frame whose chroma repeats each sample over its footprint."""
    w, h = 36, 22
    wl = synth.custom(w, h, 8, chroma, 1, seed=13, noise=5.0)
    cw, ch = synth.chroma_dims(w, h, chroma)
    sx = 1
    sy = 1 if chroma == 420 else 0

    def up(frame):
        y = frame[:w * h].reshape(h, w)
        u = frame[w * h:w * h + cw * ch].reshape(ch, cw)
        v = frame[w * h + cw * ch:].reshape(ch, cw)
        rep = lambda p: np.repeat(np.repeat(p, 1 << sy, 0), 1 << sx, 1)[:h, :w]  # noqa: E731
        return _frame(y, rep(u), rep(v))

    s1, v1, _ = oracle.score(wl.ref[0], wl.dis[0], w, h, 8, chroma)
    s2, v2, _ = oracle.score(up(wl.ref[0]), up(wl.dis[0]), w, h, 8, 444)
    assert s1 == s2 and np.array_equal(v1, v2)


def test_frame_bytes_and_rejected_geometry():
    assert oracle.frame_bytes(3840, 2160, 8, 420) == 3840 * 2160 * 3 // 2
    assert oracle.frame_bytes(853, 481, 12, 444) == 853 * 481 * 3 * 2
    assert oracle.frame_bytes(17, 13, 10, 420) == (17 * 13 + 2 * 9 * 7) * 2
    for (w, h, d, c) in ((7, 8, 8, 444), (9, 8, 8, 420), (8, 8, 7, 444), (8, 8, 8, 411)):
        f = np.zeros(oracle.frame_bytes(w, h, d, c), np.uint8)
        with pytest.raises(ValueError):
            oracle.score(f, f, w, h, d, c)
