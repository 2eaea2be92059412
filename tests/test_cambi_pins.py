"""The CAMBI c-value and top-K oracle pinned to closed forms (CPU).

"ADR-1357: Run the SYCL CAMBI extractor entirely on the device" (Decision)
fixes the per-pixel value w p0 pm / (p0 + pm), formed as (float)(w p0 pm)
times a reciprocal table, over windows up to 65 x 65, and the exact top-K
sum in units of 2^-24.  These pins hold the oracle to:
  - the reciprocal table: 1/n rounded to nearest fp32, from exact rationals;
  - planes whose window counts follow from geometry alone (a level edge, a
    three-level staircase, a mask), against the formula evaluated here from
    those counts;
  - the top-K sum against exact rational arithmetic on sorted values, with
    ties, and the window limits.
"""
from __future__ import annotations

import fractions
import math

import numpy as np
import pytest

import oracle


def _f32_nearest(q: fractions.Fraction) -> np.float32:
    """The fp32 value nearest to a positive rational (ties to even)."""
    e = math.floor(math.log2(q.numerator) - math.log2(q.denominator))
    while fractions.Fraction(2) ** e > q:
        e -= 1
    while fractions.Fraction(2) ** (e + 1) <= q:
        e += 1
    scale = fractions.Fraction(2) ** (23 - e)
    m = q * scale                       # in [2^23, 2^24)
    lo = math.floor(m)
    r = m - lo
    if r > fractions.Fraction(1, 2) or (r == fractions.Fraction(1, 2) and lo % 2):
        lo += 1
    return np.float32(lo / scale)


def test_reciprocal_table_is_correctly_rounded():
    for n in list(range(1, 300)) + list(range(4100, 4226)):
        assert np.float32(oracle.cambi_recip(n)) == _f32_nearest(fractions.Fraction(1, n)), n


def _term(w, p0, pm):
    return np.float32(np.float32(w * p0 * pm) * np.float32(oracle.cambi_recip(p0 + pm)))


def test_constant_plane_has_no_c_values():
    c = oracle.cambi_cvalues(np.full((40, 50), 321, np.uint16), 9, [1, 2], [1, 2])
    assert np.all(c == 0.0)


@pytest.mark.parametrize("window", [1, 3, 9, 65])
def test_level_edge(window):
    """Left of column e the level is L, right of it L + 2.  A pixel at
    (x, y) < e sees rows ry and columns split at e: p0 = ry (e - x0),
    pm = ry (x1 - e), with the window clipped to the plane."""
    H, W, e, L = 70, 90, 41, 500
    lv = np.full((H, W), L, np.uint16)
    lv[:, e:] = L + 2
    c = oracle.cambi_cvalues(lv, window, [1, 2], [3, 5])
    r = window // 2
    for y in (0, 5, 35, H - 1):
        ry = min(H - 1, y + r) - max(0, y - r) + 1
        for x in range(W):
            x0, x1 = max(0, x - r), min(W - 1, x + r) + 1
            if x >= e:
                want = 0.0                       # level L + 2 sees no L + 3 or L + 4
            else:
                p0, pm = ry * (min(x1, e) - x0), ry * max(0, x1 - e)
                want = _term(5, p0, pm) if pm else 0.0
            assert c[y, x] == want, (y, x, c[y, x], want)


def test_staircase_takes_the_largest_term():
    """Columns of levels L, L + 1, L + 2 in bands of 4; diffs (1, w 1) and
    (2, w 9): the c-value is the larger of the two terms."""
    H, W, L = 12, 12, 100
    lv = np.full((H, W), L, np.uint16)
    lv[:, 4:8] = L + 1
    lv[:, 8:] = L + 2
    c = oracle.cambi_cvalues(lv, 7, [1, 2], [1, 9])
    y, x = 6, 3                       # window rows 3..9 (7), columns 0..6
    p0, p1, p2 = 7 * 4, 7 * 3, 0
    assert c[y, x] == max(_term(1, p0, p1), 0.0)
    y, x = 6, 5                       # columns 2..8: L x2, L+1 x4, L+2 x1
    assert c[y, x] == max(_term(1, 7 * 4, 7), 0.0)      # level L + 1: +1 -> L + 2, +2 -> none
    y, x = 6, 2                       # columns 0..5: L x4, L+1 x2
    assert c[y, x] == _term(1, 28, 14)
    lv2 = np.full((H, W), L, np.uint16)
    lv2[:, 6:] = L + 2
    c2 = oracle.cambi_cvalues(lv2, 7, [1, 2], [1, 9])
    assert c2[6, 4] == _term(9, 7 * 5, 7 * 2)            # columns 1..7: L x5, L+2 x2


def test_mask_removes_pixels_and_counts():
    H, W, L = 30, 30, 7
    lv = np.full((H, W), L, np.uint16)
    lv[:, 15:] = L + 1
    mask = np.ones((H, W), np.uint8)
    mask[:, 15:] = 0                                     # the L + 1 side is not counted
    c = oracle.cambi_cvalues(lv, 9, [1], [1], mask=mask)
    assert np.all(c == 0.0)
    mask2 = np.ones((H, W), np.uint8)
    mask2[10, 12] = 0
    c2 = oracle.cambi_cvalues(lv, 9, [1], [1], mask=mask2)
    assert c2[10, 12] == 0.0
    # pixel (10, 13): columns 9..17 (L x6, L+1 x3) minus the masked (10, 12)
    assert c2[10, 13] == _term(1, 9 * 6 - 1, 9 * 3)


def test_window_and_level_limits():
    lv = np.zeros((70, 70), np.uint16)
    oracle.cambi_cvalues(lv, 65, [1], [1])
    for win in (67, 64, 0):
        with pytest.raises(ValueError):
            oracle.cambi_cvalues(lv, win, [1], [1])
    with pytest.raises(ValueError):
        oracle.cambi_cvalues(np.full((5, 5), 1024, np.uint16), 3, [1], [1])
    with pytest.raises(ValueError):
        oracle.cambi_cvalues(lv, 3, [1], [10])


@pytest.mark.parametrize("k", [1, 7, 500, 4096])
def test_topk_exact_sum_with_ties(k):
    rng = np.random.default_rng(k)
    c = rng.uniform(0.5, 9000.0, 4096).astype(np.float32)  # every fp32 in [0.5, 2^14) is on the 2^-24 grid
    c[::5] = c[3]                                          # many ties
    c[::7] = 0.0
    units = (c.astype(np.float64) * 2 ** 24).astype(np.int64)
    assert np.array_equal(units.astype(np.float64), c.astype(np.float64) * 2 ** 24)
    S, T, mean = oracle.cambi_topk(c, k)
    top = sorted(units.tolist(), reverse=True)[:k]
    assert S == sum(top)
    assert T == np.float32(top[-1] / 2 ** 24)
    assert mean == float(fractions.Fraction(sum(top), k * 2 ** 24))


def test_topk_tie_group_straddling_k():
    """Values 5, 3, 3, 3, 1 with k = 2: T = 3, one value above it, so the
    sum is 5 + 3; the other copies of 3 are not taken."""
    c = np.array([3, 1, 5, 3, 3], np.float32)
    S, T, mean = oracle.cambi_topk(c, 2)
    assert (S, T, mean) == (8 * 2 ** 24, 3.0, 4.0)
    S, T, mean = oracle.cambi_topk(c, 4)
    assert (S, T, mean) == (14 * 2 ** 24, 3.0, 3.5)
