"""CAMBI c-values and top-K pooling on the device vs the oracle (GPU).

Bars: c-values bitwise (exact integer window counts, then the same single
fp32 product per term); top-K sums bitwise (exact integers in units of
2^-24) with the same threshold; means within 1e-15 relative (two fp64
roundings on the device, one long-double division in the oracle).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


def _levels(h, w, seed, base=300, spread=6):
    """Banded 10-bit levels: slow ramps quantised to steps of 1, plus a
    little integer noise, so windows hold levels L .. L + 4."""
    rng = np.random.default_rng(seed)
    yy, xx = np.mgrid[0:h, 0:w]
    ramp = base + spread * (np.sin(xx / 37.0 + seed) + np.cos(yy / 23.0)) * 2
    lv = np.floor(ramp) + rng.integers(0, 2, (h, w))
    return np.clip(lv, 0, 1023).astype(np.uint16)


CASES = [  # (h, w, window, diffs, weights, masked)
    (61, 97, 9, [1], [1], False),
    (61, 97, 1, [1, 2], [1, 2], False),
    # windows around the lane-group size (cores of 0, 2, 4 and 8 columns
    # with groups of four lanes)
    (37, 45, 3, [1], [2], False),
    (44, 58, 5, [1, 3], [1, 1], True),
    (50, 70, 7, [1, 2], [3, 1], True),
    (47, 83, 11, [1, 4], [2, 2], False),
    (128, 256, 33, [1, 2, 3, 4], [1, 2, 3, 4], True),
    (270, 480, 65, [1, 3], [2, 9], False),
    (40, 33, 65, [2], [5], True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[1]}x{c[0]}w{c[2]}")
def test_cvalues_and_topk_bitwise(cuda, case):
    import torch

    from ssimulacra2_image_scoring_gb300 import Cambi
    h, w, win, d, wt, masked = case
    lv = np.stack([_levels(h, w, s) for s in range(3)])
    mask = None
    if masked:
        mask = (np.random.default_rng(9).random((3, h, w)) > 0.2).astype(np.uint8)
    with Cambi(w, h, win, d, wt, batch=2) as cb:
        dl = torch.from_numpy(np.ascontiguousarray(lv)).cuda()
        dm = None if mask is None else torch.from_numpy(mask).cuda()
        cv = cb.cvalues(dl, dm).cpu().numpy()
        for k in (1, (h * w) // 3, h * w):
            sums, thr, means = cb.topk(torch.from_numpy(cv).cuda(), k)
            psums, pthr, pmeans = cb.pool(dl, k, dm)
            for f in range(3):
                S, T, mean = oracle.cambi_topk(cv[f], k)
                assert sums[f] == S and thr[f] == T
                assert abs(means[f] - mean) <= 1e-15 * max(1.0, abs(mean))
                assert psums[f] == S and pthr[f] == T
    for f in range(3):
        want = oracle.cambi_cvalues(lv[f], win, d, wt, None if mask is None else mask[f])
        assert np.array_equal(cv[f].view(np.uint32), want.view(np.uint32)), f
        assert np.any(want > 0) == (win > 1)      # a 1x1 window holds only the pixel


def test_cvalues_4k_sampled(cuda):
    """A 3840x2160 plane with the largest window: the pixels of the four
    corners, the edges and a random sample, one by one in the oracle; the
    top-K pool against the oracle over the whole plane."""
    import torch

    from ssimulacra2_image_scoring_gb300 import Cambi
    h, w = 2160, 3840
    lv = _levels(h, w, 4)
    d, wt = [1, 2, 3, 4], [1, 2, 3, 4]
    with Cambi(w, h, 65, d, wt) as cb:
        cv = cb.cvalues(torch.from_numpy(np.ascontiguousarray(lv[None])).cuda())
        cv = cv.cpu().numpy()[0]
        k = (h * w) // 4
        sums, thr, means = cb.topk(torch.from_numpy(np.ascontiguousarray(cv[None])).cuda(), k)
    rng = np.random.default_rng(1)
    pts = [(0, 0), (0, w - 1), (h - 1, 0), (h - 1, w - 1), (31, 33), (h - 33, w - 32)]
    pts += [(int(a), int(b)) for a, b in zip(rng.integers(0, h, 60), rng.integers(0, w, 60))]
    want = oracle.cambi_cvalue_at(lv, 65, d, wt, pts)
    got = np.array([cv[y, x] for (y, x) in pts], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    S, T, mean = oracle.cambi_topk(cv, k)
    assert sums[0] == S and thr[0] == T


def test_errors(cuda):
    import torch

    from ssimulacra2_image_scoring_gb300 import Cambi, SS2Error
    with pytest.raises(SS2Error) as e:
        Cambi(64, 64, 67, [1], [1])
    assert e.value.code == -22
    with pytest.raises(SS2Error):
        Cambi(64, 64, 9, [1], [10])
    with Cambi(64, 48, 9, [1], [1]) as cb:
        bad = torch.from_numpy(np.full((1, 48, 64), 1024, np.uint16)).cuda()
        with pytest.raises(SS2Error) as e:
            cb.cvalues(bad)
        assert e.value.code == -22
        off = torch.full((1, 48, 64), 0.1, dtype=torch.float32).cuda()   # 0.1f is off the 2^-24 grid
        with pytest.raises(SS2Error) as e:
            cb.topk(off, 5)
        assert e.value.code == -22
        ok = torch.from_numpy(np.zeros((1, 48, 64), np.uint16)).cuda()
        sums, thr, means = cb.pool(ok, 10)                 # the context stays usable
        assert sums == [0] and thr[0] == 0.0 and means[0] == 0.0


def test_wide_and_narrow_level_sets_in_one_call(cuda):
    """Planes with more than 256 distinct levels take the 1024-bin kernel and
    the others the compact one; one call may hold both."""
    import torch

    from ssimulacra2_image_scoring_gb300 import Cambi
    h, w, win, d, wt = 90, 150, 17, [1, 2], [1, 3]
    wide = _levels(h, w, 1, base=512, spread=120)
    narrow = _levels(h, w, 2)
    assert len(np.unique(wide)) > 256 and len(np.unique(narrow)) <= 256
    lv = np.ascontiguousarray(np.stack([wide, narrow, wide]))
    with Cambi(w, h, win, d, wt) as cb:
        cv = cb.cvalues(torch.from_numpy(lv).cuda()).cpu().numpy()
    for f in range(3):
        want = oracle.cambi_cvalues(lv[f], win, d, wt)
        assert np.array_equal(cv[f].view(np.uint32), want.view(np.uint32)), f
        assert np.any(want > 0)
