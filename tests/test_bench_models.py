"""The work models bench.py reports rooflines with, checked against the
kernels they describe (no GPU): the CAMBI bin-update count follows the
c-value kernel's lane groups, and an interior warp's share equals the
closed form of that design."""
from __future__ import annotations

import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _kernel_group() -> int:
    src = open(os.path.join(ROOT, "ssimulacra2_image_scoring_gb300", "csrc", "cambi.cu")).read()
    return int(re.search(r"constexpr int kGroup = (\d+);", src).group(1))


def test_cambi_model_uses_the_kernels_lane_group():
    assert bench.CAMBI_GROUP == _kernel_group()


def test_cambi_updates_of_an_interior_warp():
    """Widening a plane by one warp of 32 columns adds one interior warp's
    updates: per row event, every lane's (group - 1) own columns and every
    group's 2r + 2 - group core columns (a one-row plane has one row event,
    the first window's only row)."""
    g = bench.CAMBI_GROUP
    for win in (9, 17, 33, 65):
        r = win // 2
        per_row = 32 * (g - 1) + (32 // g) * (2 * r + 2 - g)
        wide = 32 * 4 + 2 * r
        extra = bench.cambi_updates(wide + 32, 1, win) - bench.cambi_updates(wide, 1, win)
        assert extra == per_row, (win, extra, per_row)
