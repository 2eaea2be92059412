"""ss2_score_frames_noalloc against ss2_score_frames and the oracle (GPU).

The allocation-free entry point serves callers that cannot call cudaMalloc
while scoring (code inside a custom allocator or pool callback, fixed memory
budgets, plug-ins that are handed buffers).  It runs the same kernels with
their workspace in a fixed 64 MiB device array inside the library, so its
scores must equal the context-based entry point's bit for bit and lie within
the score tolerance of the oracle; they must also repeat exactly on a second
call, since the shared array keeps the last call's contents.  A wait that
runs out must show up as NaN scores, and the next call must be clean again.
This file sorts last so a stop-at-first-failure run has already run every
other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-6


@pytest.mark.parametrize("geom,frames", [((576, 324, 8, 420), 5), ((853, 481, 10, 444), 3),
                                         ((130, 66, 12, 422), 9)],
                         ids=["576x324", "853x481", "130x66"])
def test_noalloc_matches_context_entry_point(cuda, geom, frames):
    import torch

    from ssimulacra2_image_scoring_gb300 import Scorer, ss2
    w, h, d, c = geom
    wl = synth.custom(w, h, d, c, frames, seed=31)
    ref = torch.from_numpy(wl.ref).cuda()
    dis = torch.from_numpy(wl.dis).cuda()
    with Scorer(w, h, d, c) as sc:
        want = sc.score(ref, dis)
    first = ss2.score_noalloc(w, h, d, c, ref, dis)
    torch.cuda.synchronize()
    second = ss2.score_noalloc(w, h, d, c, ref, dis)
    torch.cuda.synchronize()
    a, b = first.cpu().numpy(), second.cpu().numpy()
    assert np.array_equal(a, want) and np.array_equal(b, want)
    ora, _ = oracle.score_frames(wl.ref, wl.dis, w, h, d, c)
    assert np.max(np.abs(a - ora)) <= SCORE_TOL


def test_noalloc_marks_a_timed_out_wait_with_nan(cuda):
    """The test hook makes a bounded wait run out against the call's error
    word (no fault, no hang): that call's scores are NaN; with the hook off,
    the next call clears the word and scores normally."""
    import torch

    from ssimulacra2_image_scoring_gb300 import ss2
    L = ss2.lib()
    wl = synth.custom(96, 64, 8, 420, 3, seed=12)
    ref = torch.from_numpy(wl.ref).cuda()
    dis = torch.from_numpy(wl.dis).cuda()
    good = ss2.score_noalloc(96, 64, 8, 420, ref, dis).cpu().numpy()
    assert np.all(np.isfinite(good))
    assert L.ss2_debug_noalloc_timeout(4096) == 0
    try:
        bad = ss2.score_noalloc(96, 64, 8, 420, ref, dis).cpu().numpy()
    finally:
        assert L.ss2_debug_noalloc_timeout(0) == 0
    assert np.all(np.isnan(bad))
    again = ss2.score_noalloc(96, 64, 8, 420, ref, dis).cpu().numpy()
    assert np.array_equal(again, good)


def test_noalloc_rejects_frames_beyond_its_scratch(cuda):
    from ssimulacra2_image_scoring_gb300 import ss2
    L = ss2.lib()
    out = ctypes.c_double(0.0)
    rc = L.ss2_score_frames_noalloc(3840, 2160, 8, 420, 1, 1, 1, ctypes.addressof(out), None)
    assert rc == -22
    code, msg = ss2.last_error()
    assert code == -22 and "64 MiB" in msg
    assert L.ss2_score_frames_noalloc(64, 48, 8, 420, None, None, 0, None, None) == 0
