"""Failure paths on the GPU, without faulting it.

Failures are made on the host (SS2_FAULT makes an allocation, a launch or a
read-back fail before it touches the device) or by a bounded wait that runs
out (a barrier phase that nothing completes); each must surface as an error
code and leave the context and the device usable.
"""
from __future__ import annotations

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _frames(wl):
    import torch
    return torch.from_numpy(wl.ref).cuda(), torch.from_numpy(wl.dis).cuda()


def test_injected_allocation_failure(cuda, monkeypatch):
    from ssimulacra2_image_scoring_gb300 import Scorer, SS2Error
    monkeypatch.setenv("SS2_FAULT", "alloc")
    with pytest.raises(SS2Error) as e:
        Scorer(64, 48, 8, 420)
    assert e.value.code == -12 and "injected" in str(e.value)
    monkeypatch.delenv("SS2_FAULT")
    wl = synth.custom(64, 48, 8, 420, 2, seed=4)
    with Scorer(64, 48, 8, 420) as sc:
        assert np.all(np.isfinite(sc.score(*_frames(wl))))


@pytest.mark.parametrize("kind", ["launch", "memcpy"])
def test_injected_launch_and_copy_failures(cuda, monkeypatch, kind):
    import torch
    from ssimulacra2_image_scoring_gb300 import Scorer, SS2Error
    wl = synth.custom(96, 64, 8, 420, 5, seed=6)
    ref, dis = _frames(wl)
    with Scorer(96, 64, 8, 420, batch=2) as sc:
        want = sc.score(ref, dis)
        monkeypatch.setenv("SS2_FAULT", kind)
        with pytest.raises(SS2Error) as e:
            sc.score(ref, dis)
        assert e.value.code == -5 and "injected" in str(e.value)
        with pytest.raises(SS2Error):
            sc.score_host(wl.ref, wl.dis)
        monkeypatch.delenv("SS2_FAULT")
        assert np.array_equal(sc.score(ref, dis), want)
        assert np.array_equal(sc.score_host(torch.from_numpy(wl.ref).pin_memory(),
                                            torch.from_numpy(wl.dis).pin_memory()), want)


def test_bounded_wait_gives_up_and_device_stays_usable(cuda):
    from ssimulacra2_image_scoring_gb300 import Scorer, last_error, lib
    L = lib()
    assert L.ss2_debug_wait_probe(4096, None) == -5
    assert "gave up" in last_error()[1]
    wl = synth.custom(64, 48, 8, 420, 2, seed=9)
    with Scorer(64, 48, 8, 420) as sc:
        assert np.all(np.isfinite(sc.score(*_frames(wl))))
