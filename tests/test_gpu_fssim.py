"""float_ssim with device decimation vs the oracle (GPU).

Decimated planes: bitwise (the window sum is exact on both sides).  Scores:
within 1e-6, twenty times inside the float_ssim parity gate (5e-5) of
"ADR-1405: float_ssim_hip decimates on the device, bit-identical to the CPU"
(Context).  The map's Gaussian sums are fp32 on the device, on samples
shifted by a per-tile offset, and fp64 in the oracle; an fp32 emulation of
the device arithmetic stays within 1e-8 of the oracle on these inputs.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

GEOMS = [  # (w, h, depth, chroma); the factor and the decimation kernel that runs
    (576, 324, 8, 420),      # 1: k_fssim_decimate_tma (8-bit, power of two)
    (853, 481, 8, 444),      # 3: k_fssim_decimate (rows are not whole 16-byte chunks)
    (768, 768, 10, 420),     # 3: k_fssim_decimate_tma (16-bit samples)
    (1280, 720, 12, 444),    # 3: k_fssim_decimate_tma
    (1280, 720, 8, 420),     # 3: k_fssim_decimate_tma (8-bit, 2^-52 counts)
    (1920, 1080, 16, 420),   # 4: k_fssim_decimate_tma (16-bit, power of two)
    (2304, 1296, 9, 422),    # 5: k_fssim_decimate_tma, 2 row groups
    (1024, 600, 8, 420),     # 2: k_fssim_decimate_u8
    (1920, 1080, 8, 420),    # 4: k_fssim_decimate_u8
    (3840, 2160, 8, 420),    # 8: k_fssim_decimate_u8, 2 row groups
    (4096, 4096, 8, 420),    # 16: k_fssim_decimate_u8, 4 row groups
    (5120, 2048, 8, 420),    # 8: k_fssim_decimate_tma (8-bit wider than 4096)
    (3840, 2160, 12, 444),   # 8: k_fssim_decimate_tma, 4 row groups
    (2880, 2880, 10, 444),   # 11: k_fssim_decimate_tma, 6 row groups
]


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: "x".join(map(str, g)))
def test_fssim_planes_and_scores(cuda, geom):
    import torch

    from ssimulacra2_image_scoring_gb300 import FloatSSIM
    w, h, d, c = geom
    wl = synth.custom(w, h, d, c, 3, seed=w + d, noise=4.0)
    ref = torch.from_numpy(wl.ref).cuda()
    dis = torch.from_numpy(wl.dis).cuda()
    with FloatSSIM(w, h, d, c) as fs:
        assert fs.scale == oracle.fssim_scale(w, h)
        planes = fs.decimated(ref, dis)
        got = fs.score(ref, dis)
    want = []
    for f in range(3):
        s, a, b = oracle.fssim(wl.ref[f], wl.dis[f], w, h, d)
        want.append(s)
        if f == 0:
            assert np.array_equal(planes[0].view(np.uint32), a.view(np.uint32))
            assert np.array_equal(planes[1].view(np.uint32), b.view(np.uint32))
    err = np.abs(got - np.array(want))
    assert err.max() <= 1e-6, (got, want)


def test_fssim_identical_and_batches(cuda):
    import torch

    from ssimulacra2_image_scoring_gb300 import FloatSSIM
    wl = synth.custom(1024, 600, 8, 420, 9, seed=1, noise=6.0)
    ref = torch.from_numpy(wl.ref).cuda()
    dis = torch.from_numpy(wl.dis).cuda()
    with FloatSSIM(1024, 600, 8, 420, batch=4) as a, FloatSSIM(1024, 600, 8, 420) as b:
        s1 = a.score(ref, dis)
        s2 = b.score(ref, dis)
        same = a.score(ref, ref)
    assert np.array_equal(s1, s2)
    assert np.all(np.abs(same - 1.0) <= 1e-6)


def test_fssim_refuses_small_planes(cuda):
    from ssimulacra2_image_scoring_gb300 import FloatSSIM, SS2Error
    with pytest.raises(SS2Error) as e:
        FloatSSIM(10, 10, 8, 444)
    assert e.value.code == -95


@pytest.mark.parametrize("geom", [(3840, 2160, 8, 420), (2880, 2880, 10, 444)],
                         ids=lambda g: "x".join(map(str, g)))
def test_fssim_unaligned_frames_take_the_unstaged_kernel(cuda, geom):
    """Frames at an address that is not 16-byte aligned cannot be bulk-copied;
    the unstaged kernel must give the same planes and scores bitwise."""
    import torch

    from ssimulacra2_image_scoring_gb300 import FloatSSIM
    w, h, d, c = geom
    wl = synth.custom(w, h, d, c, 2, seed=5, noise=3.0)
    ref = torch.from_numpy(wl.ref).cuda()
    dis = torch.from_numpy(wl.dis).cuda()
    n, fe = wl.ref.shape

    def shifted(x):
        buf = torch.empty(n * fe + 16, dtype=x.dtype, device="cuda")
        v = buf[1:1 + n * fe].view(n, fe)
        v.copy_(x)
        assert v.data_ptr() % 16 != 0 and v.is_contiguous()
        return v

    rs, ds = shifted(ref), shifted(dis)
    with FloatSSIM(w, h, d, c) as fs:
        a = fs.score(ref, dis)
        b = fs.score(rs, ds)
        pa = fs.decimated(ref, dis)
        pb = fs.decimated(rs, ds)
    assert np.array_equal(a, b)
    assert np.array_equal(pa.view(np.uint32), pb.view(np.uint32))
