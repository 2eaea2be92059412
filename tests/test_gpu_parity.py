"""GPU path vs the oracle, through the C ABI.

Bars (per the numerics of "Research-1363: Device-resident ssimulacra2 ...",
Findings 2 and 4):
  - XYB planes and horizontally blurred planes: bitwise equal at every scale
    (the fp32 pipeline up to the sums is reproduced exactly);
  - the 108 pooled values: relative 1e-9 (double-float sums in a fixed tree
    against the oracle's sequential fp64 sums; the page measured ~1e-12 on
    the score);
  - scores: |d| <= 1e-6 per frame, on every frame of the five workloads.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-6
VALUE_RTOL = 1e-9
VALUE_ATOL = 1e-12


def _oracle_frames(wl, params=None, frames=None):
    """Oracle scores and values for the given workload rows, frames in parallel
    (ctypes releases the GIL; the oracle keeps no global state)."""
    sp = wl.spec
    idx = list(range(wl.ref.shape[0])) if frames is None else list(frames)

    def one(j):
        s, v, _ = oracle.score(wl.ref[j], wl.dis[j], sp.width, sp.height, sp.depth, sp.chroma,
                               params)
        return s, v

    with cf.ThreadPoolExecutor(max_workers=min(len(idx), os.cpu_count() or 1)) as ex:
        res = list(ex.map(one, idx))
    return np.array([r[0] for r in res]), np.stack([r[1] for r in res])


def _to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _scorer(sp, **kw):
    from ssimulacra2_image_scoring_gb300 import Scorer
    return Scorer(sp.width, sp.height, sp.depth, sp.chroma, **kw)


def _check_values(got_v, want_v):
    err = np.abs(got_v - want_v)
    bound = VALUE_ATOL + VALUE_RTOL * np.abs(want_v)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"values differ at {bad[:5].tolist()}: got {got_v[tuple(bad[0])]} " \
                          f"want {want_v[tuple(bad[0])]}"


GEOMS = [
    # (w, h, depth, chroma): ragged tails, odd sizes, every chroma layout.
    # Rows whose starts all fall on 16 bytes take the pyramid kernel's
    # 16-byte staging copies (64x48, 224x100, 224x101, 96x70, 80x72); the
    # others take its 4-byte word staging (aligned loads inside the frame,
    # single samples at a frame's ends).
    (64, 48, 8, 420),
    (853, 481, 8, 444),
    (17, 13, 10, 444),
    (130, 66, 9, 422),
    (200, 97, 11, 420),
    (8, 8, 8, 444),
    (224, 100, 8, 420),
    (224, 101, 10, 420),
    (96, 70, 12, 422),
    (80, 72, 8, 444),
]


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: "x".join(map(str, g)))
def test_planes_bitwise(cuda, geom):
    w, h, d, c = geom
    wl = synth.custom(w, h, d, c, 1, seed=11)
    ref, dis = _to_dev(wl.ref), _to_dev(wl.dis)
    dims = oracle.scale_dims(w, h)
    with _scorer(wl.spec) as sc:
        for s in range(len(dims)):
            xyb, hb = sc.debug_planes(ref, dis, s)
            _, _, dump = oracle.score(wl.ref[0], wl.dis[0], w, h, d, c, dump_scale=s)
            assert np.array_equal(xyb.view(np.uint32), dump["xyb"].view(np.uint32)), \
                f"XYB differs at scale {s}"
            assert np.array_equal(hb.view(np.uint32), dump["hblur"].view(np.uint32)), \
                f"horizontal blur differs at scale {s}"


@pytest.mark.parametrize("geom", [(853, 481, 8, 444), (17, 13, 10, 444), (131, 67, 9, 444),
                                  (201, 99, 8, 444)],
                         ids=lambda g: "x".join(map(str, g)))
def test_planes_bitwise_from_unaligned_frame(cuda, geom):
    """Frame 1 of a batch whose frame size is not a multiple of 4 bytes,
    handed over as a view that starts at that odd offset: the pyramid
    kernel's word staging then meets every byte alignment and its
    sample-by-sample reads at the frame's first and last bytes."""
    w, h, d, c = geom
    wl = synth.custom(w, h, d, c, 2, seed=17)
    ref, dis = _to_dev(wl.ref), _to_dev(wl.dis)
    r1, d1 = ref[1:], dis[1:]
    assert r1.data_ptr() % 4 != 0, "the case must start off a word boundary"
    dims = oracle.scale_dims(w, h)
    with _scorer(wl.spec) as sc:
        for s in range(len(dims)):
            xyb, hb = sc.debug_planes(r1, d1, s)
            _, _, dump = oracle.score(wl.ref[1], wl.dis[1], w, h, d, c, dump_scale=s)
            assert np.array_equal(xyb.view(np.uint32), dump["xyb"].view(np.uint32)), \
                f"XYB differs at scale {s}"
            assert np.array_equal(hb.view(np.uint32), dump["hblur"].view(np.uint32)), \
                f"horizontal blur differs at scale {s}"


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: "x".join(map(str, g)))
def test_linear_pyramid_bitwise(cuda, geom):
    """Linear RGB at scale 0 and the 2x2-downsampled linear RGB of scales 1-5
    (which the pyramid kernel keeps on chip) bitwise against the oracle's."""
    w, h, d, c = geom
    wl = synth.custom(w, h, d, c, 1, seed=13)
    ref, dis = _to_dev(wl.ref), _to_dev(wl.dis)
    dims = oracle.scale_dims(w, h)
    with _scorer(wl.spec) as sc:
        for s in range(len(dims)):
            lin = sc.debug_linear(ref, dis, s)
            _, _, dump = oracle.score(wl.ref[0], wl.dis[0], w, h, d, c, dump_scale=s)
            assert np.array_equal(lin.view(np.uint32), dump["lin"].view(np.uint32)), \
                f"linear RGB differs at scale {s}"


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: "x".join(map(str, g)))
def test_values_and_scores(cuda, geom):
    w, h, d, c = geom
    wl = synth.custom(w, h, d, c, 3, seed=5)
    with _scorer(wl.spec) as sc:
        got_v, got_s = sc.values(_to_dev(wl.ref), _to_dev(wl.dis))
    want_s, want_v = _oracle_frames(wl)
    _check_values(got_v, want_v)
    assert np.max(np.abs(got_s - want_s)) <= SCORE_TOL


def test_identical_pair_scores_100(cuda):
    wl = synth.custom(96, 64, 8, 420, 2, seed=3)
    with _scorer(wl.spec) as sc:
        s = sc.score(_to_dev(wl.ref), _to_dev(wl.ref))
    assert np.all(s == 100.0), s


def test_random_params(cuda):
    """Non-default weights, map, opsin matrix, affine and C2 (the parity path
    must not depend on the placeholder values)."""
    rng = np.random.default_rng(123)
    p = oracle.default_params()
    p[0:108] = rng.uniform(0.0, 2.0, 108)
    p[108:112] = [90.0, -70.0, 5.0, -1.0]
    p[112:115] = [1.5, 0.8, -3.0]
    p[115:124] = rng.uniform(0.05, 0.7, 9)
    p[124:127] = rng.uniform(0.002, 0.01, 3)
    p[127:132] = [1.7, 0.3, 0.1, 0.9, 0.05]
    p[132] = 0.002
    wl = synth.custom(150, 90, 10, 420, 3, seed=9)
    with _scorer(wl.spec, params=p) as sc:
        got_v, got_s = sc.values(_to_dev(wl.ref), _to_dev(wl.dis))
        xyb, hb = sc.debug_planes(_to_dev(wl.ref), _to_dev(wl.dis), 1)
    want_s, want_v = _oracle_frames(wl, params=p)
    _check_values(got_v, want_v)
    assert np.max(np.abs(got_s - want_s)) <= SCORE_TOL
    _, _, dump = oracle.score(wl.ref[0], wl.dis[0], 150, 90, 10, 420, p, dump_scale=1)
    assert np.array_equal(xyb.view(np.uint32), dump["xyb"].view(np.uint32))
    assert np.array_equal(hb.view(np.uint32), dump["hblur"].view(np.uint32))


def test_cbrt_matches_oracle_on_reachable_domain(cuda):
    """Every float in [2^-9, 2) (the opsin outputs of [0,1] RGB lie in
    [bias, 1 + bias]) plus a stride through the rest of the positive floats
    and both zeros, bitwise against the oracle's correctly rounded cube
    root."""
    import torch
    from ssimulacra2_image_scoring_gb300 import ss2
    lo = np.float32(2.0 ** -9).view(np.uint32)
    hi = np.float32(2.0).view(np.uint32)
    bits = np.concatenate([np.array([0, 0x80000000], dtype=np.uint32),
                           np.arange(lo, hi, dtype=np.uint32),
                           np.arange(1, 0x7f800000, 9973, dtype=np.uint32)])
    x = bits.view(np.float32)
    got = ss2.debug_cbrt(torch.from_numpy(x).cuda()).cpu().numpy()
    want = oracle.cbrtf_cr_array(x)
    bad = np.flatnonzero(want.view(np.uint32) != got.view(np.uint32))
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[0]]!r}"


def test_determinism_and_batch_invariance(cuda):
    wl = synth.custom(300, 170, 8, 420, 7, seed=21)
    ref, dis = _to_dev(wl.ref), _to_dev(wl.dis)
    with _scorer(wl.spec, batch=7) as a, _scorer(wl.spec, batch=3) as b:
        v1, s1 = a.values(ref, dis)
        v2, s2 = a.values(ref, dis)
        v3, s3 = b.values(ref, dis)
    assert np.array_equal(s1, s2) and np.array_equal(v1, v2)
    assert np.array_equal(s1, s3) and np.array_equal(v1, v3)


def test_graph_replay_matches_eager_launches(cuda):
    """Device-input calls replayed from a captured CUDA graph give the bits of
    one-by-one launches: repeated calls, another frame count, with and without
    the values, under per-kernel timing (the same launches counted) and after
    new parameters (which drop the graph)."""
    wl = synth.custom(200, 97, 11, 420, 5, seed=23)
    ref, dis = _to_dev(wl.ref), _to_dev(wl.dis)
    with _scorer(wl.spec, batch=2) as sc:      # three batches over both lanes
        sc.set_graphs(False)
        v0, s0 = sc.values(ref, dis)
        sc.profile_begin()
        sc.score(ref, dis)
        sc.score(ref, dis)
        prof_eager = sc.profile_end()
        sc.set_graphs(True)
        for _ in range(3):                     # capture, then replays
            v, s = sc.values(ref, dis)
            assert np.array_equal(v, v0) and np.array_equal(s, s0)
            assert np.array_equal(sc.score(ref, dis), s0)
        assert np.array_equal(sc.score(ref[:3], dis[:3]), s0[:3])
        sc.profile_begin()
        sc.score(ref, dis)
        sc.score(ref, dis)
        prof_graph = sc.profile_end()
        assert {k: n for k, (_, n) in prof_graph.items()} == \
               {k: n for k, (_, n) in prof_eager.items()}
        assert all(ms > 0.0 for ms, _ in prof_graph.values())
        p = oracle.default_params()
        p[132] = 0.002                         # C2
        sc.set_params(p)
        s_new = sc.score(ref, dis)
        sc.set_graphs(False)
        assert np.array_equal(sc.score(ref, dis), s_new)
    assert not np.array_equal(s_new, s0)


def test_host_input_path_matches_device_path_and_oracle(cuda):
    """The host-input path (pinned and pageable frames, calls shorter than its
    short first batch) against the device-input path bitwise, and against the
    oracle within the score tolerance."""
    import torch
    wl = synth.custom(256, 144, 10, 422, 9, seed=2)
    want, _ = _oracle_frames(wl)
    with _scorer(wl.spec, batch=4) as sc:
        s_dev = sc.score(_to_dev(wl.ref), _to_dev(wl.dis))
        pr = torch.from_numpy(wl.ref).pin_memory()
        pd = torch.from_numpy(wl.dis).pin_memory()
        s_host = sc.score_host(pr, pd)
        s_page = sc.score_host(wl.ref, wl.dis)
        # calls no longer than the host path's short first batch
        s_one = sc.score_host(pr[:1], pd[:1])
        s_two = sc.score_host(pr[:2], pd[:2])
    assert np.array_equal(s_dev, s_host) and np.array_equal(s_dev, s_page)
    assert np.array_equal(s_dev[:1], s_one) and np.array_equal(s_dev[:2], s_two)
    assert np.max(np.abs(s_host - want)) <= SCORE_TOL
    assert np.max(np.abs(s_page - want)) <= SCORE_TOL


def test_context_reuse_two_geometries(cuda):
    """Two contexts of different sizes used alternately (a reused state must
    not keep the first size: Research-1369, section 7)."""
    a = synth.custom(64, 48, 8, 420, 2, seed=1)
    b = synth.custom(128, 96, 8, 420, 2, seed=1)
    want_a, _ = _oracle_frames(a)
    want_b, _ = _oracle_frames(b)
    with _scorer(a.spec) as sa, _scorer(b.spec) as sb:
        for _ in range(2):
            ga = sa.score(_to_dev(a.ref), _to_dev(a.dis))
            gb = sb.score(_to_dev(b.ref), _to_dev(b.dis))
            assert np.max(np.abs(ga - want_a)) <= SCORE_TOL
            assert np.max(np.abs(gb - want_b)) <= SCORE_TOL


@pytest.mark.parametrize("depth", [9, 11, 16])
def test_odd_and_full_depths(cuda, depth):
    wl = synth.custom(120, 72, depth, 420, 2, seed=depth)
    with _scorer(wl.spec) as sc:
        got = sc.score(_to_dev(wl.ref), _to_dev(wl.dis))
    want, _ = _oracle_frames(wl)
    assert np.max(np.abs(got - want)) <= SCORE_TOL


def test_edge_geometries(cuda):
    """Maximum width and height (with the other side small), the 8x8 minimum
    and a single-frame batch of an odd size."""
    from ssimulacra2_image_scoring_gb300 import SS2Error
    for (w, h, d, c) in [(16384, 16, 8, 444), (16, 16384, 8, 420), (8, 8, 8, 420),
                         (9, 8, 12, 444)]:
        wl = synth.custom(w, h, d, c, 1, seed=w + h)
        with _scorer(wl.spec) as sc:
            got = sc.score(_to_dev(wl.ref), _to_dev(wl.dis))
        want, _ = _oracle_frames(wl)
        assert abs(got[0] - want[0]) <= SCORE_TOL, (w, h, got, want)
    with pytest.raises(SS2Error):
        _scorer(synth.Spec("x", 16385, 16, 8, 444, 1, 0, ""))


def test_zero_frames_and_bad_calls(cuda):
    import torch
    from ssimulacra2_image_scoring_gb300 import SS2Error, lib
    wl = synth.custom(32, 32, 8, 420, 1, seed=0)
    with _scorer(wl.spec) as sc:
        e = torch.empty(0, dtype=torch.uint8, device="cuda")
        assert sc.score(e, e).shape == (0,)
        L = lib()
        assert L.ss2_score_frames(sc.handle, None, None, 1, None, None) == -22
        assert L.ss2_score_frames(sc.handle, 1, 1, -1, None, None) == -22
        assert L.ss2_debug_planes(sc.handle, 1, 1, 3, None, None, None) == -22
        with pytest.raises(SS2Error):
            sc.set_params(np.zeros(5))


# ---------------------------------------------------------------------------
# The five workloads, in the launch configuration the benchmark times
# (default batch), every frame against the oracle; the 4K workloads also
# through the host-input path.
# ---------------------------------------------------------------------------

WORKLOADS = ["c0_576x324_8b_420", "c1_853x481_8b_444", "c2_1920x1080_10b_420",
             "c3_3840x2160_8b_420", "c4_3840x2160_12b_444"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_parity(cuda, name):
    import torch
    spec = synth.SPECS[name]
    wl = synth.make(name)
    with _scorer(spec) as sc:
        got = sc.score(_to_dev(wl.ref), _to_dev(wl.dis))
        got_host = None
        if spec.width >= 3840:
            got_host = sc.score_host(torch.from_numpy(wl.ref).pin_memory(),
                                     torch.from_numpy(wl.dis).pin_memory())
    want, _ = _oracle_frames(wl)
    err = np.abs(got - want)
    assert err.max() <= SCORE_TOL, f"{name}: max |d| {err.max():.3e} at frame {int(err.argmax())}"
    if got_host is not None:
        assert np.array_equal(got_host, got)
    if name == "c1_853x481_8b_444":
        assert want[0] == 100.0 and got[0] == 100.0
    if name == "c4_3840x2160_12b_444":
        assert want[0] == 100.0 and np.all(got[0::4] == 100.0)
