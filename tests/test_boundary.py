"""The C ABI without a GPU: the library loads, exports every function that
include/ss2.h declares, rejects bad arguments with -EINVAL before touching
the device, and builds the same constant tables as the oracle."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared() -> list[str]:
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(ss2_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L(built):
    from ssimulacra2_image_scoring_gb300 import lib
    return lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


@pytest.mark.parametrize("geom,reason", [
    ((7, 8, 8, 420), "below"), ((8, 7, 8, 444), "below"), ((16385, 16, 8, 444), "above"),
    ((64, 48, 7, 420), "bit depth"), ((64, 48, 17, 420), "bit depth"),
    ((64, 48, 8, 411), "chroma"), ((63, 48, 8, 420), "odd width"), ((63, 48, 8, 422), "odd width"),
])
def test_create_rejects_bad_geometry(L, geom, reason):
    from ssimulacra2_image_scoring_gb300 import last_error
    assert L.ss2_create(*geom) is None
    code, msg = last_error()
    assert code == -22 and reason in msg


def test_bad_batch_and_null_context(L):
    from ssimulacra2_image_scoring_gb300 import last_error
    assert L.ss2_create_batch(64, 48, 8, 420, 0) is None
    assert last_error()[0] == -22
    assert L.ss2_create_batch(64, 48, 8, 420, 1025) is None
    assert L.ss2_score_frames(None, None, None, 1, None, None) == -22
    assert L.ss2_values(None, None, None, 1, None, None, None) == -22
    assert L.ss2_score_frames_host(None, None, None, 1, None, None) == -22
    assert L.ss2_set_params(None, None, 133) == -22
    assert L.ss2_profile_begin(None) == -22
    L.ss2_destroy(None)
    assert L.ss2_frame_bytes(None) == 0


def test_noalloc_rejections_happen_before_device_use(L):
    from ssimulacra2_image_scoring_gb300 import last_error
    assert L.ss2_score_frames_noalloc(7, 8, 8, 444, None, None, 1, None, None) == -22
    assert L.ss2_score_frames_noalloc(64, 48, 8, 420, None, None, 1, None, None) == -22
    assert L.ss2_score_frames_noalloc(64, 48, 8, 420, None, None, -1, None, None) == -22
    assert L.ss2_score_frames_noalloc(3840, 2160, 8, 420, 1, 1, 1, 1, None) == -22
    assert "64 MiB" in last_error()[1]
    assert L.ss2_score_frames_noalloc(64, 48, 8, 420, None, None, 0, None, None) == 0


def test_create_without_device_reports_enotsup(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    from ssimulacra2_image_scoring_gb300 import last_error
    assert L.ss2_create(64, 48, 8, 420) is None
    assert last_error()[0] == -95


def test_host_tables_equal_the_oracle_tables(L):
    """The library builds its EOTF table and recursive-Gaussian coefficients
    with its own host code; both must equal the oracle's bit for bit."""
    from ssimulacra2_image_scoring_gb300 import host_tables
    eotf, iir = host_tables()
    assert np.array_equal(eotf.view(np.uint32), oracle.eotf_table().view(np.uint32))
    _, c2, g = oracle.iir_coeffs()
    assert np.array_equal(iir[:3].view(np.uint32), c2.view(np.uint32))
    assert np.array_equal(iir[3:].view(np.uint32), g.view(np.uint32))


def test_default_params_equal_the_oracle_defaults(L):
    from ssimulacra2_image_scoring_gb300 import default_params
    assert np.array_equal(default_params(), oracle.default_params())
    bad = np.zeros(5)
    assert L.ss2_default_params(bad.ctypes.data, 5) == -22


def test_binding_has_no_fallback(monkeypatch, built):
    """Without the shared library the binding raises instead of computing."""
    from ssimulacra2_image_scoring_gb300 import _build, ss2
    monkeypatch.setattr(ss2, "_lib", None)
    monkeypatch.setattr(_build, "SO_PATH", "/nonexistent/libss2.so")
    with pytest.raises(RuntimeError):
        ss2.lib()
    _ = ctypes


def test_host_cube_root_matches_oracle(L):
    """The host cube root behind the cbrt(bias) constants: bitwise equal to
    the oracle's correctly rounded cbrtf on a sweep of bit patterns of both
    signs (subnormals, binade edges, powers of two and their neighbours,
    random finite floats, the default biases), with zeros keeping their sign
    and non-finite inputs copied."""
    from ssimulacra2_image_scoring_gb300 import ss2
    rng = np.random.default_rng(7)
    bits = [rng.integers(0, 0x7f800000, 200_000, dtype=np.uint32)]            # random finite
    bits.append(np.arange(0, 1 << 16, dtype=np.uint32))                       # subnormals
    e = np.arange(1, 255, dtype=np.uint32) << 23
    bits += [e, e + 1, e - 1, e | 0x7fffff]                                   # binade edges
    bits.append(np.arange(0x3f800000 - 50_000, 0x3f800000 + 50_000, dtype=np.uint32))
    b = np.concatenate(bits)
    x = np.concatenate([b, b | np.uint32(0x80000000)]).view(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, np.inf, -np.inf, np.nan], np.float32)])
    bias = oracle.default_params()[oracle.P_BIAS:oracle.P_BIAS + 3].astype(np.float32)
    x = np.concatenate([x, bias, -bias])
    got = ss2.debug_cbrt_host(x)
    fin = np.isfinite(x)
    want = oracle.cbrtf_cr_array(x[fin])
    assert np.array_equal(got[fin].view(np.uint32), want.view(np.uint32))
    assert np.array_equal(got[~fin].view(np.uint32), x[~fin].view(np.uint32))
    zeros = x == 0
    assert np.array_equal(np.signbit(got[zeros]), np.signbit(x[zeros]))
    assert L.ss2_debug_cbrt_host(None, None, 1) == -22
