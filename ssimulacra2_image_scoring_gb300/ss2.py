"""ctypes binding of libss2 (include/ss2.h).

Argument marshalling only: every step of the scoring path runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the current
stream.  If the shared library is missing the binding raises; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import _build

NVALUES = 108
NPARAMS = 133
EOTF_N = 4096

EINVAL, ENOMEM, ENOTSUP, EIO = -22, -12, -95, -5

_lock = threading.Lock()
_lib = None


class SS2Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libss2 error {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Loads libss2.so (built by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.SO_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is not built; call __graft_entry__.build() first")
            L = ctypes.CDLL(path)
            vp, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            L.ss2_create.argtypes = [i, i, i, i]
            L.ss2_create.restype = vp
            L.ss2_create_batch.argtypes = [i, i, i, i, i]
            L.ss2_create_batch.restype = vp
            L.ss2_destroy.argtypes = [vp]
            L.ss2_destroy.restype = None
            L.ss2_score_frames.argtypes = [vp, vp, vp, i, vp, vp]
            L.ss2_score_frames.restype = i
            L.ss2_score_frames_host.argtypes = [vp, vp, vp, i, vp, vp]
            L.ss2_score_frames_host.restype = i
            L.ss2_values.argtypes = [vp, vp, vp, i, vp, vp, vp]
            L.ss2_values.restype = i
            L.ss2_debug_planes.argtypes = [vp, vp, vp, i, vp, vp, vp]
            L.ss2_debug_planes.restype = i
            L.ss2_debug_linear.argtypes = [vp, vp, vp, i, vp, vp]
            L.ss2_debug_linear.restype = i
            L.ss2_debug_cbrt.argtypes = [vp, vp, ctypes.c_longlong, vp]
            L.ss2_debug_cbrt.restype = i
            L.ss2_debug_cbrt_host.argtypes = [vp, vp, ctypes.c_longlong]
            L.ss2_debug_cbrt_host.restype = i
            L.ss2_profile_begin.argtypes = [vp]
            L.ss2_profile_begin.restype = i
            L.ss2_profile_end.argtypes = [vp, vp, vp]
            L.ss2_profile_end.restype = i
            L.ss2_set_graphs.argtypes = [vp, i]
            L.ss2_set_graphs.restype = i
            L.ss2_score_frames_noalloc.argtypes = [i, i, i, i, vp, vp, i, vp, vp]
            L.ss2_score_frames_noalloc.restype = i
            L.ss2_debug_wait_probe.argtypes = [ctypes.c_uint, vp]
            L.ss2_debug_wait_probe.restype = i
            L.ss2_debug_noalloc_timeout.argtypes = [ctypes.c_uint]
            L.ss2_debug_noalloc_timeout.restype = i
            L.ss2_fssim_create.argtypes = [i, i, i, i, i]
            L.ss2_fssim_create.restype = vp
            L.ss2_fssim_score.argtypes = [vp, vp, vp, i, vp, vp]
            L.ss2_fssim_score.restype = i
            L.ss2_fssim_scale.argtypes = [vp]
            L.ss2_fssim_scale.restype = i
            L.ss2_fssim_debug_decimated.argtypes = [vp, vp, vp, vp, vp]
            L.ss2_fssim_debug_decimated.restype = i
            L.ss2_fssim_profile_begin.argtypes = [vp]
            L.ss2_fssim_profile_begin.restype = i
            L.ss2_fssim_profile_end.argtypes = [vp, vp, vp]
            L.ss2_fssim_profile_end.restype = i
            ll = ctypes.c_longlong
            L.ss2_cambi_create.argtypes = [i, i, i, i, vp, vp, i]
            L.ss2_cambi_create.restype = vp
            L.ss2_cambi_cvalues.argtypes = [vp, vp, vp, i, vp, vp]
            L.ss2_cambi_cvalues.restype = i
            L.ss2_cambi_topk.argtypes = [vp, vp, i, ll, vp, vp, vp, vp]
            L.ss2_cambi_topk.restype = i
            L.ss2_cambi_pool.argtypes = [vp, vp, vp, i, ll, vp, vp, vp, vp]
            L.ss2_cambi_pool.restype = i
            L.ss2_cambi_profile_begin.argtypes = [vp]
            L.ss2_cambi_profile_begin.restype = i
            L.ss2_cambi_profile_end.argtypes = [vp, vp, vp]
            L.ss2_cambi_profile_end.restype = i
            L.ss2_cambi_destroy.argtypes = [vp]
            L.ss2_cambi_destroy.restype = None
            L.ss2_msssim_create.argtypes = [i, i, i, i, i]
            L.ss2_msssim_create.restype = vp
            L.ss2_msssim_create_ex.argtypes = [i, i, i, i, i, i]
            L.ss2_msssim_create_ex.restype = vp
            L.ss2_msssim_planes.argtypes = [vp]
            L.ss2_msssim_planes.restype = i
            L.ss2_msssim_debug_pyramid_plane.argtypes = [vp, vp, vp, i, vp, vp]
            L.ss2_msssim_debug_pyramid_plane.restype = i
            L.ss2_msssim_score.argtypes = [vp, vp, vp, i, vp, vp, vp]
            L.ss2_msssim_score.restype = i
            L.ss2_msssim_debug_pyramid.argtypes = [vp, vp, vp, vp, vp]
            L.ss2_msssim_debug_pyramid.restype = i
            L.ss2_msssim_profile_begin.argtypes = [vp]
            L.ss2_msssim_profile_begin.restype = i
            L.ss2_msssim_profile_end.argtypes = [vp, vp, vp]
            L.ss2_msssim_profile_end.restype = i
            L.ss2_msssim_destroy.argtypes = [vp]
            L.ss2_msssim_destroy.restype = None
            L.ss2_fssim_destroy.argtypes = [vp]
            L.ss2_fssim_destroy.restype = None
            L.ss2_frame_bytes.argtypes = [vp]
            L.ss2_frame_bytes.restype = ctypes.c_size_t
            L.ss2_batch.argtypes = [vp]
            L.ss2_batch.restype = i
            L.ss2_workspace_bytes.argtypes = [vp]
            L.ss2_workspace_bytes.restype = ctypes.c_size_t
            L.ss2_default_params.argtypes = [vp, i]
            L.ss2_default_params.restype = i
            L.ss2_set_params.argtypes = [vp, vp, i]
            L.ss2_set_params.restype = i
            L.ss2_host_tables.argtypes = [vp, vp]
            L.ss2_host_tables.restype = i
            L.ss2_last_error.argtypes = []
            L.ss2_last_error.restype = i
            L.ss2_last_error_string.argtypes = []
            L.ss2_last_error_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def last_error() -> tuple[int, str]:
    L = lib()
    return int(L.ss2_last_error()), L.ss2_last_error_string().decode()


def _check(rc: int) -> None:
    if rc != 0:
        code, msg = last_error()
        raise SS2Error(rc, msg)


def default_params() -> np.ndarray:
    p = np.zeros(NPARAMS, np.float64)
    _check(lib().ss2_default_params(p.ctypes.data, NPARAMS))
    return p


def host_tables() -> tuple[np.ndarray, np.ndarray]:
    """The library's host-built EOTF table (4097) and IIR coefficients (6)."""
    eotf = np.zeros(EOTF_N + 1, np.float32)
    iir = np.zeros(6, np.float32)
    _check(lib().ss2_host_tables(eotf.ctypes.data, iir.ctypes.data))
    return eotf, iir


def debug_cbrt(x, out=None, stream=None):
    """The pipeline's cube root applied to a float32 CUDA tensor."""
    import torch
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32
            and x.is_contiguous()):
        raise TypeError("x must be a contiguous float32 CUDA tensor")
    out = torch.empty_like(x) if out is None else out
    _check(lib().ss2_debug_cbrt(x.data_ptr(), out.data_ptr(), x.numel(), _stream_handle(stream)))
    return out


def debug_cbrt_host(x: np.ndarray) -> np.ndarray:
    """The host's cube root (the one behind the cbrt(bias) constants)
    applied to a float32 array; needs no GPU."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    _check(lib().ss2_debug_cbrt_host(x.ctypes.data, y.ctypes.data, x.size))
    return y


def score_noalloc(width: int, height: int, bitdepth: int, chroma: int, ref, dis,
                  scores=None, stream=None):
    """Scores device frames through ss2_score_frames_noalloc, which allocates
    nothing (for callers that cannot call cudaMalloc while scoring).  Returns
    the float64 CUDA tensor of scores; the caller synchronises."""
    import torch
    for t in (ref, dis):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
            raise TypeError("frames must be contiguous CUDA tensors")
    if ref.device != dis.device:
        raise ValueError(f"ref is on {ref.device} and dis on {dis.device}")
    fe = (width * height + 2 * ((width + (chroma != 444)) >> (chroma != 444)) *
          ((height + (chroma == 420)) >> (chroma == 420)))
    fb = fe * (1 if bitdepth <= 8 else 2)
    nbytes = ref.numel() * ref.element_size()
    if nbytes % fb or dis.numel() * dis.element_size() != nbytes:
        raise ValueError("ref/dis must hold the same whole number of frames")
    n = nbytes // fb
    if scores is None:
        scores = torch.empty(n, dtype=torch.float64, device=ref.device)
    elif not (isinstance(scores, torch.Tensor) and scores.dtype == torch.float64 and
              scores.device == ref.device and scores.is_contiguous() and scores.numel() >= n):
        raise ValueError(f"scores must be a contiguous float64 tensor of at least {n} elements "
                         f"on {ref.device}")
    # the C side runs on the current device: make it the frames' device
    with torch.cuda.device(ref.device):
        _check(lib().ss2_score_frames_noalloc(width, height, bitdepth, chroma, ref.data_ptr(),
                                              dis.data_ptr(), n, scores.data_ptr(),
                                              _stream_handle(stream)))
    return scores


def _stream_handle(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


class _Context:
    """Lifetime and per-kernel profiling shared by the context classes: the
    C entry points are <prefix>_destroy, <prefix>_profile_begin and
    <prefix>_profile_end."""

    _PREFIX = ""
    KERNELS: tuple = ()
    _h = None

    def profile_begin(self) -> None:
        """Starts per-kernel CUDA-event timing of this context's launches."""
        _check(getattr(lib(), self._PREFIX + "_profile_begin")(self._h))

    def profile_end(self) -> dict:
        """Stops timing; returns {kernel: (total ms, launches)}."""
        ms = np.zeros(len(self.KERNELS), np.float64)
        n = np.zeros(len(self.KERNELS), np.int32)
        _check(getattr(lib(), self._PREFIX + "_profile_end")(self._h, ms.ctypes.data,
                                                             n.ctypes.data))
        return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(self.KERNELS)}

    def close(self) -> None:
        if self._h:
            getattr(lib(), self._PREFIX + "_destroy")(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

class FloatSSIM(_Context):
    """float_ssim with device decimation for one frame geometry (ss2_fssim_create)."""

    _PREFIX = "ss2_fssim"
    KERNELS = ("k_fssim_decimate", "k_fssim_map", "k_fssim_final")

    def __init__(self, width: int, height: int, bitdepth: int, chroma: int, batch: int = 0):
        h = lib().ss2_fssim_create(width, height, bitdepth, chroma, batch)
        if not h:
            code, msg = last_error()
            raise SS2Error(code, msg)
        self._h = h
        self.width, self.height = width, height
        self.scale = int(lib().ss2_fssim_scale(h))

    def score(self, ref, dis, stream=None) -> np.ndarray:
        import torch
        for t in (ref, dis):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
                raise TypeError("frames must be contiguous CUDA tensors")
        n = ref.shape[0]
        out = np.zeros(n, np.float64)
        _check(lib().ss2_fssim_score(self._h, ref.data_ptr(), dis.data_ptr(), n,
                                     out.ctypes.data, _stream_handle(stream)))
        return out

    def decimated(self, ref, dis, stream=None) -> np.ndarray:
        """The two decimated luma planes (2, hd, wd) of the first frame pair."""
        s = self.scale
        wd, hd = (self.width + s - 1) // s, (self.height + s - 1) // s
        out = np.zeros((2, hd, wd), np.float32)
        _check(lib().ss2_fssim_debug_decimated(self._h, ref.data_ptr(), dis.data_ptr(),
                                               out.ctypes.data, _stream_handle(stream)))
        return out


class Cambi(_Context):
    """CAMBI c-values and top-K pooling for one plane size (ss2_cambi_create)."""

    _PREFIX = "ss2_cambi"
    KERNELS = ("k_cambi_cvalues", "k_cambi_topk")

    def __init__(self, width: int, height: int, window: int, diffs, weights, batch: int = 0):
        d = np.ascontiguousarray(diffs, dtype=np.int32)
        w = np.ascontiguousarray(weights, dtype=np.int32)
        if d.size != w.size:
            raise ValueError("diffs and weights differ in length")
        h = lib().ss2_cambi_create(width, height, window, d.size, d.ctypes.data, w.ctypes.data,
                                   batch)
        if not h:
            code, msg = last_error()
            raise SS2Error(code, msg)
        self._h = h
        self.width, self.height = width, height

    @staticmethod
    def _dev(t, dtype):
        import torch
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous() and t.dtype == dtype):
            raise TypeError(f"expected a contiguous CUDA tensor of {dtype}")
        return t.data_ptr()

    def cvalues(self, levels, mask=None, stream=None):
        """levels: (n, h, w) uint16 CUDA tensor; returns (n, h, w) float32 CUDA c-values."""
        import torch
        n = levels.shape[0]
        out = torch.empty((n, self.height, self.width), dtype=torch.float32, device=levels.device)
        _check(lib().ss2_cambi_cvalues(self._h, self._dev(levels, torch.uint16),
                                       None if mask is None else self._dev(mask, torch.uint8), n,
                                       out.data_ptr(), _stream_handle(stream)))
        return out

    def _pooled(self, n):
        return np.zeros((n, 2), np.uint64), np.zeros(n, np.float32), np.zeros(n, np.float64)

    @staticmethod
    def _result(s, t, m):
        return [(int(hi) << 64) | int(lo) for lo, hi in s], t, m

    def topk(self, cvalues, k: int, stream=None):
        """(exact sums in 2^-24 units as Python ints, thresholds, means) per plane."""
        import torch
        n = cvalues.shape[0]
        s, t, m = self._pooled(n)
        _check(lib().ss2_cambi_topk(self._h, self._dev(cvalues, torch.float32), n, k,
                                    s.ctypes.data, t.ctypes.data, m.ctypes.data,
                                    _stream_handle(stream)))
        return self._result(s, t, m)

    def pool(self, levels, k: int, mask=None, stream=None):
        """c-values and top-K in one call: as topk()."""
        import torch
        n = levels.shape[0]
        s, t, m = self._pooled(n)
        _check(lib().ss2_cambi_pool(self._h, self._dev(levels, torch.uint16),
                                    None if mask is None else self._dev(mask, torch.uint8), n, k,
                                    s.ctypes.data, t.ctypes.data, m.ctypes.data,
                                    _stream_handle(stream)))
        return self._result(s, t, m)


class MSSSIM(_Context):
    """MS-SSIM for one frame geometry (ss2_msssim_create_ex): of the luma
    plane, and with enable_chroma=True of the Cb and Cr planes too."""

    _PREFIX = "ss2_msssim"
    KERNELS = ("k_msssim_level", "k_msssim_final")

    SCALES = 5

    def __init__(self, width: int, height: int, bitdepth: int, chroma: int, batch: int = 0,
                 enable_chroma: bool = False):
        h = lib().ss2_msssim_create_ex(width, height, bitdepth, chroma, batch,
                                       1 if enable_chroma else 0)
        if not h:
            code, msg = last_error()
            raise SS2Error(code, msg)
        self._h = h
        self.width, self.height, self.chroma = width, height, chroma
        self.planes = int(lib().ss2_msssim_planes(h))

    def _dims(self, plane: int = 0):
        w, h = self.width, self.height
        if plane:
            sx, sy = {420: (1, 1), 422: (1, 0), 444: (0, 0)}[self.chroma]
            w, h = (w + sx) >> sx, (h + sy) >> sy
        out = []
        for _ in range(self.SCALES):
            out.append((w, h))
            w, h = (w + 1) // 2, (h + 1) // 2
        return out

    def score(self, ref, dis, stream=None, values: bool = False):
        """Scores (n,) for the luma plane alone, (n, 3) with the chroma planes
        (Y, Cb, Cr); with values=True also the per-scale means (n, 5, 5) or
        (n, 3, 5, 5): l, c, s, cs, l cs."""
        import torch
        for t in (ref, dis):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
                raise TypeError("frames must be contiguous CUDA tensors")
        n, p = ref.shape[0], self.planes
        out = np.zeros((n, p), np.float64)
        v = np.zeros((n, p, self.SCALES, 5), np.float64) if values else None
        _check(lib().ss2_msssim_score(self._h, ref.data_ptr(), dis.data_ptr(), n, out.ctypes.data,
                                      v.ctypes.data if values else None, _stream_handle(stream)))
        if p == 1:
            out = out[:, 0]
            v = v[:, 0] if values else None
        return (out, v) if values else out

    def pyramid(self, ref, dis, stream=None, plane: int = 0):
        """Scales 2..5 of one plane of the first frame pair: ([ref planes],
        [dis planes])."""
        dims = self._dims(plane)[1:]
        total = sum(w * h for w, h in dims)
        buf = np.zeros(2 * total, np.float32)
        _check(lib().ss2_msssim_debug_pyramid_plane(self._h, ref.data_ptr(), dis.data_ptr(),
                                                    plane, buf.ctypes.data,
                                                    _stream_handle(stream)))
        out, off = [], 0
        for _ in range(2):
            planes = []
            for w, h in dims:
                planes.append(buf[off:off + w * h].reshape(h, w))
                off += w * h
            out.append(planes)
        return out[0], out[1]


class Scorer(_Context):
    """A scoring context for one frame geometry (ss2_create)."""

    _PREFIX = "ss2"
    KERNELS = ("k_pyramid", "k_hblur", "k_vblur", "k_finalize")

    def __init__(self, width: int, height: int, bitdepth: int, chroma: int,
                 batch: int | None = None, params: np.ndarray | None = None):
        L = lib()
        if batch is None:
            h = L.ss2_create(width, height, bitdepth, chroma)
        else:
            h = L.ss2_create_batch(width, height, bitdepth, chroma, batch)
        if not h:
            code, msg = last_error()
            raise SS2Error(code, msg)
        self._h = h
        self.width, self.height, self.bitdepth, self.chroma = width, height, bitdepth, chroma
        if params is not None:
            self.set_params(params)

    # -- properties --------------------------------------------------------
    @property
    def handle(self) -> int:
        if not self._h:
            raise SS2Error(EINVAL, "context is closed")
        return self._h

    @property
    def frame_bytes(self) -> int:
        return int(lib().ss2_frame_bytes(self.handle))

    @property
    def batch(self) -> int:
        return int(lib().ss2_batch(self.handle))

    @property
    def workspace_bytes(self) -> int:
        return int(lib().ss2_workspace_bytes(self.handle))

    def set_params(self, params: np.ndarray) -> None:
        p = np.ascontiguousarray(params, np.float64)
        _check(lib().ss2_set_params(self.handle, p.ctypes.data, p.size))

    def set_graphs(self, enable: bool) -> None:
        """Replays repeated device-input calls from a captured CUDA graph, or
        launches every kernel one by one (the default)."""
        _check(lib().ss2_set_graphs(self.handle, 1 if enable else 0))

    # -- scoring -----------------------------------------------------------
    def _frames(self, t) -> int:
        import torch
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError("frames must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError("frames must be contiguous")
        nbytes = t.numel() * t.element_size()
        fb = self.frame_bytes
        if nbytes % fb:
            raise ValueError(f"{nbytes} bytes is not a whole number of {fb}-byte frames")
        return nbytes // fb

    def score(self, ref, dis, stream=None) -> np.ndarray:
        """Scores device-resident frames; returns float64 scores on the host."""
        n = self._frames(ref)
        if self._frames(dis) != n:
            raise ValueError("ref and dis hold different frame counts")
        out = np.zeros(n, np.float64)
        _check(lib().ss2_score_frames(self.handle, ref.data_ptr(), dis.data_ptr(), n,
                                      out.ctypes.data, _stream_handle(stream)))
        return out

    def values(self, ref, dis, stream=None) -> tuple[np.ndarray, np.ndarray]:
        """Scores and the 108 pooled values per frame."""
        n = self._frames(ref)
        if self._frames(dis) != n:
            raise ValueError("ref and dis hold different frame counts")
        vals = np.zeros((n, NVALUES), np.float64)
        sc = np.zeros(n, np.float64)
        _check(lib().ss2_values(self.handle, ref.data_ptr(), dis.data_ptr(), n,
                                vals.ctypes.data, sc.ctypes.data, _stream_handle(stream)))
        return vals, sc

    def score_host(self, ref: np.ndarray, dis: np.ndarray, stream=None) -> np.ndarray:
        """Scores frames held in host memory (pinned memory overlaps the upload)."""
        import torch
        def _ptr_bytes(a):
            if isinstance(a, torch.Tensor):
                if a.is_cuda or not a.is_contiguous():
                    raise ValueError("host frames must be a contiguous CPU tensor or array")
                return a.data_ptr(), a.numel() * a.element_size()
            a = np.ascontiguousarray(a)
            return a.ctypes.data, a.nbytes
        pr, nr = _ptr_bytes(ref)
        pd, nd = _ptr_bytes(dis)
        fb = self.frame_bytes
        if nr != nd or nr % fb:
            raise ValueError("ref/dis must hold the same whole number of frames")
        n = nr // fb
        out = np.zeros(n, np.float64)
        _check(lib().ss2_score_frames_host(self.handle, pr, pd, n, out.ctypes.data,
                                           _stream_handle(stream)))
        return out

    def debug_planes(self, ref, dis, scale: int, stream=None):
        """XYB planes (6, hs, ws) and horizontally blurred planes (15, hs, ws)
        of one scale for the first frame pair."""
        ws, hs = self.width, self.height
        for _ in range(scale):
            ws, hs = (ws + 1) // 2, (hs + 1) // 2
        xyb = np.zeros((6, hs, ws), np.float32)
        hb = np.zeros((15, hs, ws), np.float32)
        _check(lib().ss2_debug_planes(self.handle, ref.data_ptr(), dis.data_ptr(), scale,
                                      xyb.ctypes.data, hb.ctypes.data, _stream_handle(stream)))
        return xyb, hb

    def debug_linear(self, ref, dis, scale: int, stream=None):
        """Linear RGB planes (6, hs, ws) of one scale for the first frame pair,
        as the pyramid kernel forms them (ref R, G, B then dis R, G, B)."""
        ws, hs = self.width, self.height
        for _ in range(scale):
            ws, hs = (ws + 1) // 2, (hs + 1) // 2
        lin = np.zeros((6, hs, ws), np.float32)
        _check(lib().ss2_debug_linear(self.handle, ref.data_ptr(), dis.data_ptr(), scale,
                                      lin.ctypes.data, _stream_handle(stream)))
        return lin


