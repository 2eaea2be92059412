"""Python access to the C oracle (``ss2_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The CUDA library and its
Python binding never import this package.

``build()`` compiles the oracle with contraction off into ``oracle/_build``;
``lib()`` loads it.  The wrappers below marshal numpy arrays only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
SO_PATH = os.path.join(BUILD_DIR, "libss2_oracle.so")
SOURCES = [os.path.join(HERE, "ss2_oracle.c"), os.path.join(HERE, "fssim_oracle.c"),
           os.path.join(HERE, "msssim_oracle.c"), os.path.join(HERE, "cambi_oracle.c")]
HEADERS = [os.path.join(HERE, "ss2_oracle.h")]

NPARAMS = 133
NVALUES = 108
EOTF_N = 4096
P_WEIGHTS, P_POLY, P_POWER, P_OPSIN, P_BIAS, P_AFFINE, P_C2 = 0, 108, 112, 115, 124, 127, 132

CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None

# Tests that plant a mistake in a copy of the oracle point this at the copy's
# build; nothing else sets it.
SO_OVERRIDE_ENV = "SS2_ORACLE_SO"


def _stale() -> bool:
    if not os.path.exists(SO_PATH):
        return True
    t = os.path.getmtime(SO_PATH)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS)


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, contraction off)."""
    if force or _stale():
        os.makedirs(BUILD_DIR, exist_ok=True)
        tmp = SO_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-shared", "-o", tmp, *SOURCES, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, SO_PATH)
    return SO_PATH


class Dump(ctypes.Structure):
    _fields_ = [
        ("scale", ctypes.c_int),
        ("lin", ctypes.c_void_p),
        ("xyb", ctypes.c_void_p),
        ("hblur", ctypes.c_void_p),
        ("blur", ctypes.c_void_p),
        ("terms", ctypes.c_void_p),
        ("sums", ctypes.c_void_p),
    ]


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get(SO_OVERRIDE_ENV)
            if not path:
                path = build()
            L = ctypes.CDLL(path)
            vp, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            L.ss2o_default_params.argtypes = [vp]
            L.ss2o_score.argtypes = [vp, vp, i, i, i, i, vp, vp, vp, ctypes.POINTER(Dump)]
            L.ss2o_score.restype = i
            L.ss2o_score_frames.argtypes = [vp, vp, i, i, i, i, i, vp, vp, vp]
            L.ss2o_score_frames.restype = i
            L.ss2o_frame_bytes.argtypes = [i, i, i, i]
            L.ss2o_frame_bytes.restype = ctypes.c_size_t
            L.ss2o_scale_dims.argtypes = [i, i, vp, vp]
            L.ss2o_scale_dims.restype = i
            L.ss2o_cbrtf_cr.argtypes = [ctypes.c_float]
            L.ss2o_cbrtf_cr.restype = ctypes.c_float
            L.ss2o_cbrtf_cr_array.argtypes = [vp, vp, ctypes.c_longlong]
            L.ss2o_eotf_table.argtypes = [vp]
            L.ss2o_eotf_lookup.argtypes = [vp, ctypes.c_float]
            L.ss2o_eotf_lookup.restype = ctypes.c_float
            L.ss2o_yuv_coeffs.argtypes = [vp]
            L.ss2o_iir_coeffs.argtypes = [vp, vp, vp]
            L.ss2o_xyb_pixel.argtypes = [vp, ctypes.c_float, ctypes.c_float, ctypes.c_float, vp]
            L.ss2o_fssim_scale.argtypes = [i, i]
            L.ss2o_fssim_scale.restype = i
            L.ss2o_fssim_dims.argtypes = [i, i, vp, vp]
            L.ss2o_fssim_dims.restype = i
            L.ss2o_fssim_decimate.argtypes = [vp, i, i, i, vp]
            L.ss2o_fssim_decimate.restype = i
            L.ss2o_fssim.argtypes = [vp, vp, i, i, i, vp, vp, vp]
            L.ss2o_fssim.restype = i
            L.ss2o_cambi_recip.argtypes = [i]
            L.ss2o_cambi_recip.restype = ctypes.c_float
            L.ss2o_cambi_cvalues.argtypes = [vp, vp, i, i, i, i, vp, vp, vp]
            L.ss2o_cambi_cvalues.restype = i
            L.ss2o_cambi_cvalue_at.argtypes = [vp, vp, i, i, i, i, vp, vp, i, i, vp]
            L.ss2o_cambi_cvalue_at.restype = i
            L.ss2o_cambi_topk.argtypes = [vp, ctypes.c_long, ctypes.c_long, vp, vp, vp, vp]
            L.ss2o_cambi_topk.restype = i
            L.ss2o_msssim_dims.argtypes = [i, i, vp]
            L.ss2o_msssim_dims.restype = None
            L.ss2o_msssim_pyramid_len.argtypes = [i, i]
            L.ss2o_msssim_pyramid_len.restype = ctypes.c_size_t
            L.ss2o_msssim_pyramid.argtypes = [vp, i, i, i, vp]
            L.ss2o_msssim_pyramid.restype = i
            L.ss2o_msssim.argtypes = [vp, vp, i, i, i, vp, vp]
            L.ss2o_msssim.restype = i
            L.ss2o_msssim_planes.argtypes = [vp, vp, i, i, i, i, i, vp, vp]
            L.ss2o_msssim_planes.restype = i
            L.ss2o_blur_line.argtypes = [vp, i, vp]
            L.ss2o_downsample.argtypes = [vp, i, i, vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def default_params() -> np.ndarray:
    p = np.zeros(NPARAMS, np.float64)
    lib().ss2o_default_params(_ptr(p))
    return p


def frame_bytes(w: int, h: int, depth: int, chroma: int) -> int:
    return int(lib().ss2o_frame_bytes(w, h, depth, chroma))


def scale_dims(w: int, h: int) -> list[tuple[int, int]]:
    ws = np.zeros(6, np.int32)
    hs = np.zeros(6, np.int32)
    n = lib().ss2o_scale_dims(w, h, _ptr(ws), _ptr(hs))
    return [(int(ws[k]), int(hs[k])) for k in range(n)]


def score(ref: np.ndarray, dis: np.ndarray, w: int, h: int, depth: int,
          chroma: int, params: np.ndarray | None = None, dump_scale: int | None = None):
    """Scores one frame pair.  Returns (score, values[108], dump dict or None)."""
    params = default_params() if params is None else np.ascontiguousarray(params, np.float64)
    ref = np.ascontiguousarray(ref)
    dis = np.ascontiguousarray(dis)
    fb = frame_bytes(w, h, depth, chroma)
    assert ref.nbytes == fb and dis.nbytes == fb, (ref.nbytes, fb)
    sc = np.zeros(1, np.float64)
    vals = np.zeros(NVALUES, np.float64)
    dump = None
    dptr = None
    if dump_scale is not None:
        dims = scale_dims(w, h)
        if dump_scale < len(dims):
            sw, sh = dims[dump_scale]
        else:
            sw, sh = 1, 1
        ns = sw * sh
        dump = {
            "lin": np.zeros((6, sh, sw), np.float32),
            "xyb": np.zeros((6, sh, sw), np.float32),
            "hblur": np.zeros((15, sh, sw), np.float32),
            "blur": np.zeros((15, sh, sw), np.float32),
            "terms": np.zeros((18, sh, sw), np.float64),
            "sums": np.zeros(18, np.float64),
        }
        d = Dump(dump_scale, *(dump[k].ctypes.data for k in
                               ("lin", "xyb", "hblur", "blur", "terms", "sums")))
        dptr = ctypes.byref(d)
        _ = ns
    rc = lib().ss2o_score(_ptr(ref), _ptr(dis), w, h, depth, chroma, _ptr(params),
                          _ptr(sc), _ptr(vals), dptr)
    if rc != 0:
        raise ValueError(f"oracle rejected geometry {w}x{h} depth {depth} chroma {chroma}: rc={rc}")
    return float(sc[0]), vals, dump


def score_frames(ref: np.ndarray, dis: np.ndarray, w: int, h: int, depth: int,
                 chroma: int, params: np.ndarray | None = None):
    """Scores n packed frames; ref/dis shaped (n, frame_elems).  Returns (scores, values)."""
    params = default_params() if params is None else np.ascontiguousarray(params, np.float64)
    ref = np.ascontiguousarray(ref)
    dis = np.ascontiguousarray(dis)
    n = ref.shape[0]
    sc = np.zeros(n, np.float64)
    vals = np.zeros((n, NVALUES), np.float64)
    rc = lib().ss2o_score_frames(_ptr(ref), _ptr(dis), n, w, h, depth, chroma,
                                 _ptr(params), _ptr(sc), _ptr(vals))
    if rc != 0:
        raise ValueError(f"oracle rejected geometry: rc={rc}")
    return sc, vals


def cbrtf_cr(x: float) -> float:
    return float(lib().ss2o_cbrtf_cr(ctypes.c_float(x)))


def cbrtf_cr_array(x: np.ndarray, threads: int | None = None) -> np.ndarray:
    """The oracle's cube root over a float32 array, split across threads
    (ctypes releases the GIL during the call)."""
    import concurrent.futures as cf
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty_like(x)
    L = lib()
    nt = max(1, threads or os.cpu_count() or 1)
    bounds = np.linspace(0, x.size, nt + 1, dtype=np.int64)

    def run(k):
        a, b = int(bounds[k]), int(bounds[k + 1])
        if b > a:
            L.ss2o_cbrtf_cr_array(x.ctypes.data + 4 * a, out.ctypes.data + 4 * a, b - a)

    with cf.ThreadPoolExecutor(max_workers=nt) as ex:
        list(ex.map(run, range(nt)))
    return out


def eotf_table() -> np.ndarray:
    t = np.zeros(EOTF_N + 1, np.float32)
    lib().ss2o_eotf_table(_ptr(t))
    return t


def eotf_lookup(v: float) -> float:
    t = eotf_table()
    return float(lib().ss2o_eotf_lookup(_ptr(t), ctypes.c_float(v)))


def yuv_coeffs() -> np.ndarray:
    k = np.zeros(4, np.float32)
    lib().ss2o_yuv_coeffs(_ptr(k))
    return k


def xyb_pixel(r: float, g: float, b: float, params: np.ndarray | None = None) -> np.ndarray:
    params = default_params() if params is None else np.ascontiguousarray(params, np.float64)
    out = np.zeros(3, np.float32)
    lib().ss2o_xyb_pixel(_ptr(params), ctypes.c_float(r), ctypes.c_float(g), ctypes.c_float(b),
                         _ptr(out))
    return out


def fssim_scale(w: int, h: int) -> int:
    return int(lib().ss2o_fssim_scale(w, h))


def fssim_dims(w: int, h: int) -> tuple[int, int, int]:
    """(factor, decimated width, decimated height)."""
    wd = np.zeros(1, np.int32)
    hd = np.zeros(1, np.int32)
    s = lib().ss2o_fssim_dims(w, h, _ptr(wd), _ptr(hd))
    return int(s), int(wd[0]), int(hd[0])


def fssim_decimate(frame: np.ndarray, w: int, h: int, depth: int) -> np.ndarray:
    """The decimated luma plane of one frame (float32, hd x wd)."""
    s, wd, hd = fssim_dims(w, h)
    out = np.zeros((hd, wd), np.float32)
    f = np.ascontiguousarray(frame)
    rc = lib().ss2o_fssim_decimate(_ptr(f), w, h, depth, _ptr(out))
    if rc != 0:
        raise ValueError(f"fssim decimation rejected: rc={rc}")
    return out


def fssim(ref: np.ndarray, dis: np.ndarray, w: int, h: int, depth: int):
    """(score, decimated ref plane, decimated dis plane) of one frame pair."""
    s, wd, hd = fssim_dims(w, h)
    a = np.zeros((hd, wd), np.float32)
    b = np.zeros((hd, wd), np.float32)
    sc = np.zeros(1, np.float64)
    rc = lib().ss2o_fssim(_ptr(np.ascontiguousarray(ref)), _ptr(np.ascontiguousarray(dis)),
                          w, h, depth, _ptr(sc), _ptr(a), _ptr(b))
    if rc != 0:
        raise ValueError(f"fssim rejected {w}x{h}: rc={rc}")
    return float(sc[0]), a, b


def cambi_recip(n: int) -> float:
    return float(lib().ss2o_cambi_recip(n))


def cambi_cvalues(levels: np.ndarray, window: int, diffs, weights, mask=None) -> np.ndarray:
    """c-values of one level plane (h x w uint16 levels below 1024)."""
    lv = np.ascontiguousarray(levels, dtype=np.uint16)
    h, w = lv.shape
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    d = np.ascontiguousarray(diffs, dtype=np.int32)
    wt = np.ascontiguousarray(weights, dtype=np.int32)
    out = np.zeros((h, w), np.float32)
    rc = lib().ss2o_cambi_cvalues(_ptr(lv), _ptr(m), w, h, window, len(d), _ptr(d), _ptr(wt),
                                  _ptr(out))
    if rc != 0:
        raise ValueError(f"cambi c-values rejected: rc={rc}")
    return out


def cambi_cvalue_at(levels: np.ndarray, window: int, diffs, weights, points, mask=None):
    """c-values of the listed (y, x) pixels of one level plane, one by one."""
    lv = np.ascontiguousarray(levels, dtype=np.uint16)
    h, w = lv.shape
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    d = np.ascontiguousarray(diffs, dtype=np.int32)
    wt = np.ascontiguousarray(weights, dtype=np.int32)
    out = np.zeros(1, np.float32)
    res = []
    for (y, x) in points:
        rc = lib().ss2o_cambi_cvalue_at(_ptr(lv), _ptr(m), w, h, window, len(d), _ptr(d),
                                        _ptr(wt), int(x), int(y), _ptr(out))
        if rc != 0:
            raise ValueError(f"cambi c-value rejected: rc={rc}")
        res.append(float(out[0]))
    return np.array(res, np.float32)


def cambi_topk(c: np.ndarray, k: int):
    """(exact sum in units of 2^-24 as a Python int, k-th largest value, mean)."""
    cc = np.ascontiguousarray(c, dtype=np.float32).ravel()
    lo = np.zeros(1, np.uint64)
    hi = np.zeros(1, np.uint64)
    t = np.zeros(1, np.float32)
    mean = np.zeros(1, np.float64)
    rc = lib().ss2o_cambi_topk(_ptr(cc), cc.size, k, _ptr(lo), _ptr(hi), _ptr(t), _ptr(mean))
    if rc != 0:
        raise ValueError(f"cambi top-k rejected: rc={rc}")
    return (int(hi[0]) << 64) | int(lo[0]), float(t[0]), float(mean[0])


MSSSIM_SCALES = 5
MSSSIM_BETA = (0.0448, 0.2856, 0.3001, 0.2363, 0.1333)


def msssim_dims(w: int, h: int) -> list[tuple[int, int]]:
    d = np.zeros(2 * MSSSIM_SCALES, np.int32)
    lib().ss2o_msssim_dims(w, h, _ptr(d))
    return [(int(d[2 * j]), int(d[2 * j + 1])) for j in range(MSSSIM_SCALES)]


def msssim_pyramid(frame: np.ndarray, w: int, h: int, depth: int) -> list[np.ndarray]:
    """The five luma levels of one frame (float64, h_j x w_j each)."""
    dims = msssim_dims(w, h)
    buf = np.zeros(int(lib().ss2o_msssim_pyramid_len(w, h)), np.float64)
    rc = lib().ss2o_msssim_pyramid(_ptr(np.ascontiguousarray(frame)), w, h, depth, _ptr(buf))
    if rc != 0:
        raise ValueError(f"msssim pyramid rejected: rc={rc}")
    out, off = [], 0
    for (wj, hj) in dims:
        out.append(buf[off:off + wj * hj].reshape(hj, wj))
        off += wj * hj
    return out


def msssim(ref: np.ndarray, dis: np.ndarray, w: int, h: int, depth: int):
    """(score, values[5][5]) of one frame pair: per scale the means of
    l, c, s, cs and l cs."""
    sc = np.zeros(1, np.float64)
    v = np.zeros((MSSSIM_SCALES, 5), np.float64)
    rc = lib().ss2o_msssim(_ptr(np.ascontiguousarray(ref)), _ptr(np.ascontiguousarray(dis)),
                           w, h, depth, _ptr(sc), _ptr(v))
    if rc != 0:
        raise ValueError(f"msssim rejected {w}x{h}: rc={rc}")
    return float(sc[0]), v


def iir_coeffs():
    a = np.zeros(3, np.float64)
    c2 = np.zeros(3, np.float32)
    g = np.zeros(3, np.float32)
    lib().ss2o_iir_coeffs(_ptr(a), _ptr(c2), _ptr(g))
    return a, c2, g


def blur_line(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.zeros_like(x)
    lib().ss2o_blur_line(_ptr(x), x.size, _ptr(out))
    return out


def downsample(plane: np.ndarray) -> np.ndarray:
    plane = np.ascontiguousarray(plane, np.float32)
    h, w = plane.shape
    out = np.zeros(((h + 1) // 2, (w + 1) // 2), np.float32)
    lib().ss2o_downsample(_ptr(plane), w, h, _ptr(out))
    return out


def msssim_planes(ref: np.ndarray, dis: np.ndarray, w: int, h: int, depth: int, chroma: int,
                  nplanes: int = 3):
    """(scores[nplanes], values[nplanes][5][5]) of one packed frame pair: MS-SSIM
    of the luma plane and, with nplanes = 3, of Cb and Cr at chroma resolution."""
    sc = np.zeros(nplanes, np.float64)
    v = np.zeros((nplanes, MSSSIM_SCALES, 5), np.float64)
    rc = lib().ss2o_msssim_planes(_ptr(np.ascontiguousarray(ref)), _ptr(np.ascontiguousarray(dis)),
                                  w, h, depth, chroma, nplanes, _ptr(sc), _ptr(v))
    if rc != 0:
        raise ValueError(f"msssim planes rejected {w}x{h} chroma {chroma}: rc={rc}")
    return sc, v
