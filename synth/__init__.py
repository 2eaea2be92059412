"""Seeded synthetic YUV frame pairs.

This module holds the input recipes only — none of the metric's arithmetic —
and is the one piece of Python shared by the oracle-side tests and the CUDA
side.  The five workloads stand in for the fixtures the source pages measure
on ("Research-1363 ...", section "Sources": the Netflix 576x324 pair, an
853x481 4:4:4 rescale, Big Buck Bunny 3840x2160), which are not available:
same shapes, frame counts, bit depths and chroma layouts, with seeded content.

Frames are packed planar (Y, then U, then V, no padding); 8-bit samples are
uint8, deeper ones little-endian uint16.  ``make(name)`` returns a
``Workload`` whose ``ref``/``dis`` arrays are shaped (n_frames, frame_elems).

Randomness: numpy PCG64 streams keyed by (config seed, frame, plane, stream),
so any subset of frames can be generated on its own and every frame is the
same whichever subset is asked for.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Spec:
    name: str
    width: int
    height: int
    depth: int
    chroma: int
    frames: int
    seed: int
    about: str


SPECS = {
    "c0_576x324_8b_420": Spec("c0_576x324_8b_420", 576, 324, 8, 420, 4, 0,
                              "8 drifting sinusoids + U(+-8); dis = ref + N(0, 3^2)"),
    "c1_853x481_8b_444": Spec("c1_853x481_8b_444", 853, 481, 8, 444, 48, 1,
                              "as c0; dis: frame 0 identical, then 8x8 block quantisation "
                              "(DC step 12), N(0, 5^2), 3x3 box blur in turn"),
    "c2_1920x1080_10b_420": Spec("c2_1920x1080_10b_420", 1920, 1080, 10, 420, 48, 2,
                                 "gradients + sinusoids + U(+-32) in 64-940; "
                                 "dis = ref + N(0, s^2), s = 2, 8, 16 in turn"),
    "c3_3840x2160_8b_420": Spec("c3_3840x2160_8b_420", 3840, 2160, 8, 420, 50, 3,
                                "sinusoids, 64x64 tiles: 30% U(+-40) texture, 20% of the rest "
                                "flat; dis = 4x4 block means + N(0, 4^2)"),
    "c4_3840x2160_12b_444": Spec("c4_3840x2160_12b_444", 3840, 2160, 12, 444, 16, 4,
                                 "sinusoids over 0-4095 + U(+-64); dis: identical, +100 shift, "
                                 "Gaussian blur sigma 1, N(0, 40^2) in turn"),
}
ORDER = list(SPECS)


@dataclass
class Workload:
    spec: Spec
    frames: list[int]
    ref: np.ndarray
    dis: np.ndarray

    @property
    def frame_bytes(self) -> int:
        return self.ref.shape[1] * self.ref.itemsize


def chroma_dims(w: int, h: int, chroma: int) -> tuple[int, int]:
    sx = 1 if chroma in (420, 422) else 0
    sy = 1 if chroma == 420 else 0
    return (w + sx) >> sx, (h + sy) >> sy


def frame_elems(w: int, h: int, chroma: int) -> int:
    cw, ch = chroma_dims(w, h, chroma)
    return w * h + 2 * cw * ch


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _sinusoids(key: tuple, w: int, h: int, n: int, lo: float, hi: float,
               frame: int) -> np.ndarray:
    """n drifting 2-D sinusoids, periods log-uniform in [4, 128] px, random
    orientation and phase, each phase advancing by 2 pi v / P per frame with
    v ~ U[0.5, 2] px/frame; amplitudes sum to 40% of the range, centred."""
    r = _rng(*key)
    period = np.exp(r.uniform(np.log(4.0), np.log(128.0), n))
    theta = r.uniform(0.0, np.pi, n)
    phase = r.uniform(0.0, 2.0 * np.pi, n)
    speed = r.uniform(0.5, 2.0, n)
    amp = r.uniform(0.5, 1.0, n)
    amp *= 0.4 * (hi - lo) / amp.sum()
    x = np.arange(w, dtype=np.float64)
    y = np.arange(h, dtype=np.float64)
    out = np.full((h, w), 0.5 * (lo + hi), np.float32)
    for i in range(n):
        kx = 2.0 * np.pi * np.cos(theta[i]) / period[i]
        ky = 2.0 * np.pi * np.sin(theta[i]) / period[i]
        ph = phase[i] + 2.0 * np.pi * speed[i] * frame / period[i]
        cx, sx = np.cos(kx * x + ph), np.sin(kx * x + ph)
        cy, sy = np.cos(ky * y), np.sin(ky * y)
        # cos(a + b) = cos a cos b - sin a sin b, as two outer products
        out += (amp[i] * cy)[:, None].astype(np.float32) * cx[None, :].astype(np.float32)
        out -= (amp[i] * sy)[:, None].astype(np.float32) * sx[None, :].astype(np.float32)
    return out


def _gradient(key: tuple, w: int, h: int, span: float) -> np.ndarray:
    r = _rng(*key)
    ang = r.uniform(0.0, 2.0 * np.pi)
    x = np.linspace(-0.5, 0.5, w, dtype=np.float32)
    y = np.linspace(-0.5, 0.5, h, dtype=np.float32)
    return span * (np.float32(np.cos(ang)) * x[None, :] + np.float32(np.sin(ang)) * y[:, None])


def _box3(p: np.ndarray) -> np.ndarray:
    q = np.pad(p.astype(np.int64), 1, mode="edge")
    h, w = p.shape
    s = sum(q[dy:dy + h, dx:dx + w] for dy in range(3) for dx in range(3))
    return (s + 4) // 9


def _block_mean(p: np.ndarray, b: int) -> np.ndarray:
    """Mean of each b x b block (partial blocks at the edges), float64."""
    h, w = p.shape
    hb, wb = -(-h // b), -(-w // b)
    q = np.zeros((hb * b, wb * b), np.float64)
    cnt = np.zeros_like(q)
    q[:h, :w] = p
    cnt[:h, :w] = 1.0
    s = q.reshape(hb, b, wb, b).sum(axis=(1, 3))
    c = cnt.reshape(hb, b, wb, b).sum(axis=(1, 3))
    m = s / c
    return np.repeat(np.repeat(m, b, axis=0), b, axis=1)[:h, :w]


def _gauss_blur(p: np.ndarray, sigma: float, radius: int) -> np.ndarray:
    t = np.arange(-radius, radius + 1, dtype=np.float64)
    k = np.exp(-t * t / (2.0 * sigma * sigma))
    k /= k.sum()
    q = np.pad(p.astype(np.float64), radius, mode="edge")
    h, w = p.shape
    tmp = sum(k[i] * q[:, i:i + w] for i in range(2 * radius + 1))
    return sum(k[i] * tmp[i:i + h, :] for i in range(2 * radius + 1))


def _clamp_round(p: np.ndarray, lo: int, hi: int) -> np.ndarray:
    return np.clip(np.rint(p), lo, hi).astype(np.int64)


def _planes(spec: Spec):
    w, h = spec.width, spec.height
    cw, ch = chroma_dims(w, h, spec.chroma)
    return [(0, w, h), (1, cw, ch), (2, cw, ch)]


def _frame_pair(spec: Spec, f: int) -> tuple[list[np.ndarray], list[np.ndarray]]:
    s = spec.seed
    k = 1 << (spec.depth - 8)
    refs, diss = [], []
    cfg = ORDER.index(spec.name)
    for plane, pw, ph in _planes(spec):
        luma = plane == 0
        nr = _rng(s, f, plane, 1)          # per-frame noise stream
        if cfg in (0, 1):
            lo, hi = 16, (235 if luma else 240)
            base = _sinusoids((s, plane, 0), pw, ph, 8, lo, hi, f)
            ref = _clamp_round(base + nr.integers(-8, 9, (ph, pw)), lo, hi)
            if cfg == 0:
                dis = _clamp_round(ref + nr.normal(0.0, 3.0, (ph, pw)), lo, hi)
            elif f == 0:
                dis = ref.copy()
            elif f % 3 == 0:
                dis = _box3(ref)
            elif f % 3 == 1:
                dis = _clamp_round(12.0 * np.rint(_block_mean(ref, 8) / 12.0), 0, 255)
            else:
                dis = _clamp_round(ref + nr.normal(0.0, 5.0, (ph, pw)), 0, 255)
        elif cfg == 2:
            lo, hi = 64, (940 if luma else 960)
            base = _sinusoids((s, plane, 0), pw, ph, 6, lo, hi, f)
            base = base + _gradient((s, plane, 2, f), pw, ph, 0.3 * (hi - lo))
            ref = _clamp_round(base + nr.integers(-32, 33, (ph, pw)), lo, hi)
            sigma = (2.0, 8.0, 16.0)[f % 3]
            dis = _clamp_round(ref + nr.normal(0.0, sigma, (ph, pw)), 0, 1023)
        elif cfg == 3:
            lo, hi = 16, (235 if luma else 240)
            base = _sinusoids((s, plane, 0), pw, ph, 8, lo, hi, f)
            tile = 64 if luma else 32
            tr = _rng(s, plane, 3)             # tile layout fixed over frames
            ty, tx = -(-ph // tile), -(-pw // tile)
            u = tr.uniform(size=(ty, tx))
            v = tr.uniform(size=(ty, tx))
            textured = u < 0.3
            flat = (~textured) & (v < 0.2)
            tex_mask = np.repeat(np.repeat(textured, tile, 0), tile, 1)[:ph, :pw]
            flat_mask = np.repeat(np.repeat(flat, tile, 0), tile, 1)[:ph, :pw]
            noise = nr.integers(-40, 41, (ph, pw))
            img = np.where(tex_mask, base + noise, base)
            img = np.where(flat_mask, _block_mean(img, tile), img)
            ref = _clamp_round(img, lo, hi)
            dis = _clamp_round(np.rint(_block_mean(ref, 4)) + nr.normal(0.0, 4.0, (ph, pw)), 0, 255)
        else:
            lo, hi = 0, 4095
            base = _sinusoids((s, plane, 0), pw, ph, 8, lo, hi, f)
            ref = _clamp_round(base + nr.integers(-64, 65, (ph, pw)), lo, hi)
            m = f % 4
            if m == 0:
                dis = ref.copy()
            elif m == 1:
                dis = np.clip(ref + 100, 0, 4095)
            elif m == 2:
                dis = _clamp_round(_gauss_blur(ref, 1.0, 3), 0, 4095)
            else:
                dis = _clamp_round(ref + nr.normal(0.0, 40.0, (ph, pw)), 0, 4095)
        del k
        k = 1 << (spec.depth - 8)
        refs.append(ref)
        diss.append(dis)
    return refs, diss


def _packed_pair(name: str, f: int) -> tuple[np.ndarray, np.ndarray]:
    spec = SPECS[name]
    dt = np.uint8 if spec.depth == 8 else np.uint16
    rp, dp = _frame_pair(spec, f)
    return (np.concatenate([p.ravel() for p in rp]).astype(dt),
            np.concatenate([p.ravel() for p in dp]).astype(dt))


def make(name: str, frames: int | list[int] | None = None, workers: int = 0) -> Workload:
    """Generates the named workload.  ``frames``: None (all), a count (the
    first n) or an explicit list of frame indices.  ``workers`` > 1 spreads
    the frames over that many spawned processes (call it before any CUDA
    work in the caller)."""
    spec = SPECS[name]
    if frames is None:
        idx = list(range(spec.frames))
    elif isinstance(frames, int):
        idx = list(range(frames))
    else:
        idx = list(frames)
    dt = np.uint8 if spec.depth == 8 else np.uint16
    fe = frame_elems(spec.width, spec.height, spec.chroma)
    ref = np.empty((len(idx), fe), dt)
    dis = np.empty((len(idx), fe), dt)
    if workers > 1 and len(idx) > 1:
        import concurrent.futures as cf
        import multiprocessing as mp
        with cf.ProcessPoolExecutor(max_workers=min(workers, len(idx)),
                                    mp_context=mp.get_context("spawn")) as ex:
            for j, (r, d) in enumerate(ex.map(_packed_pair, [name] * len(idx), idx)):
                ref[j], dis[j] = r, d
    else:
        for j, f in enumerate(idx):
            ref[j], dis[j] = _packed_pair(name, f)
    return Workload(spec, idx, ref, dis)


def custom(width: int, height: int, depth: int, chroma: int, n_frames: int,
           seed: int, noise: float = 3.0) -> Workload:
    """A small seeded pair of any geometry (sinusoids + uniform noise; dis =
    ref + N(0, noise^2)), full code range of the bit depth."""
    hi = (1 << depth) - 1
    spec = Spec(f"custom_{width}x{height}_{depth}b_{chroma}", width, height, depth,
                chroma, n_frames, seed, "custom")
    cw, ch = chroma_dims(width, height, chroma)
    dt = np.uint8 if depth == 8 else np.uint16
    fe = frame_elems(width, height, chroma)
    ref = np.empty((n_frames, fe), dt)
    dis = np.empty((n_frames, fe), dt)
    amp = hi / 32.0
    for f in range(n_frames):
        rp, dp = [], []
        for plane, pw, ph in [(0, width, height), (1, cw, ch), (2, cw, ch)]:
            nr = _rng(seed, f, plane, 7)
            base = _sinusoids((seed, plane, 5), pw, ph, 6, 0.1 * hi, 0.9 * hi, f)
            r = _clamp_round(base + nr.uniform(-amp, amp, (ph, pw)), 0, hi)
            d = _clamp_round(r + nr.normal(0.0, noise * (1 << (depth - 8)), (ph, pw)), 0, hi)
            rp.append(r)
            dp.append(d)
        ref[f] = np.concatenate([p.ravel() for p in rp]).astype(dt)
        dis[f] = np.concatenate([p.ravel() for p in dp]).astype(dt)
    return Workload(spec, list(range(n_frames)), ref, dis)
