// fssim.cu — float_ssim with decimation on the device (ss2_fssim_* in
// include/ss2.h).
//
// Source: "ADR-1405: float_ssim_hip decimates on the device, bit-identical
// to the CPU" (vmafx documentation), Context and Decision 1 and 4: the
// factor max(1, round(min(w, h) / 256)); a scale x scale box of weight
// 1.0f / (scale * scale) at (x * scale, y * scale), offsets -scale/2 ..
// scale-1-scale/2, symmetric edges, fp32 taps summed exactly in int64 units
// of 2^-52 and rounded once; SSIM with an 11x11 Gaussian on the decimated
// planes; -ENOTSUP for a decimated plane below 11x11 or a factor above 128.
// Samples are taken in the 8-bit range, raw / 2^(depth - 8) (exact), and
// L = 255: only then does a window sum in 2^-52 units fit an int64 at every
// depth, as the page states for 10, 12 and 16 bits.
//
//   k_fssim_decimate  one block per decimated row of one image: 16-byte
//                     loads, vertical column sums in registers, then
//                     horizontal window sums from shared memory.  The window
//                     sum is exact: an int64 count of 2^-52 units (every
//                     nonzero tap, a float product sample * w with sample a
//                     multiple of 2^-8 below 256 and w >= 2^-14, is a
//                     multiple of 2^-45 below 256, so the count stays below
//                     2^61), or for a power-of-two scale, where every tap is
//                     exact, the raw sample sum; one conversion rounds it.
//   k_fssim_map       32x16 map tiles: separable 11-tap Gaussian sums of
//                     x1, x2, x1^2, x2^2, x1 x2 in fp32 as three packed pairs
//                     (fma.rn.f32x2) on samples shifted by a per-tile offset
//                     (variances and covariance do not change, cancellation
//                     does), SSIM per pixel (four vertical outputs per
//                     thread, so one column's 14 loads serve four), fp32
//                     warp sums in a fixed tree and an fp64 sum of the
//                     block's four warps.
//   k_fssim_final     per frame: block sums in a fixed warp order (fp64), mean.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

#include "../../include/ss2.h"
#include "ss2_f32x2.cuh"
#include "ss2_host.h"
#include "ss2_tma.cuh"

#define SS2_API extern "C" __attribute__((visibility("default")))

namespace {

using namespace ss2;

constexpr int kWin = 11;                   // Gaussian window
constexpr int kTileX = 32, kTileY = 16;    // map outputs per block
constexpr int kInX = kTileX + kWin - 1;    // input tile (42 x 26)
constexpr int kInY = kTileY + kWin - 1;
constexpr int kMapThreads = 128;           // 4 warps: 4 vertical outputs per thread

struct FGeom {
  int w, h, depth, bps, scale, wd, hd, pitch;
  long long frame_bytes, plane;          // plane = pitch * hd floats
  int ow, oh, tiles_x, tiles_y;          // map outputs ("valid") and tiles
  float wt;                              // RN(1 / scale^2)
  float norm;                            // 2^(8 - depth): samples in the 8-bit range
  float c;                               // wt * norm (exact: norm is a power of two)
  int pow2;                              // scale is a power of two
  // staged decimation: rows of a band copied to shared memory rg at a time,
  // ng groups per band; staged = 1 k_fssim_decimate_tma, 2 k_fssim_decimate_u8
  int staged, rg, ng, grid_staged;
  long long row_bytes;
  unsigned col_bytes, stage_bytes, smem_staged;
  float C1, C2;
  float gauss[kWin];
};

// Symmetric extension with the edge sample repeated (-1 -> 0, n -> n-1).
// One reflection suffices: a window overshoots an edge by at most scale/2
// samples and a plane that passes the 11x11 check spans more than 10 scales.
__device__ __forceinline__ int mirror1(int i, int n) {
  return i < 0 ? -1 - i : (i >= n ? 2 * n - 1 - i : i);
}

// Exact count of 2^-52 units in the fp32 tap RN(raw * c), c = RN(1/s^2) *
// 2^(8 - depth): a nonzero tap is m * 2^(e - 150) (m the 24-bit significand,
// e the biased exponent) with e >= 105 (tap >= 2^-22) and e <= 134
// (tap < 256), so its count is m << (e - 98) < 2^61.
__device__ __forceinline__ unsigned long long tap_units(unsigned raw, float c) {
  const unsigned b = __float_as_uint(__fmul_rn((float)raw, c));
  if (b == 0u) return 0ull;
  const unsigned long long m = (b & 0x7FFFFFu) | 0x800000u;
  return m << ((b >> 23) - 98u);
}

// One block per (decimated row y, image, frame).
// Pass 1: each thread takes 16-byte column chunks of the band's `scale`
// input rows (mirrored row indices; 16-byte loads when the frame and its
// rows are 16-byte aligned) and sums every column vertically: raw samples
// when the scale is a power of two (each tap raw * 2^-2k * 2^(8 - depth) is
// then exact, so the exact tap sum is the raw sum times that power of two,
// below 2^30), otherwise tap_units counts (below 2^61 per window).
// Pass 2: each output adds `scale` column sums (mirrored column indices) and
// rounds once to fp32.
template <int BPS, bool POW2>
__global__ void __launch_bounds__(256, POW2 ? 4 : 2)
    k_fssim_decimate(FGeom g, const uint8_t *__restrict__ ref, const uint8_t *__restrict__ dis,
                     float *__restrict__ D) {
  using Acc = typename std::conditional<POW2, unsigned, unsigned long long>::type;
  extern __shared__ __align__(128) unsigned char fssim_smem[];
  Acc *col = reinterpret_cast<Acc *>(fssim_smem);
  constexpr int kCW = 16 / BPS;  // columns per 16-byte chunk
  const int y = blockIdx.x, img = blockIdx.y, frame = blockIdx.z;
  const uint8_t *f = (img ? dis : ref) + (long long)frame * g.frame_bytes;
  const int s = g.scale, lo = -(s / 2);
  const long long row_bytes = (long long)g.w * BPS;
  const bool vec = ((reinterpret_cast<uintptr_t>(f) | (uintptr_t)row_bytes) & 15u) == 0;
  const int chunks = (g.w + kCW - 1) / kCW;  // exact when vec (rows are whole chunks)
  for (int q = threadIdx.x; q < chunks; q += blockDim.x) {
    Acc acc[kCW];
#pragma unroll
    for (int k = 0; k < kCW; ++k) acc[k] = 0;
#pragma unroll 4
    for (int j = 0; j < s; ++j) {
      const uint8_t *row = f + (long long)mirror1(y * s + lo + j, g.h) * row_bytes;
      unsigned v[kCW];
      if (vec) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(row) + q);
        const unsigned wd4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < kCW; ++k)
          v[k] = BPS == 1 ? (wd4[k >> 2] >> (8 * (k & 3))) & 0xFFu
                          : (wd4[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
      } else {
#pragma unroll
        for (int k = 0; k < kCW; ++k) {
          const int x = q * kCW + k;
          v[k] = x >= g.w ? 0u
                 : BPS == 1 ? (unsigned)__ldg(row + x)
                            : (unsigned)__ldg(reinterpret_cast<const uint16_t *>(row) + x);
        }
      }
#pragma unroll
      for (int k = 0; k < kCW; ++k) {
        if constexpr (POW2) acc[k] += v[k];
        else acc[k] += tap_units(v[k], g.c);
      }
    }
#pragma unroll
    for (int k = 0; k < kCW; ++k) {
      const int x = q * kCW + k;
      if (x < g.w) col[x] = acc[k];
    }
  }
  __syncthreads();
  float *out = D + (long long)frame * 2 * g.plane + (long long)img * g.plane +
               (long long)y * g.pitch;
  for (int x = threadIdx.x; x < g.wd; x += blockDim.x) {
    Acc sum = 0;
#pragma unroll 4
    for (int i = 0; i < s; ++i) sum += col[mirror1(x * s + lo + i, g.w)];
    if constexpr (POW2)
      out[x] = __fmul_rn(__uint2float_rn(sum), g.c);        // times 2^-n: exact
    else
      out[x] = __fmul_rn(__ull2float_rn(sum), 1.0f / 4503599627370496.0f);  // times 2^-52
  }
}

// The staged form of k_fssim_decimate for frames whose rows are whole
// 16-byte chunks: a persistent loop over (band, image, frame) items; each
// band's `scale` rows (mirrored indices) arrive in shared memory by bulk
// copies, rg rows per group, into two stages, so the copies of the unit after
// next are in flight while a unit is summed.  The sums are those of
// k_fssim_decimate: column sums in shared memory (partial across groups),
// then each output adds `scale` of them and rounds once.  The column sums
// are double-buffered by item parity (one barrier per unit) and padded by
// one word per 16 columns (no bank conflicts between the threads' chunks).
// Every wait is bounded; on a timeout the block raises kErrTmaTimeout in
// err, waits (again bounded) for its copies and returns.
template <int BPS, bool POW2>
__global__ void __launch_bounds__(256)
    k_fssim_decimate_tma(FGeom g, const uint8_t *__restrict__ ref,
                         const uint8_t *__restrict__ dis, float *__restrict__ D, int nb,
                         int *__restrict__ err) {
  using Acc = typename std::conditional<POW2, unsigned, unsigned long long>::type;
  extern __shared__ __align__(128) unsigned char fssim_smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(fssim_smem);           // 2 barriers
  Acc *col2 = reinterpret_cast<Acc *>(fssim_smem + 128);              // 2 column-sum buffers
  unsigned char *stage0 = fssim_smem + 128 + 2 * (size_t)g.col_bytes;
  const int col_stride = (int)(g.col_bytes / sizeof(Acc));
  auto cpad = [](int c) { return c + (c >> 4); };                    // padded column index
  constexpr int kCW = 16 / BPS;
  const int t = threadIdx.x;
  const int s = g.scale, lo = -(s / 2);
  const int n_items = nb * 2 * g.hd;
  const int chunks = (int)(g.row_bytes / 16);

  // unit u of this block -> (item, group); item < 0 when past the end
  auto unit = [&](int u, int &grp) {
    const long long it = blockIdx.x + (long long)(u / g.ng) * gridDim.x;
    grp = u % g.ng;
    return it < n_items ? (int)it : -1;
  };
  auto issue = [&](int u) {
    int grp;
    const int it = unit(u, grp);
    if (it < 0) return;
    const int frame = it / (2 * g.hd), img = (it / g.hd) & 1, y = it % g.hd;
    const uint8_t *f = (img ? dis : ref) + (long long)frame * g.frame_bytes;
    const int j0 = grp * g.rg, j1 = min(s, j0 + g.rg);
    unsigned char *dst = stage0 + (size_t)(u & 1) * g.stage_bytes;
    mbar_arrive_expect_tx(&bar[u & 1], (uint32_t)((j1 - j0) * g.row_bytes));
    for (int j = j0; j < j1; ++j)
      bulk_load(dst + (size_t)(j - j0) * g.row_bytes,
                f + (long long)mirror1(y * s + lo + j, g.h) * g.row_bytes, (uint32_t)g.row_bytes,
                &bar[u & 1]);
  };

  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (t == 0) {
    issue(0);
    issue(1);
  }
  for (int u = 0;; ++u) {
    int grp;
    const int it = unit(u, grp);
    if (it < 0) break;
    const bool ok = mbar_wait(&bar[u & 1], (u >> 1) & 1);
    if (!__syncthreads_and(ok)) {
      if (t == 0) {
        atomicOr(err, kErrTmaTimeout);
        mbar_wait(&bar[u & 1], (u >> 1) & 1);             // copies still in flight
        int g2;
        if (unit(u + 1, g2) >= 0) mbar_wait(&bar[(u + 1) & 1], ((u + 1) >> 1) & 1);
      }
      return;
    }
    // vertical column sums of this group's rows (added to the partial sums)
    const unsigned char *sb = stage0 + (size_t)(u & 1) * g.stage_bytes;
    Acc *col = col2 + ((u / g.ng) & 1) * col_stride;
    const int nrows = min(s, (grp + 1) * g.rg) - grp * g.rg;
    for (int q = t; q < chunks; q += blockDim.x) {
      Acc acc[kCW];
      if constexpr (BPS == 1 && POW2) {
        // two bytes of each word summed per pass in 16-bit lanes: even
        // bytes (w & 0x00FF00FF) and odd bytes; a group holds at most 128
        // rows, so a lane stays below 128 * 255 < 2^16
        unsigned ev[4] = {0, 0, 0, 0}, od[4] = {0, 0, 0, 0};
#pragma unroll 4
        for (int jr = 0; jr < nrows; ++jr) {
          const uint4 w4 =
              *reinterpret_cast<const uint4 *>(sb + (size_t)jr * g.row_bytes + 16 * q);
          const unsigned wd4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            ev[k] += wd4[k] & 0x00FF00FFu;
            od[k] += (wd4[k] >> 8) & 0x00FF00FFu;
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[4 * k + 0] = ev[k] & 0xFFFFu;
          acc[4 * k + 1] = od[k] & 0xFFFFu;
          acc[4 * k + 2] = ev[k] >> 16;
          acc[4 * k + 3] = od[k] >> 16;
        }
        if (grp != 0) {
#pragma unroll
          for (int k = 0; k < kCW; ++k) acc[k] += col[cpad(q * kCW + k)];
        }
      } else {
#pragma unroll
        for (int k = 0; k < kCW; ++k) acc[k] = grp == 0 ? (Acc)0 : col[cpad(q * kCW + k)];
#pragma unroll 4
        for (int jr = 0; jr < nrows; ++jr) {
          const uint4 w4 =
              *reinterpret_cast<const uint4 *>(sb + (size_t)jr * g.row_bytes + 16 * q);
          const unsigned wd4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int k = 0; k < kCW; ++k) {
            const unsigned v = BPS == 1 ? (wd4[k >> 2] >> (8 * (k & 3))) & 0xFFu
                                        : (wd4[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
            if constexpr (POW2) acc[k] += v;
            else acc[k] += tap_units(v, g.c);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kCW; ++k) col[cpad(q * kCW + k)] = acc[k];
    }
    // stage u & 1 read and the column sums complete; the other column buffer
    // was last read by the item before, which every thread finished before
    // this barrier.  The stage's reads (generic proxy) are ordered before
    // the bulk copy that refills it (async proxy) by a proxy fence.
    fence_async_smem();
    __syncthreads();
    if (t == 0) issue(u + 2);
    if (grp == g.ng - 1) {
      const int frame = it / (2 * g.hd), img = (it / g.hd) & 1, y = it % g.hd;
      float *out = D + (long long)frame * 2 * g.plane + (long long)img * g.plane +
                   (long long)y * g.pitch;
      for (int x = t; x < g.wd; x += blockDim.x) {
        Acc sum = 0;
        const int x0 = x * s + lo;
        if (x0 >= 0 && x0 + s <= g.w) {
#pragma unroll 4
          for (int i = 0; i < s; ++i) sum += col[cpad(x0 + i)];
        } else {
#pragma unroll 1
          for (int i = 0; i < s; ++i) sum += col[cpad(mirror1(x0 + i, g.w))];
        }
        if constexpr (POW2)
          out[x] = __fmul_rn(__uint2float_rn(sum), g.c);
        else
          out[x] = __fmul_rn(__ull2float_rn(sum), 1.0f / 4503599627370496.0f);
      }
    }
  }
}

// Staged decimation of 8-bit luma at a power-of-two scale S in 2..16 for
// widths that are a multiple of 16 up to 4096 (at most 256 chunks of 16
// columns, one per thread).  Window x covers columns [S x - S/2, S x + S/2):
// in chunk q the windows 16q/S + 1 .. 16(q+1)/S - 1 lie inside the chunk and
// window 16q/S straddles the boundary at column 16q, made of the last S/2
// columns of chunk q-1 (its tail) and the first S/2 of chunk q (its head);
// at q = 0 the mirrored tail is the head again.  No window reaches past the
// right edge (w = 16 chunks).  So each thread sums its chunk's columns over
// the band's rows in 16-bit lanes (rows staged by bulk copies, rg per unit,
// kNst stages; partial sums stay in registers across a band's units), then
// writes its inner windows from registers and its boundary window from its
// head and the previous thread's tail in shared memory (double-buffered by
// item parity).  One barrier per unit; every wait bounded as in
// k_fssim_decimate_tma.  Sums are exact integers, rounded once.
constexpr int kNst = 4;

template <int S>
__global__ void __launch_bounds__(256)
    k_fssim_decimate_u8(FGeom g, const uint8_t *__restrict__ ref,
                        const uint8_t *__restrict__ dis, float *__restrict__ D, int nb,
                        int *__restrict__ err) {
  extern __shared__ __align__(128) unsigned char fssim_smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(fssim_smem);            // kNst barriers
  unsigned *tails = reinterpret_cast<unsigned *>(fssim_smem + 128);    // [2][256]
  unsigned char *stage0 = fssim_smem + 128 + 2 * 256 * sizeof(unsigned);
  const int t = threadIdx.x;
  const int planes = 2 * nb;                 // (frame, image) pairs: plane index 2 frame + image
  const bool owner = t < g.w / 16;

  // Items run plane-major, band y fastest; a block takes items blockIdx.x,
  // blockIdx.x + gridDim.x, ... and each item's ng row groups in order.
  // advance() moves an iterator (plane, y, group) to the next unit.
  auto advance = [&](int &pl, int &y, int &grp) {
    if (++grp == g.ng) {
      grp = 0;
      y += gridDim.x;
      while (y >= g.hd) {
        y -= g.hd;
        ++pl;
      }
    }
  };
  auto plane_base = [&](int pl) {
    return (pl & 1 ? dis : ref) + (long long)(pl >> 1) * g.frame_bytes;
  };
  // producer state (thread 0): the next unit to copy and the units issued
  int ppl = 0, py = blockIdx.x, pgrp = 0, issued = 0;
  while (py >= g.hd) {
    py -= g.hd;
    ++ppl;
  }
  auto issue_next = [&](int slot) {
    if (ppl >= planes) return;
    const uint8_t *f = plane_base(ppl);
    const int j0 = pgrp * g.rg, j1 = min(S, j0 + g.rg);
    unsigned char *dst = stage0 + (size_t)slot * g.stage_bytes;
    mbar_arrive_expect_tx(&bar[slot], (uint32_t)((j1 - j0) * g.row_bytes));
    for (int j = j0; j < j1; ++j)
      bulk_load(dst + (size_t)(j - j0) * g.row_bytes,
                f + (long long)mirror1(py * S - S / 2 + j, g.h) * g.row_bytes,
                (uint32_t)g.row_bytes, &bar[slot]);
    advance(ppl, py, pgrp);
    ++issued;
  };

  if (t == 0) {
    for (int i = 0; i < kNst; ++i) mbar_init(&bar[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (t == 0)
    for (int i = 0; i < kNst; ++i) issue_next(i);

  int pl = 0, y = blockIdx.x, grp = 0;       // consumer state (every thread)
  while (y >= g.hd) {
    y -= g.hd;
    ++pl;
  }
  int slot = 0, phase = 0, ib = 0;           // stage slot, its phase, tail buffer
  unsigned ev[4] = {0, 0, 0, 0}, od[4] = {0, 0, 0, 0};
  for (int u = 0; pl < planes; ++u) {
    const bool ok = mbar_wait(&bar[slot], phase);
    const bool last = grp == g.ng - 1;
    unsigned head = 0;
    const long long orow = (long long)pl * g.plane + (long long)y * g.pitch;  // D offset of row y
    if (owner) {
      if (grp == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) ev[k] = od[k] = 0;
      }
      const unsigned char *sb = stage0 + (size_t)slot * g.stage_bytes + 16 * t;
      const int nrows = min(S - grp * g.rg, g.rg);
#pragma unroll 4
      for (int jr = 0; jr < nrows; ++jr) {
        const uint4 w4 = *reinterpret_cast<const uint4 *>(sb + (size_t)jr * g.row_bytes);
        const unsigned wd4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ev[k] += wd4[k] & 0x00FF00FFu;          // a lane holds at most 16 * 255
          od[k] += (wd4[k] >> 8) & 0x00FF00FFu;
        }
      }
      if (last) {
        unsigned c[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          c[4 * k + 0] = ev[k] & 0xFFFFu;
          c[4 * k + 1] = od[k] & 0xFFFFu;
          c[4 * k + 2] = ev[k] >> 16;
          c[4 * k + 3] = od[k] >> 16;
        }
        float *out = D + orow + (16 / S) * t;
#pragma unroll
        for (int k = 0; k < S / 2; ++k) head += c[k];
        unsigned tail = 0;
#pragma unroll
        for (int k = 16 - S / 2; k < 16; ++k) tail += c[k];
#pragma unroll
        for (int j = 0; j + 1 < 16 / S; ++j) {
          unsigned sum = 0;
#pragma unroll
          for (int k = 0; k < S; ++k) sum += c[S / 2 + j * S + k];
          out[1 + j] = __fmul_rn(__uint2float_rn(sum), g.c);
        }
        tails[ib * 256 + t] = tail;
      }
    }
    // One barrier per unit: the stage is read, this item's tails are written
    // (the other tail buffer was last read by the item before, finished
    // before this barrier), and every thread's wait agreed.  A failed wait
    // leaves garbage sums behind and ends the kernel here.  The stage's
    // reads are ordered before the bulk copy that refills it (a proxy
    // fence, then the barrier).
    fence_async_smem();
    if (!__syncthreads_and(ok)) {
      if (t == 0) {
        atomicOr(err, kErrTmaTimeout);
        for (int i = 0; i < issued - u; ++i)       // copies still in flight
          mbar_wait(&bar[(slot + i) % kNst], phase ^ (slot + i >= kNst ? 1 : 0));
      }
      return;
    }
    if (t == 0) issue_next(slot);
    if (last && owner) {
      const unsigned prev = t == 0 ? head : tails[ib * 256 + t - 1];
      D[orow + (16 / S) * t] = __fmul_rn(__uint2float_rn(prev + head), g.c);
    }
    if (last) ib ^= 1;
    if (++slot == kNst) {
      slot = 0;
      phase ^= 1;
    }
    advance(pl, y, grp);
  }
}

// a * b per half, one rounding each (mul.rn.f32x2): the same bits as two
// scalar __fmul_rn.  Its results here only feed fma multiplicands, which
// cannot absorb it (a pair product feeding a pair add is contracted into
// one fused operation despite .rn).
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__global__ void __launch_bounds__(kMapThreads, 5)
    k_fssim_map(FGeom g, const float *__restrict__ D, double *__restrict__ part) {
  // the five quantities as three fp32 pairs (a, b), (a a, b b), (a b, 0):
  // PP holds (a, b) and (a b, 0) of the input tile ((a a, b b) is formed
  // from (a, b) in the horizontal pass), HH the horizontal sums of all three
  // for every input row (rows padded by one pair: the horizontal pass runs
  // row-fastest)
  __shared__ __align__(16) f2 PP[2][kInY][kInX + 1];
  __shared__ __align__(16) f2 HH[3][kInY][kTileX + 1];
  __shared__ float wsum[kMapThreads / 32];
  const int frame = blockIdx.z;
  const int ox0 = blockIdx.x * kTileX, oy0 = blockIdx.y * kTileY;
  const float *pa = D + (long long)frame * 2 * g.plane;
  const float *pb = pa + g.plane;
  const int t = threadIdx.x;
  // per-tile offset: the reference sample at the tile origin (same for both)
  const float off = pa[(long long)oy0 * g.pitch + ox0];
  // every load of a thread is issued before the first is used; thread
  // t < 126 takes column t % 42 and rows t / 42, + 3, + 6, ...
  constexpr int kRowStep = kMapThreads / kInX;             // 3
  constexpr int kPer = (kInY + kRowStep - 1) / kRowStep;   // 9
  const int c = t % kInX, r0 = t / kInX;
  const bool loader = t < kRowStep * kInX;
  const int xc = min(ox0 + c, g.wd - 1);
  float va[kPer], vb[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int r = r0 + kRowStep * k;
    if (loader && r < kInY) {
      const long long at = (long long)min(oy0 + r, g.hd - 1) * g.pitch + xc;
      va[k] = pa[at];
      vb[k] = pb[at];
    }
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int r = r0 + kRowStep * k;
    if (loader && r < kInY) {
      const float p = __fsub_rn(va[k], off);
      const float q = __fsub_rn(vb[k], off);
      PP[0][r][c] = f2_pack(p, q);
      PP[1][r][c] = f2_pack(__fmul_rn(p, q), 0.0f);
    }
  }
  f2 gk[kWin];
#pragma unroll
  for (int k = 0; k < kWin; ++k) gk[k] = f2_pack(g.gauss[k], g.gauss[k]);
  __syncthreads();
  // horizontal sums: a task is 4 adjacent outputs of one input row, rows
  // fastest across threads (conflict-free 64-bit shared accesses)
  for (int task = t; task < kInY * (kTileX / 4); task += kMapThreads) {
    const int r = task % kInY, c0 = 4 * (task / kInY);
    f2 v[kWin + 3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      // q = 0: (a, b) as loaded; q = 1: its squares; q = 2: (a b, 0)
#pragma unroll
      for (int k = 0; k < kWin + 3; ++k)
        v[k] = q == 0 ? PP[0][r][c0 + k] : (q == 1 ? f2_mul(v[k], v[k]) : PP[1][r][c0 + k]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f2 acc = 0ull;
#pragma unroll
        for (int k = 0; k < kWin; ++k) acc = f2_fma(gk[k], v[j + k], acc);
        HH[q][r][c0 + j] = acc;
      }
    }
  }
  __syncthreads();
  // vertical sums and the SSIM terms of four outputs (rows 4 w .. 4 w + 3,
  // w = thread / 32): 14 loads of a column serve four outputs
  const int oc = t % kTileX, orow = 4 * (t / kTileX);
  const int ox = ox0 + oc;
  f2 m[4][3];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    f2 v[kWin + 3];
#pragma unroll
    for (int k = 0; k < kWin + 3; ++k) v[k] = HH[q][orow + k][oc];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f2 acc = 0ull;
#pragma unroll
      for (int k = 0; k < kWin; ++k) acc = f2_fma(gk[k], v[j + k], acc);
      m[j][q] = acc;
    }
  }
  float tile = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int oy = oy0 + orow + j;
    if (ox < g.ow && oy < g.oh) {
      float m1, m2, e11, e22, e12, unused;
      f2_unpack(m[j][0], m1, m2);
      f2_unpack(m[j][1], e11, e22);
      f2_unpack(m[j][2], e12, unused);
      const float v1 = __fsub_rn(e11, __fmul_rn(m1, m1));
      const float v2 = __fsub_rn(e22, __fmul_rn(m2, m2));
      const float cv = __fsub_rn(e12, __fmul_rn(m1, m2));
      const float mu1 = __fadd_rn(m1, off), mu2 = __fadd_rn(m2, off);
      const float num = __fmul_rn(__fadd_rn(__fmul_rn(2.0f, __fmul_rn(mu1, mu2)), g.C1),
                                  __fadd_rn(__fmul_rn(2.0f, cv), g.C2));
      const float den = __fmul_rn(
          __fadd_rn(__fadd_rn(__fmul_rn(mu1, mu1), __fmul_rn(mu2, mu2)), g.C1),
          __fadd_rn(__fadd_rn(v1, v2), g.C2));
      tile = __fadd_rn(tile, __fdiv_rn(num, den));
    }
  }
  // warp sums in fp32 (a fixed xor tree; lane 0's order is fixed), then the
  // block's four warp sums in fp64 in warp order (fp64 is slow on this part)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tile = __fadd_rn(tile, __shfl_xor_sync(0xffffffffu, tile, o));
  if ((t & 31) == 0) wsum[t >> 5] = tile;
  __syncthreads();
  if (t == 0) {
    double acc = 0.0;
#pragma unroll
    for (int w = 0; w < kMapThreads / 32; ++w) acc = __dadd_rn(acc, (double)wsum[w]);
    part[(long long)frame * g.tiles_x * g.tiles_y + blockIdx.y * g.tiles_x + blockIdx.x] = acc;
  }
}

// One warp per frame: lane l adds the block sums l, l + 32, ... in order,
// then a fixed xor-shuffle tree; the same order every run.
__global__ void k_fssim_final(FGeom g, const double *__restrict__ part, double *__restrict__ out) {
  const int frame = blockIdx.x, lane = threadIdx.x;
  const int n = g.tiles_x * g.tiles_y;
  const double *p = part + (long long)frame * n;
  double s = 0.0;
  for (int i = lane; i < n; i += 32) s = __dadd_rn(s, p[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  if (lane == 0) out[frame] = s / ((double)g.ow * (double)g.oh);
}

}  // namespace

using namespace ss2;

struct ss2_fssim {
  FGeom g;
  int batch, device;
  float *d_dec = nullptr;      // 2 planes per frame
  double *d_part = nullptr, *d_scores = nullptr, *h_scores = nullptr;
  size_t h_cap = 0;
  int *d_err = nullptr, *h_err = nullptr;   // error bits raised by kernels (bounded waits)
  KernelTimer timer;                         // per-kernel event timing
};

static void fssim_free(ss2_fssim *c) {
  if (!c) return;
  cudaFree(c->d_dec);
  cudaFree(c->d_part);
  cudaFree(c->d_scores);
  cudaFree(c->d_err);
  if (c->h_scores) cudaFreeHost(c->h_scores);
  if (c->h_err) cudaFreeHost(c->h_err);
  delete c;
}

// Plans the staged decimation: frames whose rows are whole 16-byte chunks
// (and whose packed size keeps every frame 16-byte aligned) stage rg rows of
// a band at a time, two stages of at most kStageBudget bytes, with two
// padded column-sum buffers beside them; the grid is the resident block count.  Other geometries
// use k_fssim_decimate.
constexpr long long kStageBudget = 16 * 1024;
constexpr unsigned kSmemLimit = 227 * 1024;

template <int BPS, bool POW2>
static int fssim_plan_one(FGeom &g, int dev) {
  int sms = 0, per_sm = 0;
  cudaError_t e = cudaFuncSetAttribute(k_fssim_decimate_tma<BPS, POW2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)g.smem_staged);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fssim_decimate_tma<BPS, POW2>,
                                                      256, g.smem_staged);
  if (e != cudaSuccess) return cuda_fail(e, "float_ssim staged decimation setup");
  g.grid_staged = std::max(1, per_sm) * sms;
  return 0;
}

template <int S>
static int fssim_plan_u8(FGeom &g, int dev) {
  int sms = 0, per_sm = 0;
  cudaError_t e = cudaFuncSetAttribute(k_fssim_decimate_u8<S>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)g.smem_staged);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fssim_decimate_u8<S>, 256,
                                                      g.smem_staged);
  if (e != cudaSuccess) return cuda_fail(e, "float_ssim staged decimation setup");
  g.grid_staged = std::max(1, per_sm) * sms;
  return 0;
}

static int fssim_plan_staged(FGeom &g, int dev) {
  g.row_bytes = (long long)g.w * g.bps;
  g.staged = 0;
  if (g.row_bytes % 16 || g.frame_bytes % 16) return 0;
  if (g.bps == 1 && g.pow2 && g.scale >= 2 && g.scale <= 16 && g.w <= 16 * 256) {
    g.rg = (int)std::min<long long>(g.scale, std::max<long long>(1, kStageBudget / g.row_bytes));
    g.ng = (g.scale + g.rg - 1) / g.rg;
    g.stage_bytes = (unsigned)(g.rg * g.row_bytes);
    g.smem_staged = 128 + 2 * 256 * sizeof(unsigned) + kNst * g.stage_bytes;
    g.staged = 2;
    switch (g.scale) {
      case 2: return fssim_plan_u8<2>(g, dev);
      case 4: return fssim_plan_u8<4>(g, dev);
      case 8: return fssim_plan_u8<8>(g, dev);
      default: return fssim_plan_u8<16>(g, dev);
    }
  }
  const size_t acc = g.pow2 ? sizeof(unsigned) : sizeof(unsigned long long);
  g.col_bytes = (unsigned)(((size_t)(g.w + g.w / 16 + 1) * acc + 127) & ~(size_t)127);
  g.rg = (int)std::min<long long>(g.scale, std::max<long long>(1, kStageBudget / g.row_bytes));
  g.ng = (g.scale + g.rg - 1) / g.rg;
  g.stage_bytes = (unsigned)(g.rg * g.row_bytes);
  const size_t smem = 128 + 2 * (size_t)g.col_bytes + 2 * (size_t)g.stage_bytes;
  if (smem > kSmemLimit) return 0;
  g.smem_staged = (unsigned)smem;
  g.staged = 1;
  if (g.bps == 1)
    return g.pow2 ? fssim_plan_one<1, true>(g, dev) : fssim_plan_one<1, false>(g, dev);
  return g.pow2 ? fssim_plan_one<2, true>(g, dev) : fssim_plan_one<2, false>(g, dev);
}

SS2_API ss2_fssim *ss2_fssim_create(int width, int height, int bitdepth, int chroma,
                                    int max_batch) {
  if (check_geometry(width, height, bitdepth, chroma)) return nullptr;
  if (max_batch < 0 || max_batch > 4096) {
    fail(SS2_EINVAL, "batch %d is outside 0..4096", max_batch);
    return nullptr;
  }
  FGeom g;
  std::memset(&g, 0, sizeof(g));
  g.w = width; g.h = height; g.depth = bitdepth; g.bps = bitdepth > 8 ? 2 : 1;
  Geom full;
  make_geom(width, height, bitdepth, chroma, full);
  g.frame_bytes = full.frame_bytes;
  const int m = std::min(width, height);
  g.scale = std::max(1, (int)std::lround((double)m / 256.0));
  g.wd = (width + g.scale - 1) / g.scale;
  g.hd = (height + g.scale - 1) / g.scale;
  if (g.scale > 128 || g.wd < kWin || g.hd < kWin) {
    fail(SS2_ENOTSUP, "float_ssim: decimated plane %dx%d (factor %d) is below 11x11 or the "
                      "factor exceeds 128", g.wd, g.hd, g.scale);
    return nullptr;
  }
  g.pitch = (g.wd + 31) & ~31;
  g.plane = (long long)g.pitch * g.hd;
  g.ow = g.wd - kWin + 1;
  g.oh = g.hd - kWin + 1;
  g.tiles_x = (g.ow + kTileX - 1) / kTileX;
  g.tiles_y = (g.oh + kTileY - 1) / kTileY;
  g.wt = 1.0f / (float)(g.scale * g.scale);
  g.norm = 1.0f / (float)(1 << (bitdepth - 8));
  g.c = g.wt * g.norm;
  g.pow2 = (g.scale & (g.scale - 1)) == 0;
  const double L = 255.0;
  g.C1 = (float)((0.01 * L) * (0.01 * L));
  g.C2 = (float)((0.03 * L) * (0.03 * L));
  double gs[kWin], tot = 0.0;
  for (int i = 0; i < kWin; ++i) {
    const double t = i - kWin / 2;
    gs[i] = std::exp(-t * t / (2.0 * 1.5 * 1.5));
    tot += gs[i];
  }
  for (int i = 0; i < kWin; ++i) g.gauss[i] = (float)(gs[i] / tot);
  int dev = 0;
  if (check_device(&dev)) return nullptr;
  if (fssim_plan_staged(g, dev)) return nullptr;
  ss2_fssim *c = new (std::nothrow) ss2_fssim();
  if (!c) {
    fail(SS2_ENOMEM, "host allocation failed");
    return nullptr;
  }
  c->g = g;
  c->device = dev;
  c->batch = max_batch ? max_batch : 64;
  const size_t B = (size_t)c->batch;
  if (cudaMalloc(&c->d_dec, B * 2 * g.plane * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&c->d_part, B * g.tiles_x * g.tiles_y * sizeof(double)) != cudaSuccess ||
      cudaMalloc(&c->d_scores, B * sizeof(double)) != cudaSuccess ||
      cudaMalloc(&c->d_err, sizeof(int)) != cudaSuccess ||
      cudaMallocHost(&c->h_err, sizeof(int)) != cudaSuccess ||
      cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess ||
      // the memset is ordered on the legacy stream only: wait for it
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    fail(SS2_ENOMEM, "float_ssim workspace allocation failed");
    fssim_free(c);
    return nullptr;
  }
  *c->h_err = 0;
  return c;
}

SS2_API void ss2_fssim_destroy(ss2_fssim *ctx) { fssim_free(ctx); }

SS2_API int ss2_fssim_scale(const ss2_fssim *ctx) { return ctx ? ctx->g.scale : 0; }

SS2_API int ss2_fssim_profile_begin(ss2_fssim *ctx) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  ctx->timer.begin();
  return 0;
}

SS2_API int ss2_fssim_profile_end(ss2_fssim *ctx, double *ms, int *launches) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  const cudaError_t e = ctx->timer.finish(3, ms, launches);
  return e == cudaSuccess ? 0 : cuda_fail(e, "float_ssim profile events");
}

static size_t fssim_decimate_smem(const FGeom &g) {
  return (size_t)g.w * (g.pow2 ? sizeof(unsigned) : sizeof(unsigned long long));
}

template <int BPS, bool POW2>
static cudaError_t fssim_decimate_one(const FGeom &g, const uint8_t *ref, const uint8_t *dis,
                                      float *D, int nb, cudaStream_t st) {
  const size_t smem = fssim_decimate_smem(g);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_fssim_decimate<BPS, POW2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_fssim_decimate<BPS, POW2><<<dim3(g.hd, 2, nb), 256, smem, st>>>(g, ref, dis, D);
  return cudaGetLastError();
}

template <int BPS, bool POW2>
static cudaError_t fssim_staged_one(const FGeom &g, const uint8_t *ref, const uint8_t *dis,
                                    float *D, int nb, int *err, cudaStream_t st) {
  const int items = nb * 2 * g.hd;
  k_fssim_decimate_tma<BPS, POW2><<<std::min(items, g.grid_staged), 256, g.smem_staged, st>>>(
      g, ref, dis, D, nb, err);
  return cudaGetLastError();
}

template <int S>
static cudaError_t fssim_u8_one(const FGeom &g, const uint8_t *ref, const uint8_t *dis, float *D,
                                int nb, int *err, cudaStream_t st) {
  const int items = nb * 2 * g.hd;
  k_fssim_decimate_u8<S><<<std::min(items, g.grid_staged), 256, g.smem_staged, st>>>(
      g, ref, dis, D, nb, err);
  return cudaGetLastError();
}

static cudaError_t fssim_launch_decimate(const FGeom &g, const uint8_t *ref, const uint8_t *dis,
                                         float *D, int nb, int *err, cudaStream_t st) {
  const bool aligned =
      ((reinterpret_cast<uintptr_t>(ref) | reinterpret_cast<uintptr_t>(dis)) & 15) == 0;
  if (g.staged == 2 && aligned) {
    switch (g.scale) {
      case 2: return fssim_u8_one<2>(g, ref, dis, D, nb, err, st);
      case 4: return fssim_u8_one<4>(g, ref, dis, D, nb, err, st);
      case 8: return fssim_u8_one<8>(g, ref, dis, D, nb, err, st);
      default: return fssim_u8_one<16>(g, ref, dis, D, nb, err, st);
    }
  }
  if (g.staged == 1 && aligned) {
    if (g.bps == 1)
      return g.pow2 ? fssim_staged_one<1, true>(g, ref, dis, D, nb, err, st)
                    : fssim_staged_one<1, false>(g, ref, dis, D, nb, err, st);
    return g.pow2 ? fssim_staged_one<2, true>(g, ref, dis, D, nb, err, st)
                  : fssim_staged_one<2, false>(g, ref, dis, D, nb, err, st);
  }
  if (g.bps == 1)
    return g.pow2 ? fssim_decimate_one<1, true>(g, ref, dis, D, nb, st)
                  : fssim_decimate_one<1, false>(g, ref, dis, D, nb, st);
  return g.pow2 ? fssim_decimate_one<2, true>(g, ref, dis, D, nb, st)
                : fssim_decimate_one<2, false>(g, ref, dis, D, nb, st);
}

// Reports (and clears) error bits the kernels raised; h_err must hold a
// copy of d_err taken after the launches.
static int fssim_check_err(ss2_fssim *c, cudaStream_t st) {
  if (*c->h_err == 0) return 0;
  const int bits = *c->h_err;
  *c->h_err = 0;
  cudaMemsetAsync(c->d_err, 0, sizeof(int), st);
  cudaStreamSynchronize(st);
  return fail(SS2_EIO, "float_ssim: a bounded wait for a bulk copy gave up (error bits %#x)", bits);
}

SS2_API int ss2_fssim_score(ss2_fssim *ctx, const void *ref, const void *dis, int n_frames,
                            double *scores, void *stream) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  if (n_frames < 0) return fail(SS2_EINVAL, "negative frame count %d", n_frames);
  if (n_frames == 0) return 0;
  if (!ref || !dis || !scores) return fail(SS2_EINVAL, "NULL pointer");
  if ((size_t)n_frames > ctx->h_cap) {
    if (ctx->h_scores) cudaFreeHost(ctx->h_scores);
    ctx->h_scores = nullptr;
    ctx->h_cap = 0;
    if (cudaMallocHost(&ctx->h_scores, (size_t)n_frames * sizeof(double)) != cudaSuccess) {
      cudaGetLastError();
      return fail(SS2_ENOMEM, "pinned allocation failed");
    }
    ctx->h_cap = (size_t)n_frames;
  }
  const FGeom &g = ctx->g;
  cudaStream_t st = (cudaStream_t)stream;
  const uint8_t *r8 = (const uint8_t *)ref, *d8 = (const uint8_t *)dis;
  for (int f0 = 0; f0 < n_frames; f0 += ctx->batch) {
    const int nb = std::min(ctx->batch, n_frames - f0);
    cudaError_t e = ctx->timer.mark(0, true, st);
    if (e == cudaSuccess)
      e = fssim_launch_decimate(g, r8 + f0 * g.frame_bytes, d8 + f0 * g.frame_bytes, ctx->d_dec,
                                nb, ctx->d_err, st);
    if (e == cudaSuccess) e = ctx->timer.mark(0, false, st);
    if (e == cudaSuccess) e = ctx->timer.mark(1, true, st);
    if (e == cudaSuccess) {
      k_fssim_map<<<dim3(g.tiles_x, g.tiles_y, nb), kMapThreads, 0, st>>>(g, ctx->d_dec, ctx->d_part);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = ctx->timer.mark(1, false, st);
    if (e == cudaSuccess) e = ctx->timer.mark(2, true, st);
    if (e == cudaSuccess) {
      k_fssim_final<<<nb, 32, 0, st>>>(g, ctx->d_part, ctx->d_scores);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = ctx->timer.mark(2, false, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ctx->h_scores + f0, ctx->d_scores, nb * sizeof(double),
                          cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "float_ssim launch");
  }
  cudaError_t e = cudaMemcpyAsync(ctx->h_err, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (int rc = fssim_check_err(ctx, st)) return rc;
  std::memcpy(scores, ctx->h_scores, (size_t)n_frames * sizeof(double));
  return 0;
}

SS2_API int ss2_fssim_debug_decimated(ss2_fssim *ctx, const void *ref, const void *dis,
                                      float *planes, void *stream) {
  if (!ctx || !ref || !dis || !planes) return fail(SS2_EINVAL, "NULL argument");
  const FGeom &g = ctx->g;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = fssim_launch_decimate(g, (const uint8_t *)ref, (const uint8_t *)dis,
                                        ctx->d_dec, 1, ctx->d_err, st);
  for (int p = 0; p < 2 && e == cudaSuccess; ++p)
    e = cudaMemcpy2DAsync(planes + (size_t)p * g.wd * g.hd, g.wd * sizeof(float),
                          ctx->d_dec + p * g.plane, g.pitch * sizeof(float), g.wd * sizeof(float),
                          g.hd, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ctx->h_err, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "float_ssim decimation");
  return fssim_check_err(ctx, st);
}
