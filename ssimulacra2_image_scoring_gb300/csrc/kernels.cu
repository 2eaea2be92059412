// kernels.cu — the ssimulacra2 hot path on sm_103a.
//
//   k_pyramid   YUV -> linear RGB -> XYB at scale 0, then the 2x2 downsample
//               of linear RGB and XYB at scales 1..5, one 32x32 scale-0 tile
//               per block (the tile's pyramid stays in shared memory, so the
//               YUV planes are read once and only XYB reaches HBM).
//   k_hblur     horizontal recursive Gaussian of the five quantities
//               (x1, x2, x1^2, x2^2, x1 x2) of one row and channel; the
//               products are formed in registers (multiply_3plane fused).
//   k_vblur     vertical recursive Gaussian of the same five quantities down
//               one column, fused with ssim_map and edge_diff_map and the six
//               double-float sums; one partial per warp and (channel, sum).
//   k_finalize  partials -> 108 values -> pool_score, one block per frame.
//
// Source: "Research-1363: Device-resident ssimulacra2 and a single-wait
// MS-SSIM on SYCL" (vmafx documentation), "Sources" (the steps) and
// Findings 2, 4, 7 (numerics, float pairs and the fixed reduction tree, the
// sequential IIR along each line).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <utility>

#include "ss2_device.cuh"
#include "ss2_f32x2.cuh"
#include "ss2_tma.cuh"
#include "ss2_impl.h"
#include "ss2_kernels.h"

namespace ss2 {

// ---------------------------------------------------------------------------
// k_pyramid: one 64x64 scale-0 tile of one frame pair per block.
//
// Scale 0 and 1.  Warp w takes the tile's row pairs w, w + 8, w + 16, w + 24;
// lane l takes the 2x2 quad at tile columns 2l, 2l + 1 of the row pair.  The
// row pair's samples (two luma rows and their chroma rows, both frames) are
// staged in a per-warp shared-memory buffer: 16-byte asynchronous copies
// when the geometry keeps every row start on 16 bytes, else sample by
// sample.  The next row pair's copies are in flight while the current one is
// computed (two buffers per warp).  Each thread converts its quad's four
// pixels (YUV -> R'G'B' -> linear RGB -> XYB, stored two columns at a time),
// averages the quad's linear RGB into the scale-1 pixel, forms that pixel's
// XYB at once and keeps its linear RGB in shared memory: no barrier sits
// between scale 0 and scale 1.
//
// Scales 2-5 are halved from the shared scale-1 tile (16x16, 8x8, 4x4, 2x2
// pixels): one block barrier before scale 2, then scale 3 on two warps (a
// named barrier) and scales 4-5 on one warp; the other warps leave.
//
// Only XYB reaches HBM; linear RGB never does (lin_dbg, when set, receives
// the linear RGB of scale dbg_scale for the parity tests).
// ---------------------------------------------------------------------------

constexpr int kPT = 64;  // scale-0 tile edge; 64 = 2^6 keeps 5 halvings inside the tile
constexpr int kPyrThreads = 256;
constexpr int kPyrWarps = kPyrThreads / 32;
constexpr int kPyrIters = kPT / 2 / kPyrWarps;  // row pairs per warp
// Shared tiles of linear RGB: scale 1 (32 x 32 per plane) in a region of
// its own, scales 2-5 (16^2 + 8^2 + 4^2 + 2^2 = 340 floats per plane) in a
// region that the row staging of scales 0-1 uses first.  Offset of the
// scale-s tile (s >= 2) in a plane's part of that region:
// sum_{k=2}^{s-1} (64 >> k)^2 = (1024 - (4096 >> 2(s-1))) / 3
constexpr int kLvl1 = 1024;
__host__ __device__ constexpr int lvl_off(int s) { return (1024 - (4096 >> (2 * (s - 1)))) / 3; }
constexpr int kLvlRest = lvl_off(kMaxScales);  // 340 floats per plane

// Staging geometry, fixed per instantiation (sample width and chroma
// layout), and the per-launch choices.
template <int BPS, int SX, int SY>
struct StageGeo {
  static constexpr int ybytes = kPT * BPS;            // one staged luma row
  static constexpr int cbytes = (kPT >> SX) * BPS;    // one staged chroma row
  static constexpr int crows = SY ? 1 : 2;            // chroma rows per luma row pair
  static constexpr int img_bytes = 2 * ybytes + 2 * crows * cbytes;  // a multiple of 16
  static constexpr int buf_bytes = 2 * img_bytes;     // both frames
  static_assert(buf_bytes % 128 == 0, "a whole number of 4-byte words per lane");
  // the staging (two buffers per warp) shares its region with scales 2-5
  static constexpr int stage_bytes = kPyrWarps * 2 * buf_bytes;
  static constexpr int union_bytes =
      stage_bytes > 6 * kLvlRest * 4 ? stage_bytes : 6 * kLvlRest * 4;
};
struct PyrStage {
  int vec;        // 1: 16-byte copies (every staged row starts on 16 bytes)
  int dbg_scale;  // scale whose linear RGB is written to lin_dbg, or -1
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Source of byte `off` of one frame's staged rows for the row pair starting
// at luma row r0 (layout: luma row r0, luma row r0 + 1, the U rows, the V
// rows), and whether that byte lies inside the frame.
template <int BPS, int SX, int SY>
__device__ __forceinline__ const uint8_t *stage_src(const Geom &g, const uint8_t *f, int tx0,
                                                    int r0, int off, bool &ok) {
  using SG = StageGeo<BPS, SX, SY>;
  if (off < 2 * SG::ybytes) {
    const int r = off >= SG::ybytes;
    const int col = off - (r ? SG::ybytes : 0);
    const int y = r0 + r;
    ok = y < g.h && tx0 * BPS + col < g.w * BPS;
    return f + (y * g.w + tx0) * BPS + col;
  }
  off -= 2 * SG::ybytes;
  const int plane = off >= SG::crows * SG::cbytes;
  off -= plane ? SG::crows * SG::cbytes : 0;
  const int r = SG::crows == 2 && off >= SG::cbytes;
  const int col = off - (r ? SG::cbytes : 0);
  const int cy = (r0 >> SY) + r, cx0 = tx0 >> SX;
  ok = cy < g.ch && cx0 * BPS + col < g.cw * BPS;
  return f + (g.w * g.h + plane * g.cw * g.ch + cy * g.cw + cx0) * BPS + col;
}

template <int BPS>
__device__ __forceinline__ int stage_sample(const unsigned char *p) {
  if (BPS == 1) return *p;
  return *reinterpret_cast<const uint16_t *>(p);
}

// Index arithmetic is 32-bit inside a frame: a plane holds at most
// 16384 x 16384 samples and the byte offset of a V sample stays below
// 2 x 1.5 x 2^28; each scale's XYB block is reached from a 64-bit base and
// its six planes lie within 6 x 2^28 floats of it.
//
// Four blocks per SM (up to 64 registers): at five (48 registers) the loop
// spilled a register pair to local memory (0.78 M spill stores and 1.04 M
// spill loads, in warp instructions, per launch over four 4K frames), which
// cost more than the fifth block gained.
template <int BPS, int SX, int SY, bool DBG>
__global__ void __launch_bounds__(kPyrThreads, 4)
    k_pyramid(Geom g, Pix px, PyrTabs tabs, PyrStage ps, const uint8_t *__restrict__ ref,
              const uint8_t *__restrict__ dis, float *__restrict__ X,
              float *__restrict__ lin_dbg) {
  using SG = StageGeo<BPS, SX, SY>;
  extern __shared__ __align__(16) unsigned char psm[];
  float(*L1)[kLvl1] = reinterpret_cast<float(*)[kLvl1]>(psm);
  unsigned char *stage = psm + sizeof(float) * 6 * kLvl1;           // scales 0-1 ...
  float(*Lr)[kLvlRest] = reinterpret_cast<float(*)[kLvlRest]>(stage);  // ... then 2-5
  float *ntab = reinterpret_cast<float *>(stage + SG::union_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int frame = blockIdx.z;
  const int tx0 = blockIdx.x * kPT, ty0 = blockIdx.y * kPT;
  float *Xf = X + (long long)frame * g.x_fs;
  const uint8_t *fref = ref + (long long)frame * g.frame_bytes;
  const uint8_t *fdis = dis + (long long)frame * g.frame_bytes;
  constexpr int buf_bytes = SG::buf_bytes;
  unsigned char *wst = stage + warp * 2 * buf_bytes;  // this warp's two buffers

  // row pair i of this warp -> buffer i & 1 (vec: one copy group per row pair)
  auto stage_rows = [&](int i) {
    const int r0 = ty0 + 2 * (warp + kPyrWarps * i);
    unsigned char *dst = wst + (i & 1) * buf_bytes;
    if (ps.vec) {
      if (r0 < g.h) {
        for (int c = lane; c < (buf_bytes >> 4); c += 32) {
          int off = c << 4;
          const int img = off >= SG::img_bytes;
          off -= img ? SG::img_bytes : 0;
          bool ok;
          const uint8_t *src = stage_src<BPS, SX, SY>(g, img ? fdis : fref, tx0, r0, off, ok);
          if (ok) cp_async16(dst + (c << 4), src);
        }
      }
      cp_async_commit();  // possibly empty: keeps one group per row pair
    } else if (r0 < g.h) {
      // rows that do not all start on 16 bytes: 4-byte words, each the
      // funnel shift of the two aligned words that cover it.  A word whose
      // first byte lies outside its row is skipped (nothing reads it); one
      // whose first byte is inside may run past the row's end into bytes
      // that nothing reads, so the aligned loads are only taken when both
      // lie inside the frame, and a word at the frame's first or last bytes
      // is read sample by sample up to the frame's end.  The segments (luma
      // and chroma rows) are multiples of 4 bytes, so no word spans two.
#pragma unroll
      for (int it = 0; it < buf_bytes / 128; ++it) {
        const int e = lane + 32 * it;
        int off = e * 4;
        const int img = off >= SG::img_bytes;
        off -= img ? SG::img_bytes : 0;
        const uint8_t *f = img ? fdis : fref;
        bool ok;
        const uint8_t *src = stage_src<BPS, SX, SY>(g, f, tx0, r0, off, ok);
        if (!ok) continue;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
        const uintptr_t a = sa & ~uintptr_t(3);
        const uint32_t sh = (uint32_t)(sa & 3u) * 8u;
        const uintptr_t lo = reinterpret_cast<uintptr_t>(f);
        const uintptr_t hi = lo + (uintptr_t)g.frame_bytes;
        uint32_t w = 0;
        if (a >= lo && a + (sh ? 8u : 4u) <= hi) {
          const uint32_t *wp = reinterpret_cast<const uint32_t *>(a);
          const uint32_t w0 = __ldg(wp);
          const uint32_t w1 = sh ? __ldg(wp + 1) : 0u;
          w = __funnelshift_r(w0, w1, sh);
        } else {
          for (int b = 0; b < 4; b += BPS)
            if (sa + (uintptr_t)b < hi) {
              const uint32_t v = BPS == 1 ? (uint32_t)__ldg(src + b)
                                          : (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(src + b));
              w |= v << (8 * b);
            }
        }
        reinterpret_cast<uint32_t *>(dst)[e] = w;
      }
    }
  };
  stage_rows(0);

  // the 8-bit normalisation tables, once per block
  if (BPS == 1 && tabs.ynorm) {
    for (int i = threadIdx.x; i < 256; i += kPyrThreads) {
      ntab[i] = __ldg(tabs.ynorm + i);
      ntab[256 + i] = __ldg(tabs.cnorm + i);
    }
  }
  __syncthreads();
  float cb[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) cb[i] = px.cbias[i];

  const int k = 1 << (g.depth - 8);
  const float dy = (float)(219 * k), dc = (float)(224 * k);
  const bool two_scales = g.nscales > 1;
  float *P0 = Xf + g.xoff[0];
  float *P1 = Xf + g.xoff[1];
  const int plane0 = (int)g.plane[0], pitch0 = g.pitch[0];
  const int plane1 = (int)g.plane[1], pitch1 = g.pitch[1];
  const int lx0 = 2 * lane;                             // the quad's tile columns
  const int lx1 = min(lx0 + 1, g.w - 1 - tx0);          // clamped at an odd right edge
  const bool has_x1 = tx0 + lx0 + 1 < g.w;
  const bool dbg0 = DBG && ps.dbg_scale == 0, dbg1 = DBG && ps.dbg_scale == 1;

  // ---- scales 0 and 1 ----
  for (int i = 0; i < kPyrIters; ++i) {
    if (i + 1 < kPyrIters) stage_rows(i + 1);
    if (ps.vec) {
      if (i + 1 < kPyrIters)
        cp_async_wait<1>();
      else
        cp_async_wait<0>();
    }
    __syncwarp();
    const int rp = warp + kPyrWarps * i;
    const int y0 = ty0 + 2 * rp;
    if (y0 < g.h && tx0 + lx0 < g.w) {
      const bool has_y1 = y0 + 1 < g.h;
      const unsigned char *sb = wst + (i & 1) * buf_bytes;
      const int x1 = (tx0 >> 1) + lane, y1 = (ty0 >> 1) + rp;  // the scale-1 pixel
      // one image at a time (not unrolled: the body holds three cube roots
      // per pixel, and one copy of it keeps the code in the instruction cache)
#pragma unroll 1
      for (int img = 0; img < 2; ++img) {
        const unsigned char *sY = sb + img * SG::img_bytes;
        const unsigned char *sU = sY + 2 * SG::ybytes;
        const unsigned char *sV = sU + SG::crows * SG::cbytes;
        // normalised chroma of (staged row crr, chroma column cl)
        auto chroma = [&](int crr, int cl, float &cbv, float &crv) {
          const int cofs = crr * SG::cbytes + cl * BPS;
          const int Us = stage_sample<BPS>(sU + cofs);
          const int Vs = stage_sample<BPS>(sV + cofs);
          if (BPS == 1 && tabs.ynorm) {
            cbv = ntab[256 + Us];
            crv = ntab[256 + Vs];
          } else {
            cbv = norm_div(Us - 128 * k, dc, tabs.rdc);
            crv = norm_div(Vs - 128 * k, dc, tabs.rdc);
          }
        };
        // horizontally subsampled chroma: both pixels of a quad row share
        // one chroma sample (column lane, also when the right one is
        // clamped); vertically subsampled: both rows share one chroma row
        float cbq[2][2], crq[2][2];   // [dyy][dxx]
        if (SY) {
          chroma(0, lx0 >> SX, cbq[0][0], crq[0][0]);
          if (SX) {
            cbq[0][1] = cbq[0][0];
            crq[0][1] = crq[0][0];
          } else {
            chroma(0, lx1, cbq[0][1], crq[0][1]);
          }
        }
        float acc[3];
#pragma unroll 1
        for (int dyy = 0; dyy < 2; ++dyy) {
          const int rr = dyy && has_y1 ? 1 : 0;  // clamped at an odd bottom edge
          float cbr[2], crr_[2];
          if (SY) {
#pragma unroll
            for (int d = 0; d < 2; ++d) {
              cbr[d] = cbq[0][d];
              crr_[d] = crq[0][d];
            }
          } else {
            chroma(rr, lx0 >> SX, cbr[0], crr_[0]);
            if (SX) {
              cbr[1] = cbr[0];
              crr_[1] = crr_[0];
            } else {
              chroma(rr, lx1, cbr[1], crr_[1]);
            }
          }
          float o[2][3];
#pragma unroll
          for (int dxx = 0; dxx < 2; ++dxx) {
            const int lx = dxx ? lx1 : lx0;
            const int Ys = stage_sample<BPS>(sY + rr * SG::ybytes + lx * BPS);
            const float yn = BPS == 1 && tabs.ynorm ? ntab[Ys] : norm_div(Ys - 16 * k, dy, tabs.rdy);
            const float cbv = cbr[dxx], crv = crr_[dxx];
            // R'G'B' clamped to [0, 1] as part of the matrix's last fma
            const float R = eotf_lookup(tabs.eotf, fma_sat(px.yuv[0], crv, yn));
            const float G = eotf_lookup(
                tabs.eotf, fma_sat(-px.yuv[2], crv, __fmaf_rn(-px.yuv[1], cbv, yn)));
            const float B = eotf_lookup(tabs.eotf, fma_sat(px.yuv[3], cbv, yn));
            // the 2x2 mean in the order ((p00 + p01) + p10) + p11
            if (dyy == 0 && dxx == 0) {
              acc[0] = R;
              acc[1] = G;
              acc[2] = B;
            } else {
              acc[0] = __fadd_rn(acc[0], R);
              acc[1] = __fadd_rn(acc[1], G);
              acc[2] = __fadd_rn(acc[2], B);
            }
            if (dbg0 && (dyy == 0 || has_y1) && (dxx == 0 || has_x1)) {
              const long long q = (long long)(y0 + dyy) * g.w + tx0 + lx;
              const long long n0 = (long long)g.w * g.h;
              lin_dbg[(3 * img + 0) * n0 + q] = R;
              lin_dbg[(3 * img + 1) * n0 + q] = G;
              lin_dbg[(3 * img + 2) * n0 + q] = B;
            }
            pixel_xyb(px, cb, R, G, B, o[dxx][0], o[dxx][1], o[dxx][2]);
          }
          if (dyy == 0 || has_y1) {
            float *P = P0 + ((y0 + dyy) * pitch0 + tx0 + lx0);
#pragma unroll
            for (int c = 0; c < 3; ++c) {
              float *q = P + (3 * img + c) * plane0;
              if (has_x1)
                *reinterpret_cast<float2 *>(q) = make_float2(o[0][c], o[1][c]);
              else
                *q = o[0][c];
            }
          }
        }
        if (two_scales) {
          float lin1[3];
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            lin1[c] = __fmul_rn(acc[c], 0.25f);
            L1[3 * img + c][rp * 32 + lane] = lin1[c];
          }
          float *P = P1 + (y1 * pitch1 + x1);
          float xo, yo, bo;
          pixel_xyb(px, cb, lin1[0], lin1[1], lin1[2], xo, yo, bo);
          P[(3 * img + 0) * plane1] = xo;
          P[(3 * img + 1) * plane1] = yo;
          P[(3 * img + 2) * plane1] = bo;
          if (dbg1) {
            const long long n1 = (long long)g.ws[1] * g.hs[1];
            const long long q = (long long)y1 * g.ws[1] + x1;
#pragma unroll
            for (int c = 0; c < 3; ++c) lin_dbg[(3 * img + c) * n1 + q] = lin1[c];
          }
        }
      }
    }
    __syncwarp();  // buffer i & 1 is refilled by stage_rows(i + 2)
  }
  if (g.nscales <= 2) return;
  // every warp's staging reads and copies are done: the region holds
  // scales 2-5 from here on
  __syncthreads();

  // ---- scales 2..: halve the shared tile, then XYB ----
  for (int s = 2; s < g.nscales; ++s) {
    if (s == 3 && warp >= 2) return;  // 64 pixels: warps 0-1
    if (s == 4 && warp >= 1) return;  // 16 and 4 pixels: warp 0
    const int lw = 6 - s;             // log2 of the tile edge at scale s
    const int tw = 1 << lw;
    const int ox = tx0 >> s, oy = ty0 >> s;               // tile origin at scale s
    const int pox = tx0 >> (s - 1), poy = ty0 >> (s - 1);  // at scale s-1
    const int pw = 2 * tw;
    const int ww = g.ws[s - 1], hh = g.hs[s - 1];
    float *Ps = Xf + g.xoff[s];
    const int planes = (int)g.plane[s], pitchs = g.pitch[s];
    const int p = threadIdx.x;
    if (p < tw * tw) {
      const int lx = p & (tw - 1), ly = p >> lw;
      const int x = ox + lx, y = oy + ly;
      if (x < g.ws[s] && y < g.hs[s]) {
        const int x0 = 2 * x, x1 = min(2 * x + 1, ww - 1);
        const int y0 = 2 * y, y1 = min(2 * y + 1, hh - 1);
        const int i00 = (y0 - poy) * pw + (x0 - pox), i01 = (y0 - poy) * pw + (x1 - pox);
        const int i10 = (y1 - poy) * pw + (x0 - pox), i11 = (y1 - poy) * pw + (x1 - pox);
        float *P = Ps + (y * pitchs + x);
#pragma unroll 1
        for (int img = 0; img < 2; ++img) {
          float v[3];
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            const float *Lp = s == 2 ? L1[3 * img + c] : &Lr[3 * img + c][lvl_off(s - 1)];
            float t = __fadd_rn(Lp[i00], Lp[i01]);
            t = __fadd_rn(t, Lp[i10]);
            t = __fadd_rn(t, Lp[i11]);
            v[c] = __fmul_rn(t, 0.25f);
            Lr[3 * img + c][lvl_off(s) + p] = v[c];
          }
          float xo, yo, bo;
          pixel_xyb(px, cb, v[0], v[1], v[2], xo, yo, bo);
          P[(3 * img + 0) * planes] = xo;
          P[(3 * img + 1) * planes] = yo;
          P[(3 * img + 2) * planes] = bo;
          if (DBG && ps.dbg_scale == s) {
            const long long ns = (long long)g.ws[s] * g.hs[s];
            const long long q = (long long)y * g.ws[s] + x;
#pragma unroll
            for (int c = 0; c < 3; ++c) lin_dbg[(3 * img + c) * ns + q] = v[c];
          }
        }
      }
    }
    if (s + 1 < g.nscales) {
      if (s == 2)
        __syncthreads();
      else if (s == 3)
        asm volatile("bar.sync 1, 64;" ::: "memory");  // warps 0 and 1
      else
        __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------
// Recursive Gaussian step (shared by both passes): three resonators of one
// quantity.  prev = Y[i-1], cur = Y[i]; in = x[i+N] + x[i-N].
// ---------------------------------------------------------------------------

struct Res3 {
  float prev[3], cur[3];
};

__device__ __forceinline__ float res_step(Res3 &r, const Pix &px, float in) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    float u = __fmaf_rn(px.iir_g[k], in, -r.prev[k]);
    float n = __fmaf_rn(px.iir_c2[k], r.cur[k], u);
    r.prev[k] = r.cur[k];
    r.cur[k] = n;
  }
  return __fadd_rn(__fadd_rn(r.cur[0], r.cur[1]), r.cur[2]);
}

__device__ __forceinline__ void res_zero(Res3 &r) {
#pragma unroll
  for (int k = 0; k < 3; ++k) r.prev[k] = r.cur[k] = 0.0f;
}

// The same recursion on two quantities at once, in packed fp32 pairs
// (fma.rn.f32x2, add.rn.f32x2).  The pair instructions have no negation, so
// the state is kept as Z_t = s_t Y_t with the sign pattern s = (+, +, -, -)
// repeating over the step index t: s_t s_{t-2} = -1 for every t, so the
// -Y_{t-2} term becomes +Z_{t-2}, and the other two coefficients take a sign
// fixed by t mod 4 (c2 times s_t s_{t-1}: - for even t, + for odd; g times
// s_t).  Round-to-nearest is symmetric, so s_t Z_t and the returned sum
// times s_t equal the scalar recursion's values bit for bit.  m = t mod 4
// must fold to a constant at every call (the callers' loops are unrolled).
struct Res3x2 {
  f2 prev[3], cur[3];
};
struct ResConsts2 {
  f2 cp[3], cn[3], gp[3], gn[3];  // +c2, -c2, +g, -g in both halves
};

__device__ __forceinline__ void res2_init(Res3x2 &r, ResConsts2 &k, const Pix &px) {
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    r.prev[i] = r.cur[i] = f2_pack(0.0f, 0.0f);
    k.cp[i] = f2_pack(px.iir_c2[i], px.iir_c2[i]);
    k.cn[i] = f2_pack(-px.iir_c2[i], -px.iir_c2[i]);
    k.gp[i] = f2_pack(px.iir_g[i], px.iir_g[i]);
    k.gn[i] = f2_pack(-px.iir_g[i], -px.iir_g[i]);
  }
}

// One step at t = m mod 4; returns s_t times the output sum (Y0 + Y1) + Y2.
__device__ __forceinline__ f2 res2_step(Res3x2 &r, const ResConsts2 &k, int m, f2 in) {
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const f2 cc = (m & 1) ? k.cp[i] : k.cn[i];
    const f2 gg = (m & 2) ? k.gn[i] : k.gp[i];
    const f2 n = f2_fma(cc, r.cur[i], f2_fma(gg, in, r.prev[i]));
    r.prev[i] = r.cur[i];
    r.cur[i] = n;
  }
  return f2_add(f2_add(r.cur[0], r.cur[1]), r.cur[2]);
}

// ---------------------------------------------------------------------------
// k_hblur: one warp per 32 rows of one (frame, scale, channel); lane = row.
//
// The rows are walked left to right in chunks of 8 columns.  TMA brings each
// chunk of the two XYB planes (x1, x2) into a kHSlots-slot shared-memory ring
// (8 x 32 floats per plane, zero-filled outside the image, which is exactly
// the recursion's zero extension), up to kHSlots - 1 chunks ahead of the walk.
// Each lane reads its row with 16-byte loads; the recursion needs the
// samples 5 ahead and 5 behind the step (the window of radius R = 4 has
// taps at +-(R+1)), kept in rolling registers.  The five quantities
// (x1, x2, x1^2, x2^2, x1 x2) are formed in registers.  The chunk's 5 x 8
// outputs per lane go to a ring of kHOutBufs shared tiles (mu1, mu2, s11,
// s22 as one float4 per pixel, s12 on its own) and leave with two TMA
// stores (clipped to the image), so global traffic is whole boxes both ways;
// a tile is rewritten once the store issued from it kHOutBufs chunks earlier
// has read it.  Every mbarrier wait is bounded; a timeout raises
// kErrTmaTimeout.
// ---------------------------------------------------------------------------

// Two-warp blocks of 46 KB (23 KB per warp): four per SM.  Measured at 4K
// against four-warp blocks with two output tiles (three per SM), the third
// tile takes the stall on the previous stores' reads out of the walk (2.69
// -> 2.50 ms per 7-frame launch inside the pipeline); one-warp blocks, six
// or eight input slots and two output tiles all measured slower.
constexpr int kHWarps = 2;
constexpr int kHSlots = 4;
constexpr int kHOutBufs = 3;
constexpr int kHBox = kBoxRows * kBoxCols;  // floats in one plane box (1 KB)

// Output tiles: per buffer, the quads (mu1, mu2, s11, s22) of the 32 x 8
// pixels in the 128-byte-swizzled order their TMA map expects (16-byte unit
// swz128(row * 8 + col)), then the s12 tile.
struct HWarpSmem {
  float quad[kHOutBufs][4 * kHBox];  // [buffer][swizzled (row, col), quantity 0..3]
  float s12[kHOutBufs][kHBox];       // [buffer][32-byte-swizzled (row, col)]
  float in[kHSlots][2][kHBox];       // [slot][x1 | x2][32-byte-swizzled (row, col)]
};
static_assert(sizeof(HWarpSmem) % 1024 == 0, "every quad tile starts on 1024 bytes");
// warp tiles, then the mbarriers; +1024 to align the base for the swizzle
constexpr int kHSmemBytes = kHWarps * (int)sizeof(HWarpSmem) + kHWarps * kHSlots * 8 + 1024;

__global__ void __launch_bounds__(kHWarps * 32)
    k_hblur(Geom g, Pix px, const __grid_constant__ HMaps maps, int nframes,
            int *__restrict__ err) {
  extern __shared__ __align__(16) unsigned char hsm_raw[];
  unsigned char *hsm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(hsm_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // units in scale-major order over the batch (every frame's scale-0 rows
  // first): the longest walks start first and the shortest fill the tail
  const int gu = blockIdx.x * kHWarps + warp;
  if (gu >= g.hunit_off[g.nscales] * nframes) return;  // whole warp
  int s = 0;
  while (gu >= g.hunit_off[s + 1] * nframes) ++s;
  const int ns = g.hunit_off[s + 1] - g.hunit_off[s];
  const int frame = (gu - g.hunit_off[s] * nframes) / ns;
  const int local = (gu - g.hunit_off[s] * nframes) % ns;
  const int nrb = (g.hs[s] + kBoxRows - 1) / kBoxRows;
  const int c = local / nrb, row0 = (local % nrb) * kBoxRows;
  const int nchunk = (g.ws[s] + kBoxCols - 1) / kBoxCols;
  HWarpSmem &sm = reinterpret_cast<HWarpSmem *>(hsm)[warp];
  uint64_t *bar = reinterpret_cast<uint64_t *>(hsm + kHWarps * sizeof(HWarpSmem)) + warp * kHSlots;
  const CUtensorMap *mx = &maps.x[s];
  const CUtensorMap *mq = &maps.q4[s];
  const CUtensorMap *ms = &maps.s1[s];

  if (lane == 0) {
    for (int i = 0; i < kHSlots; ++i) mbar_init(&bar[i], 1);
    fence_barrier_init();
  }
  __syncwarp();
  // chunk m (columns 8m .. 8m+7) of both planes -> slot m % kHSlots
  auto issue = [&](int m) {
    const int slot = m % kHSlots;
    mbar_arrive_expect_tx(&bar[slot], 2 * kHBox * (int)sizeof(float));
    tma_load_4d(sm.in[slot][0], mx, &bar[slot], m * kBoxCols, row0, c, frame);
    tma_load_4d(sm.in[slot][1], mx, &bar[slot], m * kBoxCols, row0, 3 + c, frame);
  };
  if (lane == 0)
    for (int m = 0; m < kHSlots && m <= nchunk; ++m) issue(m);
  auto wait_chunk = [&](int m) -> bool {
    const bool ok = mbar_wait(&bar[m % kHSlots], (uint32_t)(m / kHSlots) & 1u);
    return __all_sync(0xffffffffu, ok);
  };
  auto bail = [&]() {
    if (lane == 0) {
      atomicOr(err, kErrTmaTimeout);
      bulk_wait<0>();
    }
  };

  // (mu1, mu2) and (s11, s22) recurse as packed pairs, s12 alone
  Res3x2 rm, rs;
  ResConsts2 rk;
  res2_init(rm, rk, px);
  res2_init(rs, rk, px);
  Res3 r12;
  res_zero(r12);
  const f2 zero2 = f2_pack(0.0f, 0.0f);

  // rolling 4-column groups of both planes: gm0 = cols 8k-8..8k-5,
  // gm1 = 8k-4..8k-1, g0 = 8k..8k+3 (all zero before column 0)
  float4 gm0[2], gm1[2], g0[2];
  if (!wait_chunk(0)) { bail(); return; }
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    gm0[p] = make_float4(0.f, 0.f, 0.f, 0.f);
    gm1[p] = gm0[p];
    g0[p] = reinterpret_cast<const float4 *>(sm.in[0][p])[swz32(2 * lane)];
  }
  // warm-up steps producing Y[-4] .. Y[-1]: inputs x[0..3] ahead, zeros behind
  {
    const float a1[4] = {g0[0].x, g0[0].y, g0[0].z, g0[0].w};
    const float a2[4] = {g0[1].x, g0[1].y, g0[1].z, g0[1].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // steps t = 0..3
      res2_step(rm, rk, j, f2_add(f2_pack(a1[j], a2[j]), zero2));
      res2_step(rs, rk, j, f2_add(f2_pack(__fmul_rn(a1[j], a1[j]), __fmul_rn(a2[j], a2[j])), zero2));
      res_step(r12, px, __fadd_rn(__fmul_rn(a1[j], a2[j]), 0.0f));
    }
  }

  for (int k = 0; k < nchunk; ++k) {
    if (!wait_chunk(k + 1)) { bail(); return; }
    const int sk = k % kHSlots, sk1 = (k + 1) % kHSlots;
    float4 g1[2], gn[2];  // cols 8k+4..8k+7 and 8k+8..8k+11
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      g1[p] = reinterpret_cast<const float4 *>(sm.in[sk][p])[swz32(2 * lane + 1)];
      gn[p] = reinterpret_cast<const float4 *>(sm.in[sk1][p])[swz32(2 * lane)];
    }
    // slot k is free once every lane's reads of it are ordered before the
    // copy that refills it: the reads are generic-proxy accesses and the
    // copy writes through the async proxy, so a proxy fence precedes the
    // warp barrier (without it a read still in flight under heavy
    // shared-memory traffic could return the refilled data)
    fence_async_smem();
    __syncwarp();
    if (lane == 0 && k + kHSlots <= nchunk) issue(k + kHSlots);
    f2 om[kBoxCols], os[kBoxCols];  // (mu1, mu2), (s11, s22)
    float o12[kBoxCols];
    {
      // step producing Y[8k + j] takes x[8k + j + 4] + x[8k + j - 6]
      const float ah1[8] = {g1[0].x, g1[0].y, g1[0].z, g1[0].w, gn[0].x, gn[0].y, gn[0].z, gn[0].w};
      const float ah2[8] = {g1[1].x, g1[1].y, g1[1].z, g1[1].w, gn[1].x, gn[1].y, gn[1].z, gn[1].w};
      const float bh1[8] = {gm0[0].z, gm0[0].w, gm1[0].x, gm1[0].y, gm1[0].z, gm1[0].w, g0[0].x, g0[0].y};
      const float bh2[8] = {gm0[1].z, gm0[1].w, gm1[1].x, gm1[1].y, gm1[1].z, gm1[1].w, g0[1].x, g0[1].y};
#pragma unroll
      for (int j = 0; j < kBoxCols; ++j) {
        // step t = 4 + 8k + j, so t mod 4 = j mod 4; the pairs carry s_t,
        // taken off by 0 - v where s_t = -1 (a zero stays +0, as in the
        // scalar recursion)
        // (the squares are scalar products: a pair product feeding a pair
        // sum is contracted into one fused operation, which would skip the
        // squares' own rounding)
        const f2 sa = f2_pack(__fmul_rn(ah1[j], ah1[j]), __fmul_rn(ah2[j], ah2[j]));
        const f2 sb = f2_pack(__fmul_rn(bh1[j], bh1[j]), __fmul_rn(bh2[j], bh2[j]));
        om[j] = res2_step(rm, rk, j, f2_add(f2_pack(ah1[j], ah2[j]), f2_pack(bh1[j], bh2[j])));
        os[j] = res2_step(rs, rk, j, f2_add(sa, sb));
        if (j & 2) {
          om[j] = f2_sub(zero2, om[j]);
          os[j] = f2_sub(zero2, os[j]);
        }
        o12[j] = res_step(r12, px, __fadd_rn(__fmul_rn(ah1[j], ah2[j]), __fmul_rn(bh1[j], bh2[j])));
      }
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      gm0[p] = g0[p];
      gm1[p] = g1[p];
      g0[p] = gn[p];
    }
    // the store issued from this buffer kHOutBufs chunks ago must have read it
    if (lane == 0) bulk_wait_read<kHOutBufs - 1>();
    __syncwarp();
    const int ob = k % kHOutBufs;
    // lane = row: column j's quad is 16-byte unit row * 8 + j of the tile
    // (eight lanes of a phase hit eight different units of their lines)
    float4 *dq = reinterpret_cast<float4 *>(sm.quad[ob]);
#pragma unroll
    for (int j = 0; j < kBoxCols; ++j) {
      float4 v;
      f2_unpack(om[j], v.x, v.y);
      f2_unpack(os[j], v.z, v.w);
      dq[swz128(lane * kBoxCols + j)] = v;
    }
    float4 *ds = reinterpret_cast<float4 *>(sm.s12[ob]);
    ds[swz32(2 * lane)] = make_float4(o12[0], o12[1], o12[2], o12[3]);
    ds[swz32(2 * lane + 1)] = make_float4(o12[4], o12[5], o12[6], o12[7]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_4d(mq, sm.quad[ob], 4 * k * kBoxCols, row0, c, frame);
      tma_store_4d(ms, sm.s12[ob], k * kBoxCols, row0, c, frame);
      bulk_commit();
    }
  }
  if (lane == 0) bulk_wait<0>();
}

// ---------------------------------------------------------------------------
// k_vblur: one warp per 32 columns of one (scale, channel) of a frame; each
// lane walks its column, forms the map terms at every output row and keeps
// six float-pair sums, then a fixed shuffle tree gives one pair per warp.
// ---------------------------------------------------------------------------

// Six float-pair sums per lane.  An addition keeps the high word exact
// (two_sum) and folds the rounding error and the term's low word into the
// low word without renormalising; acc_renorm restores |lo| <= ulp(hi)/2
// once per chunk of rows, which bounds the low word's own rounding.
struct Acc6 {
  ff v[kNSum];
};

// Every sum and every term here is non-negative (d, d^4, |r|, r^4 and their
// running sums), so the exact error of hi + hi comes from Dekker's
// quick_two_sum on (max, min): the same two words as Knuth's two_sum, one
// instruction fewer.
__device__ __forceinline__ ff acc_add(ff s, ff t) {
  const float a = fmaxf(s.hi, t.hi), b = fminf(s.hi, t.hi);
  const ff h = quick_two_sum(a, b);
  return {h.hi, __fadd_rn(s.lo, __fadd_rn(h.lo, t.lo))};
}

__device__ __forceinline__ void acc_renorm(Acc6 &a) {
#pragma unroll
  for (int k = 0; k < kNSum; ++k) a.v[k] = quick_two_sum(a.v[k].hi, a.v[k].lo);
}

__device__ __forceinline__ void ssim_edge_terms(const Pix &px, float mu1, float mu2, float s11,
                                                float s22, float s12, float x1, float x2,
                                                Acc6 &acc) {
  // ssim_map (fp32 part as the CPU computes it)
  const float dm = __fsub_rn(mu1, mu2);
  const float num_m = __fsub_rn(1.0f, __fmul_rn(dm, dm));
  const float cov = __fsub_rn(s12, __fmul_rn(mu1, mu2));
  const float num_s = __fadd_rn(__fmul_rn(2.0f, cov), px.c2);
  const float v1 = __fsub_rn(s11, __fmul_rn(mu1, mu1));
  const float v2 = __fsub_rn(s22, __fmul_rn(mu2, mu2));
  const float den_s = __fadd_rn(__fadd_rn(v1, v2), px.c2);
  // float-pair part: d = max(1 - num_m num_s / den_s, 0), formed as
  // (den_s - num_m num_s) / den_s with the product exact as a pair and the
  // numerator's leading difference exact (two_sum)
  // den_s - p.hi exactly: quick_two_sum on (max, min) is exact whenever the
  // larger operand has the larger magnitude, which holds for every outcome
  // that survives the clamp below (den_s > 0: either -p.hi >= 0, or
  // -p.hi < 0 with |p.hi| <= den_s, else the difference is negative and d
  // is clamped to zero)
  const ff p = two_prod(num_m, num_s);
  const ff nd = quick_two_sum(fmaxf(den_s, -p.hi), fminf(den_s, -p.hi));
  ff d = ff_div_f(quick_two_sum(nd.hi, __fsub_rn(nd.lo, p.lo)), den_s);
  if (!(d.hi > 0.0f)) d = {0.0f, 0.0f};
  const ff d2 = ff_sqr_lazy(d);
  const ff d4 = ff_sqr_lazy(d2);
  acc.v[0] = acc_add(acc.v[0], d);
  acc.v[1] = acc_add(acc.v[1], d4);
  // edge_diff_map: r = (1 + a2) / (1 + a1) - 1 = (a2 - a1) / (1 + a1), with
  // a = |x - mu|; the numerator and denominator are exact pairs
  const float a2 = fabsf(__fsub_rn(x2, mu2));
  const float a1 = fabsf(__fsub_rn(x1, mu1));
  // 1 + a1 with a1 >= 0: quick_two_sum on (max, min) is exact
  const ff r = ff_div(two_sum(a2, -a1), quick_two_sum(fmaxf(1.0f, a1), fminf(1.0f, a1)));
  const ff r2 = ff_sqr_lazy(r);
  const ff r4 = ff_sqr_lazy(r2);
  // artifact (r > 0) and detail lost (r < 0) are exclusive: one addition each
  // into the sum that the sign selects (r = 0 adds zero to detail lost)
  const bool pos = r.hi > 0.0f;
  const ff ar = pos ? r : ff{-r.hi, -r.lo};
  ff s1 = pos ? acc.v[2] : acc.v[4];
  ff s4 = pos ? acc.v[3] : acc.v[5];
  s1 = acc_add(s1, ar);
  s4 = acc_add(s4, r4);
  if (pos) {
    acc.v[2] = s1;
    acc.v[3] = s4;
  } else {
    acc.v[4] = s1;
    acc.v[5] = s4;
  }
}

// Column walkers.  One warp per 32 columns of one (frame, scale, channel);
// lane = column.  TMA brings 8-row chunks of the channel's blurred planes
// (a 32 x 8 box of quads and one of s12) into a 3-slot ring, so a tap is
// one 16-byte and one 4-byte shared load; the slot of chunk k - 1 is
// refilled with chunk k + 2 as soon as its last row has been read (after
// step 5 of chunk k), six steps before that chunk is first needed.  The two
// XYB rows each step needs are loaded from global memory one chunk ahead
// into registers.  Step n of the recursion takes rows n+4 and n-6 of the
// blurred planes (taps at +-(R+1)); its outputs mu1, mu2, s11, s22, s12
// feed the SSIM and edge terms of row n at once, so the vertically blurred
// planes never exist in memory.
constexpr int kVWarps = 4;
constexpr int kVSlots = 3;
constexpr int kVBox = kVRows * kVCols;          // floats per plane box (1 KB)

// Per slot: the quads (mu1, mu2, s11, s22) of the 8 x 32 pixels, then the
// s12 box.
struct VWarpSmem {
  float quad[kVSlots][4 * kVBox];  // [slot][(row * 32 + col) * 4 + quantity]
  float s12[kVSlots][kVBox];       // [slot][row * 32 + col]
};
static_assert(sizeof(VWarpSmem) == 15360, "per-warp tiles");
constexpr int kVSmemBytes = kVWarps * (int)sizeof(VWarpSmem) + kVWarps * 4 * 8 + 1024;

__global__ void __launch_bounds__(kVWarps * 32)
    k_vblur(Geom g, Pix px, const __grid_constant__ VMaps maps, const float *__restrict__ X,
            int nframes, float2 *__restrict__ part, int *__restrict__ err) {
  extern __shared__ __align__(16) unsigned char vsm_raw[];
  unsigned char *vsm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(vsm_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // column walkers in scale-major order over the batch (every frame's
  // scale-0 columns first): the longest walks start first
  const int gw = blockIdx.x * kVWarps + warp;
  if (gw >= g.vwarp_off[g.nscales] * nframes) return;  // whole warp exits together
  int s = 0;
  while (gw >= g.vwarp_off[s + 1] * nframes) ++s;
  const int ns = g.vwarp_off[s + 1] - g.vwarp_off[s];
  const int frame = (gw - g.vwarp_off[s] * nframes) / ns;
  const int local = (gw - g.vwarp_off[s] * nframes) % ns;
  const int c = local % 3, cb = local / 3;
  const int col0 = cb * kVCols;
  const bool active = col0 + lane < g.ws[s];
  const int h = g.hs[s];
  const int nchunk = (h + kVRows - 1) / kVRows;
  VWarpSmem &sm = reinterpret_cast<VWarpSmem *>(vsm)[warp];
  uint64_t *hbar = reinterpret_cast<uint64_t *>(vsm + kVWarps * sizeof(VWarpSmem)) + warp * 4;
  const CUtensorMap *mq = &maps.vq4[s];
  const CUtensorMap *ms = &maps.vs1[s];
  // XYB rows of this lane's column (pitch padding keeps every lane in bounds)
  // (32-bit indices inside this (frame, scale) block: its six planes hold at
  // most 6 x 2^28 floats)
  const int pitch = g.pitch[s];
  const float *xs = X + (long long)frame * g.x_fs + g.xoff[s];
  const int xi1 = c * (int)g.plane[s] + col0 + lane, xi2 = xi1 + 3 * (int)g.plane[s];

  if (lane == 0) {
    for (int i = 0; i < kVSlots; ++i) mbar_init(&hbar[i], 1);
    fence_barrier_init();
  }
  __syncwarp();
  // blurred-plane chunk m (rows 8m .. 8m+7), m >= -1, lives in slot (m+1) % 3
  auto slot_of = [](int m) { return (m + 1) % kVSlots; };
  auto issue_h = [&](int m) {
    const int slot = slot_of(m);
    mbar_arrive_expect_tx(&hbar[slot], kNq * kVBox * (int)sizeof(float));
    tma_load_4d(sm.quad[slot], mq, &hbar[slot], 4 * col0, m * kVRows, c, frame);
    tma_load_4d(sm.s12[slot], ms, &hbar[slot], col0, m * kVRows, c, frame);
  };
  if (lane == 0)
    for (int m = -1; m <= 1 && m <= nchunk; ++m) issue_h(m);
  auto wait_h = [&](int m) -> bool {
    const bool ok = mbar_wait(&hbar[slot_of(m)], (uint32_t)((m + 1) / kVSlots) & 1u);
    return __all_sync(0xffffffffu, ok);
  };
  auto load_x = [&](int m, float (&xa)[kVRows], float (&xb)[kVRows]) {
#pragma unroll
    for (int j = 0; j < kVRows; ++j) {
      const int row = m * kVRows + j;
      xa[j] = row < h ? __ldg(xs + (xi1 + row * pitch)) : 0.0f;
      xb[j] = row < h ? __ldg(xs + (xi2 + row * pitch)) : 0.0f;
    }
  };

  Acc6 acc;
#pragma unroll
  for (int k = 0; k < kNSum; ++k) acc.v[k] = {0.0f, 0.0f};
  // (mu1, mu2) and (s11, s22) recurse as packed pairs, s12 alone
  Res3x2 rm, rs;
  ResConsts2 rk;
  res2_init(rm, rk, px);
  res2_init(rs, rk, px);
  Res3 r12;
  res_zero(r12);
  const f2 zero2 = f2_pack(0.0f, 0.0f);
  // this lane's quad of row r of a slot as two pairs
  auto pairs_at = [&](int slot, int r) -> ulonglong2 {
    return reinterpret_cast<const ulonglong2 *>(sm.quad[slot])[r * kVCols + lane];
  };
  float xc1[kVRows], xc2[kVRows];
  load_x(0, xc1, xc2);

  if (!wait_h(-1) || !wait_h(0)) {
    if (lane == 0) atomicOr(err, kErrTmaTimeout);
    return;
  }
  // warm-up steps producing Y[-4] .. Y[-1]: rows 0..3 ahead, zeros behind
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // steps t = 0..3
    const ulonglong2 a = pairs_at(slot_of(0), j);
    res2_step(rm, rk, j, f2_add(a.x, zero2));
    res2_step(rs, rk, j, f2_add(a.y, zero2));
    res_step(r12, px, __fadd_rn(sm.s12[slot_of(0)][j * kVCols + lane], 0.0f));
  }

  for (int k = 0; k < nchunk; ++k) {
    if (!wait_h(k + 1)) {
      if (lane == 0) atomicOr(err, kErrTmaTimeout);
      return;
    }
    float xn1[kVRows], xn2[kVRows];
    load_x(k + 1, xn1, xn2);
    const int sp = slot_of(k - 1), sk = slot_of(k), sn = slot_of(k + 1);
#pragma unroll
    for (int j = 0; j < kVRows; ++j) {
      // ahead row 8k + j + 4, behind row 8k + j - 6
      const int sa = j < 4 ? sk : sn, ra = j < 4 ? j + 4 : j - 4;
      const int sb = j < 6 ? sp : sk, rb = j < 6 ? j + 2 : j - 6;
      const ulonglong2 qa = pairs_at(sa, ra), qb = pairs_at(sb, rb);
      // step t = 4 + 8k + j, so t mod 4 = j mod 4; the pairs carry s_t
      const f2 om = res2_step(rm, rk, j, f2_add(qa.x, qb.x));
      const f2 os = res2_step(rs, rk, j, f2_add(qa.y, qb.y));
      float o[kNq];
      f2_unpack(om, o[0], o[1]);
      f2_unpack(os, o[2], o[3]);
      if (j & 2) {
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = -o[q];
      }
      o[4] = res_step(r12, px, __fadd_rn(sm.s12[sa][ra * kVCols + lane], sm.s12[sb][rb * kVCols + lane]));
      if (j == 5) {
        // chunk k - 1 is read for the last time: refill its slot with k + 2
        // (the reads are ordered before the async-proxy refill by a proxy
        // fence and the warp barrier)
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && k + 2 <= nchunk) issue_h(k + 2);
      }
      if (active && k * kVRows + j < h)
        ssim_edge_terms(px, o[0], o[1], o[2], o[3], o[4], xc1[j], xc2[j], acc);
    }
    acc_renorm(acc);
#pragma unroll
    for (int j = 0; j < kVRows; ++j) {
      xc1[j] = xn1[j];
      xc2[j] = xn2[j];
    }
  }
  // fixed tree: lane l adds lane l + 2^m for m = 4..0
#pragma unroll
  for (int k = 0; k < kNSum; ++k) {
    ff v = acc.v[k];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      ff o;
      o.hi = __shfl_down_sync(0xffffffffu, v.hi, off);
      o.lo = __shfl_down_sync(0xffffffffu, v.lo, off);
      v = ff_add(v, o);
    }
    if (lane == 0) {
      part[(long long)frame * g.p_fs + g.poff[s] + (c * kNSum + k) * g.nw[s] + cb] =
          make_float2(v.hi, v.lo);
    }
  }
}

// ---------------------------------------------------------------------------
// k_finalize: one block per frame.  Thread j < 108 owns value j: it adds the
// warp partials of its (scale, channel, sum) in index order, forms the
// 1-norm (mean) or 4-norm (fourth root of the mean fourth power) in fp64 and
// its pooling term w_j |v_j|.  Thread 0 pools: P = sum_i w_i |v_i| in index
// order (the terms formed in parallel, the additions one after another, as
// the sequential sum rounds them), then the map.
// With an error word given and set, the batch's values and scores are NaN.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128)
    k_finalize(Geom g, const float2 *__restrict__ part, const double *__restrict__ params,
               double *__restrict__ values, double *__restrict__ scores,
               const int *__restrict__ err) {
  __shared__ double wv[kNValues];  // the pooling terms w_j |v_j|
  const int frame = blockIdx.x;
  const int j = threadIdx.x;
  if (err && *err != 0) {
    const double nan = __longlong_as_double(0x7ff8000000000000LL);
    if (j < kNValues) values[(long long)frame * kNValues + j] = nan;
    if (j == 0) scores[frame] = nan;
    return;
  }
  if (j < kNValues) {
    const int kind = j % 3, n = (j / 3) % 2, s = (j / 6) % 6, c = j / 36;
    double out = 0.0;
    if (s < g.nscales) {
      const int k = 2 * kind + n;
      const float2 *p = part + (long long)frame * g.p_fs + g.poff[s] + (c * kNSum + k) * g.nw[s];
      ff acc = {0.0f, 0.0f};
      for (int i = 0; i < g.nw[s]; ++i) {
        const float2 t = p[i];
        acc = ff_add(acc, ff{t.x, t.y});
      }
      const double S = (double)acc.hi + (double)acc.lo;
      const double N = (double)g.ws[s] * (double)g.hs[s];
      out = n == 0 ? S / N : sqrt(sqrt(S / N));
    }
    values[(long long)frame * kNValues + j] = out;
    wv[j] = params[kPWeights + j] * fabs(out);
  }
  __syncthreads();
  if (j == 0) {
    double P = 0.0;
    for (int i = 0; i < kNValues; ++i) P = P + wv[i];
    const double *pc = params + kPPoly;
    double sc = pc[3] * P;
    sc = sc + pc[2];
    sc = sc * P;
    sc = sc + pc[1];
    sc = sc * P;
    sc = sc + pc[0];
    const double *pw = params + kPPower;
    if (sc > 0.0) {
      double t = pw[1] == 1.0 ? sc : pow(sc, pw[1]);
      t = pw[0] * t;
      sc = t + pw[2];
    }
    scores[frame] = sc;
  }
}

// ---------------------------------------------------------------------------
// k_cbrt: the pipeline's cube root on an array (checks against the oracle).
// ---------------------------------------------------------------------------

__global__ void k_cbrt(const float *__restrict__ x, float *__restrict__ y, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float v = x[i];
    y[i] = v >= 0.0f && v < __int_as_float(0x7f800000) ? cbrt_cr(v) : v;
  }
}

// ---------------------------------------------------------------------------
// k_wait_probe: a barrier phase that nothing completes (one arrival with a
// transaction count that no copy ever delivers); the bounded wait must give
// up, raise the error bit and return.
// ---------------------------------------------------------------------------

__global__ void k_wait_probe(uint32_t spins, int *__restrict__ err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar, 1024);
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0, spins);
  if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicOr(err, kErrTmaTimeout);
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

cudaError_t launch_wait_probe(uint32_t spins, int *err, cudaStream_t st) {
  k_wait_probe<<<1, 32, 0, st>>>(spins, err);
  return cudaGetLastError();
}

cudaError_t launch_cbrt(const float *x, float *y, long long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long long blocks = std::min<long long>((n + 255) / 256, 152LL * 16);
  k_cbrt<<<(unsigned)blocks, 256, 0, st>>>(x, y, n);
  return cudaGetLastError();
}

// Dynamic shared memory of one instantiation: the scale-1 tiles, the region
// shared by the staging buffers and the scale 2-5 tiles, and the 8-bit
// normalisation tables.
template <int BPS, int SX, int SY>
constexpr int pyr_smem() {
  return (int)sizeof(float) * (6 * kLvl1 + (BPS == 1 ? 512 : 0)) +
         StageGeo<BPS, SX, SY>::union_bytes;
}

template <int BPS, int SX, int SY, bool DBG>
static cudaError_t launch_pyr_dbg(const Geom &g, const Pix &px, const PyrTabs &tabs,
                                  PyrStage ps, const uint8_t *ref, const uint8_t *dis, float *X,
                                  float *lin_dbg, int nframes, cudaStream_t st) {
  constexpr int smem = pyr_smem<BPS, SX, SY>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> configured[64];
  if (dev < 64 && !configured[dev].load()) {
    e = cudaFuncSetAttribute(k_pyramid<BPS, SX, SY, DBG>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev].store(true);
  }
  dim3 grid((g.w + kPT - 1) / kPT, (g.h + kPT - 1) / kPT, nframes);
  k_pyramid<BPS, SX, SY, DBG>
      <<<grid, kPyrThreads, smem, st>>>(g, px, tabs, ps, ref, dis, X, lin_dbg);
  return cudaGetLastError();
}

// The linear-RGB dump of the parity tests is a separate instantiation: the
// scoring kernels carry no trace of it.
template <int BPS, int SX, int SY>
static cudaError_t launch_pyr(const Geom &g, const Pix &px, const PyrTabs &tabs, PyrStage ps,
                              const uint8_t *ref, const uint8_t *dis, float *X, float *lin_dbg,
                              int nframes, cudaStream_t st) {
  if (lin_dbg)
    return launch_pyr_dbg<BPS, SX, SY, true>(g, px, tabs, ps, ref, dis, X, lin_dbg, nframes, st);
  return launch_pyr_dbg<BPS, SX, SY, false>(g, px, tabs, ps, ref, dis, X, nullptr, nframes, st);
}

cudaError_t launch_pyramid(const Geom &g, const Pix &px, const PyrTabs &tabs, const uint8_t *ref,
                           const uint8_t *dis, float *X, int nframes, cudaStream_t st,
                           float *lin_dbg, int dbg_scale) {
  PyrStage ps;
  // every staged row starts on 16 bytes: frame bases, plane offsets and row
  // pitches of both planes, and the tile origins (multiples of 64 samples)
  ps.vec = (reinterpret_cast<uintptr_t>(ref) % 16 == 0) &&
           (reinterpret_cast<uintptr_t>(dis) % 16 == 0) && g.frame_bytes % 16 == 0 &&
           (g.w * g.bps) % 16 == 0 && (g.cw * g.bps) % 16 == 0;
  ps.dbg_scale = lin_dbg ? dbg_scale : -1;
  const int layout = g.sx * 2 + g.sy;  // 3: 4:2:0, 2: 4:2:2, 0: 4:4:4
  if (g.bps == 1) {
    if (layout == 3) return launch_pyr<1, 1, 1>(g, px, tabs, ps, ref, dis, X, lin_dbg, nframes, st);
    if (layout == 2) return launch_pyr<1, 1, 0>(g, px, tabs, ps, ref, dis, X, lin_dbg, nframes, st);
    return launch_pyr<1, 0, 0>(g, px, tabs, ps, ref, dis, X, lin_dbg, nframes, st);
  }
  if (layout == 3) return launch_pyr<2, 1, 1>(g, px, tabs, ps, ref, dis, X, lin_dbg, nframes, st);
  if (layout == 2) return launch_pyr<2, 1, 0>(g, px, tabs, ps, ref, dis, X, lin_dbg, nframes, st);
  return launch_pyr<2, 0, 0>(g, px, tabs, ps, ref, dis, X, lin_dbg, nframes, st);
}

cudaError_t launch_hblur(const Geom &g, const Pix &px, const PlaneMaps &maps, int *err,
                         int nframes, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> configured[64];
  if (dev < 64 && !configured[dev].load()) {
    e = cudaFuncSetAttribute(k_hblur, cudaFuncAttributeMaxDynamicSharedMemorySize, kHSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(true);
  }
  const int units = g.hunit_off[g.nscales];
  const dim3 grid((units * nframes + kHWarps - 1) / kHWarps);
  k_hblur<<<grid, kHWarps * 32, kHSmemBytes, st>>>(g, px, maps.h, nframes, err);
  return cudaGetLastError();
}

cudaError_t launch_vblur(const Geom &g, const Pix &px, const PlaneMaps &maps, const float *X,
                         float2 *part, int *err, int nframes, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> configured[64];
  if (dev < 64 && !configured[dev].load()) {
    e = cudaFuncSetAttribute(k_vblur, cudaFuncAttributeMaxDynamicSharedMemorySize, kVSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(true);
  }
  const int warps = g.vwarp_off[g.nscales];
  const dim3 grid((warps * nframes + kVWarps - 1) / kVWarps);
  k_vblur<<<grid, kVWarps * 32, kVSmemBytes, st>>>(g, px, maps.v, X, nframes, part, err);
  return cudaGetLastError();
}

// k_finalize is launched at the device's highest priority: its few blocks
// then take the next free SM slots ahead of the other lane's pending blocks,
// and the lane's stream moves on to its next batch sooner.
cudaError_t launch_finalize(const Geom &g, const float2 *part, const double *params,
                            double *values, double *scores, int nframes, cudaStream_t st,
                            const int *err) {
  // numerically lowest priority value, read once (thread-safe initialisation)
  static const std::pair<cudaError_t, int> greatest = [] {
    int least = 0, hi = 0;
    const cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &hi);
    return std::make_pair(e, hi);
  }();
  if (greatest.first != cudaSuccess) return greatest.first;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nframes);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributePriority;
  attr[0].val.priority = greatest.second;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_finalize, g, part, params, values, scores, err);
}

}  // namespace ss2
