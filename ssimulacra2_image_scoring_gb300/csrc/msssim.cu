// msssim.cu — MS-SSIM on the device (ss2_msssim_* in include/ss2.h): of the
// luma plane, and with enable_chroma of the Cb and Cr planes as well, each
// on its own at chroma resolution.
//
// Source: "Research-1363: Device-resident ssimulacra2 and a single-wait
// MS-SSIM on SYCL" (vmafx documentation), Finding 6: every scale of a frame
// is enqueued at once, each (plane, scale) has a span of partial sums of its
// own, and the host waits once; the outputs are the default score, the
// per-scale terms (enable_lcs) and the chroma planes (enable_chroma).  The method is Wang, Simoncelli and Bovik,
// "Multi-scale structural similarity for image quality assessment" (2003):
// five scales of a 2x2-average pyramid (edge sample repeated), the SSIM
// statistics of an 11x11 Gaussian window (sigma 1.5) wherever it fits,
// K1 = 0.01, K2 = 0.03, C3 = C2 / 2, L = 255 on samples in the 8-bit range
// (raw / 2^(depth - 8)); per scale the means of l, c, s, cs and l cs; the
// score prod_{j<5} mean(cs_j)^beta_j * mean(l cs)_5^beta_5 with the
// published exponents.
//
//   k_msssim_level  one launch per scale over the batch; a block walks a
//                   strip of 32 window positions across, down a band of up
//                   to 512 rows, 16 rows at a time: each step loads the 16
//                   new input rows of the 42-column strip (raw luma at
//                   scale 1, fp32 planes after), shifted by the band's
//                   first reference sample (variances and covariance do not
//                   change, cancellation does), keeps (p, q) and (p q, 0)
//                   per pixel, and forms the horizontal Gaussian sums of
//                   (p, q), its squares and (p q, 0) once into a 32-row
//                   ring, from which the vertical sums of the step's 16
//                   output rows are read (36 KB and 76 registers: six
//                   four-warp blocks per SM);
//                   the five Gaussian means in fp32 as three packed pairs
//                   (fma.rn.f32x2, products formed once per pixel); l, c,
//                   s, cs, l cs per position (approximate reciprocals and
//                   root refined to about an ulp); a thread takes four
//                   adjacent positions of a row (horizontal pass) and of a
//                   column (vertical pass); per step fp32 sums per warp
//                   (fixed tree), then fp64 over the steps and the block's
//                   four warps into the (frame, scale, block) span (fp64 is
//                   slow on this part).  It also writes its share of the
//                   next scale: 2x2 means, exact in fp32 (a level-5 value is
//                   at most 2^24 units of 2^-16, so every partial sum is
//                   representable).
//   k_msssim_final  per frame: each span summed in a fixed warp order, the
//                   means, and the product of powers (fp64).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/ss2.h"
#include "ss2_f32x2.cuh"
#include "ss2_host.h"

#define SS2_API extern "C" __attribute__((visibility("default")))

namespace {

using namespace ss2;

constexpr int kScales = 5;
constexpr int kQ = 5;                      // l, c, s, cs, l cs
constexpr int kWin = 11;
constexpr int kTX = 32;                    // window positions across a strip
constexpr int kIX = kTX + kWin - 1;        // input columns of a strip: 42
constexpr int kCH = 16;                    // output rows per step
constexpr int kBH = 512;                   // output rows per band (32 steps)
constexpr int kRing = 32;                  // rows of horizontal sums kept (>= kCH + kWin - 1)
constexpr int kHalo = kWin - 1;            // input rows ahead of a band's first step
constexpr int kLevelThreads = 128;         // 4 warps: 4 positions per thread in both passes
static_assert(kCH % 2 == 0 && kHalo % 2 == 0 && kBH % kCH == 0, "row pairs stay in one step");

struct MGeom {
  int w, h, depth, bps;          // the plane's size (luma, or a chroma plane)
  long long frame_bytes;
  long long plane_off;           // byte offset of the plane inside a frame
  float norm;                    // 2^(8 - depth)
  int ws[kScales], hs[kScales];  // plane size per scale
  int pitch[kScales];            // fp32 pitch of scales 2..5 (index 1..4)
  long long lvl_off[kScales];    // float offset of scales 2..5 in an image's pyramid
  long long img_floats;          // floats of one image's scales 2..5
  int tx[kScales], ty[kScales];  // tiles per scale
  int tile_off[kScales], tiles_total;
  float C1, C2, C3;
  float gauss[kWin];
  double beta[kScales];
};

// Sample (x, y) of image `img` of frame `frame` at scale j (MODE 0: raw
// 8-bit luma, 1: raw 16-bit luma, 2: an fp32 pyramid plane), 8-bit range.
template <int MODE>
__device__ __forceinline__ float sample(const MGeom &g, int j, const uint8_t *__restrict__ raw,
                                        const float *__restrict__ plane, int x, int y) {
  if (MODE == 0) return (float)__ldg(raw + (long long)y * g.w + x);   // norm = 1
  if (MODE == 1)
    return __fmul_rn((float)__ldg(reinterpret_cast<const uint16_t *>(raw) + (long long)y * g.w + x),
                     g.norm);
  return __ldg(plane + (long long)y * g.pitch[j] + x);
}

// The terms need about 1e-7 relative, not IEEE exactness: quotients from
// the approximate reciprocal (MUFU) and one Newton step on the residual
// (Markstein, IBM J. Res. Dev. 34(1), 1990), faithful to about an ulp; the
// square root from the approximate MUFU root (relative error near 2^-22).
// Both in the .ftz form, which spares the subnormal handling: every
// reciprocal is of a sum holding C1, C2 or C3 (normal, with a normal
// reciprocal), and a subnormal v1 v2 under the root would give s1 s2 below
// 2^-63, which vanishes beside C2 and C3 in every term that uses it.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float sqrt_approx(float x) {
  float r;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// a / b given rb ~ 1 / b
__device__ __forceinline__ float div_by(float a, float b, float rb) {
  const float q = __fmul_rn(a, rb);
  return __fmaf_rn(__fmaf_rn(-q, b, a), rb, q);
}

__device__ __forceinline__ float div_fast(float a, float b) { return div_by(a, b, rcp_approx(b)); }

// a * b per half, one rounding each (mul.rn.f32x2): the same bits as two
// scalar __fmul_rn.  Its results here only feed fma multiplicands, which
// cannot absorb it (a pair product feeding a pair add is contracted into
// one fused operation despite .rn).
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

template <int MODE>
__global__ void __launch_bounds__(kLevelThreads, 6)
    k_msssim_level(MGeom g, int j, const uint8_t *__restrict__ ref, const uint8_t *__restrict__ dis,
                   float *__restrict__ pyr, double *__restrict__ part) {
  // the five quantities as three fp32 pairs (p, q), (p p, q q), (p q, 0):
  // PP holds (p, q) and (p q, 0) of a step's new input rows ((p p, q q) is
  // formed from (p, q) in the horizontal pass), HH the ring of horizontal
  // sums of all three (rows padded by one pair: the horizontal pass runs
  // row-fastest)
  __shared__ __align__(16) f2 PP[2][kCH][kIX + 1];
  __shared__ __align__(16) f2 HH[3][kRing][kTX + 1];
  __shared__ double wsum[kLevelThreads / 32][kQ];
  const int frame = blockIdx.z, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int W = g.ws[j], Hh = g.hs[j];
  const int ox0 = blockIdx.x * kTX, oy0 = blockIdx.y * kBH;
  const int ow = W - kWin + 1, oh = Hh - kWin + 1;
  const int nsteps = (min(kBH, oh - oy0) + kCH - 1) / kCH;
  const uint8_t *ra = ref + (long long)frame * g.frame_bytes + g.plane_off;
  const uint8_t *rb = dis + (long long)frame * g.frame_bytes + g.plane_off;
  const float *pa = pyr + (long long)(2 * frame) * g.img_floats + g.lvl_off[j];
  const float *pb = pa + g.img_floats;
  const float off = sample<MODE>(g, j, ra, pa, ox0, oy0);
  f2 gk[kWin];
#pragma unroll
  for (int k = 0; k < kWin; ++k) gk[k] = f2_pack(g.gauss[k], g.gauss[k]);

  // input rows row0 .. row0 + n - 1 of the band (clamped to the plane) into
  // PP rows 0 .. n - 1; thread t < 126 takes column t % 42 and rows t / 42,
  // + 3, + 6, ..., every load issued before the first is used
  constexpr int kRowStep = kLevelThreads / kIX;          // 3
  constexpr int kPer = (kCH + kRowStep - 1) / kRowStep;  // 6
  const int lc = t % kIX, lr0 = t / kIX;
  const bool loader = t < kRowStep * kIX;
  const int xc = min(ox0 + lc, W - 1);
  // the loads (issue) and the PP stores (commit) are separate so that a
  // step's loads are in flight during the previous step's vertical pass
  auto load_issue = [&](int row0, int n, float (&va)[kPer], float (&vb)[kPer]) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int r = lr0 + kRowStep * k;
      if (loader && r < n) {
        const int y = min(oy0 + row0 + r, Hh - 1);
        va[k] = sample<MODE>(g, j, ra, pa, xc, y);
        vb[k] = sample<MODE>(g, j, rb, pb, xc, y);
      }
    }
  };
  auto load_commit = [&](int n, const float (&va)[kPer], const float (&vb)[kPer]) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int r = lr0 + kRowStep * k;
      if (loader && r < n) {
        const float p = __fsub_rn(va[k], off);     // exact: both lie on the same grid below 256
        const float q = __fsub_rn(vb[k], off);
        PP[0][r][lc] = f2_pack(p, q);
        PP[1][r][lc] = f2_pack(__fmul_rn(p, q), 0.0f);
      }
    }
  };
  // horizontal sums of PP rows 0 .. n - 1 into ring rows (row0 + r) % 32: a
  // thread takes 4 adjacent positions of one row, rows fastest across threads
  auto hpass = [&](int row0, int n) {
    if (t < n * (kTX / 4)) {
      const int r = t % n, c0 = 4 * (t / n);
      const int hr = (row0 + r) & (kRing - 1);
      f2 v[kWin + 3];
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        // q = 0: (p, q) as loaded; q = 1: its squares; q = 2: (p q, 0)
#pragma unroll
        for (int k = 0; k < kWin + 3; ++k)
          v[k] = q == 0 ? PP[0][r][c0 + k] : (q == 1 ? f2_mul(v[k], v[k]) : PP[1][r][c0 + k]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          f2 acc = 0ull;                                 // (+0, +0)
#pragma unroll
          for (int k = 0; k < kWin; ++k) acc = f2_fma(gk[k], v[i + k], acc);
          HH[q][hr][c0 + i] = acc;
        }
      }
    }
  };
  // the block's share of the next scale whose source rows are PP rows 0 ..
  // n - 1 (p + off restores each sample exactly; clamping matches the
  // loads').  A block owns next-scale columns 16 bx .. and rows 256 by ..,
  // the last strip and band up to the plane's edge; row pairs never
  // straddle two steps (even band origin, step and halo).
  const bool next = j + 1 < kScales;
  const int Wn = next ? g.ws[j + 1] : 0, Hn = next ? g.hs[j + 1] : 0;
  const int X0 = blockIdx.x * (kTX / 2), Y0 = blockIdx.y * (kBH / 2);
  const int X1 = blockIdx.x + 1 == gridDim.x ? Wn : X0 + kTX / 2;
  const int Y1 = blockIdx.y + 1 == gridDim.y ? Hn : Y0 + kBH / 2;
  auto next_scale = [&](int row0, int n) {
    if (!next) return;
    const int ya = max(Y0, (oy0 + row0) / 2), yb = min(Y1, (oy0 + row0 + n) / 2);
    const int nx = X1 - X0, cnt = nx * (yb - ya);
    float *na = pyr + (long long)(2 * frame) * g.img_floats + g.lvl_off[j + 1];
    float *nb = na + g.img_floats;
    for (int i = t; i < cnt; i += kLevelThreads) {
      const int X = X0 + i % nx, Y = ya + i / nx;
      const int c0 = 2 * X - ox0, c1 = min(2 * X + 1, W - 1) - ox0;
      const int r0 = 2 * Y - oy0 - row0, r1 = min(2 * Y + 1, Hh - 1) - oy0 - row0;
      float a00, b00, a01, b01, a10, b10, a11, b11;
      f2_unpack(PP[0][r0][c0], a00, b00);
      f2_unpack(PP[0][r0][c1], a01, b01);
      f2_unpack(PP[0][r1][c0], a10, b10);
      f2_unpack(PP[0][r1][c1], a11, b11);
      const float a = __fadd_rn(__fadd_rn(__fadd_rn(a00, off), __fadd_rn(a01, off)),
                                __fadd_rn(__fadd_rn(a10, off), __fadd_rn(a11, off)));
      const float b = __fadd_rn(__fadd_rn(__fadd_rn(b00, off), __fadd_rn(b01, off)),
                                __fadd_rn(__fadd_rn(b10, off), __fadd_rn(b11, off)));
      na[(long long)Y * g.pitch[j + 1] + X] = __fmul_rn(a, 0.25f);
      nb[(long long)Y * g.pitch[j + 1] + X] = __fmul_rn(b, 0.25f);
    }
  };

  double dsum[kQ] = {0.0, 0.0, 0.0, 0.0, 0.0};        // lane 0: the warp's steps in order
  float va[kPer], vb[kPer];
  // the halo rows ahead of the first step
  load_issue(0, kHalo, va, vb);
  load_commit(kHalo, va, vb);
  __syncthreads();
  hpass(0, kHalo);
  next_scale(0, kHalo);
  load_issue(kHalo, kCH, va, vb);                       // the first step's rows
  __syncthreads();                                      // PP is free
  for (int st = 0; st < nsteps; ++st) {
    const int row0 = kHalo + st * kCH;                  // the step's new input rows
    load_commit(kCH, va, vb);
    __syncthreads();                                    // PP complete; the last vertical pass is done
    hpass(row0, kCH);
    next_scale(row0, kCH);
    __syncthreads();                                    // the ring is complete; PP is free
    if (st + 1 < nsteps) load_issue(row0 + kCH, kCH, va, vb);
    // vertical sums and the terms of four positions (output rows 4 w .. 4 w
    // + 3 of the step, w = thread / 32)
    const int oc = t % kTX, orow = st * kCH + 4 * (t / kTX);
    const int ox = ox0 + oc;
    f2 m[4][3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      f2 v[kWin + 3];
#pragma unroll
      for (int k = 0; k < kWin + 3; ++k) v[k] = HH[q][(orow + k) & (kRing - 1)][oc];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f2 acc = 0ull;
#pragma unroll
        for (int k = 0; k < kWin; ++k) acc = f2_fma(gk[k], v[i + k], acc);
        m[i][q] = acc;
      }
    }
    float sum[kQ] = {0, 0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int oy = oy0 + orow + i;
      if (ox < ow && oy < oh) {
        float m1, m2, e11, e22, e12, unused;
        f2_unpack(m[i][0], m1, m2);
        f2_unpack(m[i][1], e11, e22);
        f2_unpack(m[i][2], e12, unused);
        const float v1 = fmaxf(__fsub_rn(e11, __fmul_rn(m1, m1)), 0.0f);
        const float v2 = fmaxf(__fsub_rn(e22, __fmul_rn(m2, m2)), 0.0f);
        const float cv = __fsub_rn(e12, __fmul_rn(m1, m2));
        const float mu1 = __fadd_rn(m1, off), mu2 = __fadd_rn(m2, off);
        // s1 s2 = sqrt(v1 v2) (0 for a flat window); c and cs share 1 / vden
        const float sd12 = sqrt_approx(__fmul_rn(v1, v2));
        const float vden = __fadd_rn(__fadd_rn(v1, v2), g.C2);
        const float rv = rcp_approx(vden);
        const float l = div_fast(__fadd_rn(__fmul_rn(2.0f, __fmul_rn(mu1, mu2)), g.C1),
                                 __fadd_rn(__fadd_rn(__fmul_rn(mu1, mu1), __fmul_rn(mu2, mu2)), g.C1));
        const float c = div_by(__fadd_rn(__fmul_rn(2.0f, sd12), g.C2), vden, rv);
        const float s = div_fast(__fadd_rn(cv, g.C3), __fadd_rn(sd12, g.C3));
        const float cs = div_by(__fadd_rn(__fmul_rn(2.0f, cv), g.C2), vden, rv);
        sum[0] = __fadd_rn(sum[0], l);
        sum[1] = __fadd_rn(sum[1], c);
        sum[2] = __fadd_rn(sum[2], s);
        sum[3] = __fadd_rn(sum[3], cs);
        sum[4] = __fadd_rn(sum[4], __fmul_rn(l, cs));
      }
    }
    // the step's warp sums in fp32 (a fixed xor tree), added in fp64 by lane 0
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum[q] = __fadd_rn(sum[q], __shfl_xor_sync(0xffffffffu, sum[q], o));
      if (lane == 0) dsum[q] = __dadd_rn(dsum[q], (double)sum[q]);
    }
  }
  // the block's warp sums in fp64 in warp order
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < kQ; ++q) wsum[warp][q] = dsum[q];
  }
  __syncthreads();
  if (t < kQ) {
    double acc = 0.0;
#pragma unroll
    for (int w = 0; w < kLevelThreads / 32; ++w) acc = __dadd_rn(acc, wsum[w][t]);
    const long long tile = g.tile_off[j] + blockIdx.y * g.tx[j] + blockIdx.x;
    part[((long long)frame * g.tiles_total + tile) * kQ + t] = acc;
  }
}

// One block per frame, one warp per (scale, quantity): the span summed with
// lane l taking tiles l, l + 32, ... in order and a fixed xor tree; then the
// means and the score of one plane.  scores / values point at the plane's
// entry of frame 0; frames are nplanes entries apart.
__global__ void __launch_bounds__(kScales * kQ * 32)
    k_msssim_final(MGeom g, const double *__restrict__ part, double *__restrict__ scores,
                   double *__restrict__ values, int nplanes) {
  __shared__ double mean[kScales * kQ];
  const int frame = blockIdx.x, wq = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j = wq / kQ, q = wq % kQ;
  const int n = g.tx[j] * g.ty[j];
  const double *p = part + ((long long)frame * g.tiles_total + g.tile_off[j]) * kQ + q;
  double s = 0.0;
  for (int i = lane; i < n; i += 32) s = __dadd_rn(s, p[(long long)i * kQ]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  if (lane == 0) {
    const double cnt = (double)(g.ws[j] - kWin + 1) * (double)(g.hs[j] - kWin + 1);
    mean[wq] = s / cnt;
    values[(long long)frame * nplanes * kScales * kQ + wq] = s / cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double ms = 1.0;
    for (int k = 0; k + 1 < kScales; ++k) ms *= pow(mean[k * kQ + 3], g.beta[k]);
    ms *= pow(mean[(kScales - 1) * kQ + 4], g.beta[kScales - 1]);
    scores[(long long)frame * nplanes] = ms;
  }
}

}  // namespace

struct ss2_msssim {
  int nplanes;                             // 1 (luma) or 3 (luma, Cb, Cr)
  MGeom g[3];
  int batch, device;
  float *d_pyr[3] = {};                    // per plane: scales 2..5 of both images, per frame
  double *d_part[3] = {};                  // per plane: the (frame, scale, tile) spans
  double *d_scores = nullptr, *d_values = nullptr;   // frame-major, nplanes per frame
  double *h_scores = nullptr, *h_values = nullptr;
  size_t h_cap = 0;
  KernelTimer timer;                         // per-kernel event timing
};

static void msssim_free(ss2_msssim *c) {
  if (!c) return;
  for (int p = 0; p < 3; ++p) {
    cudaFree(c->d_pyr[p]);
    cudaFree(c->d_part[p]);
  }
  cudaFree(c->d_scores);
  cudaFree(c->d_values);
  if (c->h_scores) cudaFreeHost(c->h_scores);
  if (c->h_values) cudaFreeHost(c->h_values);
  delete c;
}

// Geometry of one plane (pw x ph samples at byte offset plane_off of each
// frame); -ENOTSUP when its scale-5 plane is below the 11x11 window.
static int make_mgeom(int pw, int ph, int bitdepth, long long frame_bytes, long long plane_off,
                      const char *name, MGeom &g) {
  std::memset(&g, 0, sizeof(g));
  g.w = pw; g.h = ph; g.depth = bitdepth; g.bps = bitdepth > 8 ? 2 : 1;
  g.frame_bytes = frame_bytes;
  g.plane_off = plane_off;
  g.norm = 1.0f / (float)(1 << (bitdepth - 8));
  int w = pw, h = ph;
  long long off = 0;
  for (int j = 0; j < kScales; ++j) {
    g.ws[j] = w;
    g.hs[j] = h;
    if (j > 0) {
      g.pitch[j] = (w + 31) & ~31;
      g.lvl_off[j] = off;
      off += (long long)g.pitch[j] * h;
    }
    w = (w + 1) / 2;
    h = (h + 1) / 2;
  }
  g.img_floats = (off + 63) & ~63LL;
  if (g.ws[kScales - 1] < kWin || g.hs[kScales - 1] < kWin)
    return fail(SS2_ENOTSUP, "MS-SSIM: the %s plane's scale-5 plane %dx%d is below the 11x11 window",
                name, g.ws[kScales - 1], g.hs[kScales - 1]);
  int tiles = 0;
  for (int j = 0; j < kScales; ++j) {
    g.tx[j] = (g.ws[j] - kWin + 1 + kTX - 1) / kTX;
    g.ty[j] = (g.hs[j] - kWin + 1 + kBH - 1) / kBH;
    g.tile_off[j] = tiles;
    tiles += g.tx[j] * g.ty[j];
  }
  g.tiles_total = tiles;
  const double L = 255.0;
  g.C1 = (float)((0.01 * L) * (0.01 * L));
  g.C2 = (float)((0.03 * L) * (0.03 * L));
  g.C3 = (float)((0.03 * L) * (0.03 * L) / 2.0);
  double gs[kWin], tot = 0.0;
  for (int i = 0; i < kWin; ++i) {
    const double t = i - kWin / 2;
    gs[i] = std::exp(-t * t / (2.0 * 1.5 * 1.5));
    tot += gs[i];
  }
  for (int i = 0; i < kWin; ++i) g.gauss[i] = (float)(gs[i] / tot);
  const double beta[kScales] = {0.0448, 0.2856, 0.3001, 0.2363, 0.1333};
  for (int j = 0; j < kScales; ++j) g.beta[j] = beta[j];
  return 0;
}

SS2_API ss2_msssim *ss2_msssim_create_ex(int width, int height, int bitdepth, int chroma,
                                         int max_batch, int enable_chroma) {
  if (check_geometry(width, height, bitdepth, chroma)) return nullptr;
  if (max_batch < 0 || max_batch > 4096) {
    fail(SS2_EINVAL, "batch %d is outside 0..4096", max_batch);
    return nullptr;
  }
  Geom full;
  make_geom(width, height, bitdepth, chroma, full);
  const int np = enable_chroma ? 3 : 1;
  MGeom g[3];
  const long long bps = full.bps, ysz = (long long)width * height,
                  csz = (long long)full.cw * full.ch;
  static const char *names[3] = {"luma", "Cb", "Cr"};
  for (int p = 0; p < np; ++p) {
    const int pw = p ? full.cw : width, ph = p ? full.ch : height;
    const long long off = p == 0 ? 0 : (ysz + (p - 1) * csz) * bps;
    if (make_mgeom(pw, ph, bitdepth, full.frame_bytes, off, names[p], g[p])) return nullptr;
  }
  int dev = 0;
  if (check_device(&dev)) return nullptr;
  ss2_msssim *c = new (std::nothrow) ss2_msssim();
  if (!c) {
    fail(SS2_ENOMEM, "host allocation failed");
    return nullptr;
  }
  c->nplanes = np;
  for (int p = 0; p < np; ++p) c->g[p] = g[p];
  c->device = dev;
  c->batch = max_batch ? max_batch : 32;
  const size_t B = (size_t)c->batch;
  bool ok = true;
  for (int p = 0; p < np && ok; ++p)
    ok = cudaMalloc(&c->d_pyr[p], B * 2 * g[p].img_floats * sizeof(float)) == cudaSuccess &&
         cudaMalloc(&c->d_part[p], B * g[p].tiles_total * kQ * sizeof(double)) == cudaSuccess;
  ok = ok && cudaMalloc(&c->d_scores, B * np * sizeof(double)) == cudaSuccess &&
       cudaMalloc(&c->d_values, B * np * kScales * kQ * sizeof(double)) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    fail(SS2_ENOMEM, "MS-SSIM workspace allocation failed");
    msssim_free(c);
    return nullptr;
  }
  return c;
}

SS2_API ss2_msssim *ss2_msssim_create(int width, int height, int bitdepth, int chroma,
                                      int max_batch) {
  return ss2_msssim_create_ex(width, height, bitdepth, chroma, max_batch, 0);
}

SS2_API int ss2_msssim_planes(const ss2_msssim *ctx) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  return ctx->nplanes;
}

SS2_API void ss2_msssim_destroy(ss2_msssim *ctx) { msssim_free(ctx); }

SS2_API int ss2_msssim_profile_begin(ss2_msssim *ctx) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  ctx->timer.begin();
  return 0;
}

SS2_API int ss2_msssim_profile_end(ss2_msssim *ctx, double *ms, int *launches) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  const cudaError_t e = ctx->timer.finish(2, ms, launches);
  return e == cudaSuccess ? 0 : cuda_fail(e, "MS-SSIM profile events");
}

// For each plane, the five scale launches and the final one, for nb frames
// (all enqueued; the caller waits once).
static cudaError_t msssim_batch(ss2_msssim *c, const uint8_t *ref, const uint8_t *dis, int nb,
                                cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  for (int p = 0; p < c->nplanes && e == cudaSuccess; ++p) {
    const MGeom &g = c->g[p];
    for (int j = 0; j < kScales && e == cudaSuccess; ++j) {
      e = c->timer.mark(0, true, st);
      if (e != cudaSuccess) break;
      const dim3 grid(g.tx[j], g.ty[j], nb);
      if (j > 0)
        k_msssim_level<2><<<grid, kLevelThreads, 0, st>>>(g, j, ref, dis, c->d_pyr[p], c->d_part[p]);
      else if (g.bps == 1)
        k_msssim_level<0><<<grid, kLevelThreads, 0, st>>>(g, j, ref, dis, c->d_pyr[p], c->d_part[p]);
      else
        k_msssim_level<1><<<grid, kLevelThreads, 0, st>>>(g, j, ref, dis, c->d_pyr[p], c->d_part[p]);
      e = cudaGetLastError();
      if (e == cudaSuccess) e = c->timer.mark(0, false, st);
    }
    if (e == cudaSuccess) e = c->timer.mark(1, true, st);
    if (e == cudaSuccess) {
      k_msssim_final<<<nb, kScales * kQ * 32, 0, st>>>(
          g, c->d_part[p], c->d_scores + p, c->d_values + (size_t)p * kScales * kQ, c->nplanes);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = c->timer.mark(1, false, st);
  }
  return e;
}

SS2_API int ss2_msssim_score(ss2_msssim *ctx, const void *ref, const void *dis, int n_frames,
                             double *scores, double *values, void *stream) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  if (n_frames < 0) return fail(SS2_EINVAL, "negative frame count %d", n_frames);
  if (n_frames == 0) return 0;
  if (!ref || !dis || !scores) return fail(SS2_EINVAL, "NULL pointer");
  if ((size_t)n_frames > ctx->h_cap) {
    if (ctx->h_scores) cudaFreeHost(ctx->h_scores);
    if (ctx->h_values) cudaFreeHost(ctx->h_values);
    ctx->h_scores = ctx->h_values = nullptr;
    ctx->h_cap = 0;
    if (cudaMallocHost(&ctx->h_scores, (size_t)n_frames * ctx->nplanes * sizeof(double)) !=
            cudaSuccess ||
        cudaMallocHost(&ctx->h_values,
                       (size_t)n_frames * ctx->nplanes * kScales * kQ * sizeof(double)) !=
            cudaSuccess) {
      cudaGetLastError();
      return fail(SS2_ENOMEM, "pinned allocation failed");
    }
    ctx->h_cap = (size_t)n_frames;
  }
  const long long fb = ctx->g[0].frame_bytes;
  const size_t np = (size_t)ctx->nplanes;
  cudaStream_t st = (cudaStream_t)stream;
  const uint8_t *r8 = (const uint8_t *)ref, *d8 = (const uint8_t *)dis;
  for (int f0 = 0; f0 < n_frames; f0 += ctx->batch) {
    const int nb = std::min(ctx->batch, n_frames - f0);
    cudaError_t e = msssim_batch(ctx, r8 + f0 * fb, d8 + f0 * fb, nb, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ctx->h_scores + f0 * np, ctx->d_scores, nb * np * sizeof(double),
                          cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && values)
      e = cudaMemcpyAsync(ctx->h_values + (size_t)f0 * np * kScales * kQ, ctx->d_values,
                          (size_t)nb * np * kScales * kQ * sizeof(double),
                          cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "MS-SSIM launch");
  }
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  std::memcpy(scores, ctx->h_scores, (size_t)n_frames * np * sizeof(double));
  if (values)
    std::memcpy(values, ctx->h_values, (size_t)n_frames * np * kScales * kQ * sizeof(double));
  return 0;
}

SS2_API int ss2_msssim_debug_pyramid_plane(ss2_msssim *ctx, const void *ref, const void *dis,
                                           int plane, float *planes, void *stream) {
  if (!ctx || !ref || !dis || !planes) return fail(SS2_EINVAL, "NULL argument");
  if (plane < 0 || plane >= ctx->nplanes)
    return fail(SS2_EINVAL, "plane %d is not scored by this context", plane);
  const MGeom &g = ctx->g[plane];
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = msssim_batch(ctx, (const uint8_t *)ref, (const uint8_t *)dis, 1, st);
  size_t off = 0;
  for (int img = 0; img < 2 && e == cudaSuccess; ++img)
    for (int j = 1; j < kScales && e == cudaSuccess; ++j) {
      e = cudaMemcpy2DAsync(planes + off, g.ws[j] * sizeof(float),
                            ctx->d_pyr[plane] + img * g.img_floats + g.lvl_off[j],
                            g.pitch[j] * sizeof(float), g.ws[j] * sizeof(float), g.hs[j],
                            cudaMemcpyDeviceToHost, st);
      off += (size_t)g.ws[j] * g.hs[j];
    }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "MS-SSIM pyramid");
  return 0;
}

SS2_API int ss2_msssim_debug_pyramid(ss2_msssim *ctx, const void *ref, const void *dis,
                                     float *planes, void *stream) {
  return ss2_msssim_debug_pyramid_plane(ctx, ref, dis, 0, planes, stream);
}
