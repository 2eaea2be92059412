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
//   k_fssim_decimate  one thread per decimated pixel of both images; the
//                     window sum is an int64 count of 2^-52 units: every
//                     nonzero tap (a float product sample * w, sample a
//                     multiple of 2^-8 below 256, w >= 2^-14) is a multiple
//                     of 2^-45 below 256, so the count stays below 2^61, is
//                     exact, and one conversion rounds it.
//   k_fssim_map       16x16 map tiles: separable 11-tap Gaussian sums of
//                     x1, x2, x1^2, x2^2, x1 x2 in fp32 on samples shifted by
//                     a per-tile offset (variances and covariance do not
//                     change, cancellation does), SSIM per pixel, one
//                     fixed-order fp64 block sum.
//   k_fssim_final     per frame: block sums in index order (fp64), mean.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/ss2.h"
#include "ss2_host.h"

#define SS2_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kWin = 11;                 // Gaussian window
constexpr int kTileO = 16;               // map outputs per tile edge
constexpr int kTileI = kTileO + kWin - 1;  // input tile edge (26)

struct FGeom {
  int w, h, depth, bps, scale, wd, hd, pitch;
  long long frame_bytes, plane;          // plane = pitch * hd floats
  int ow, oh, tiles_x, tiles_y;          // map outputs ("valid") and tiles
  float wt;                              // RN(1 / scale^2)
  float norm;                            // 2^(8 - depth): samples in the 8-bit range
  float C1, C2;
  float gauss[kWin];
};

__device__ __forceinline__ int mirror(int i, int n) {
  // symmetric extension with the edge sample repeated; any overshoot
#pragma unroll 1
  while (i < 0 || i >= n) {
    if (i < 0) i = -1 - i;
    if (i >= n) i = 2 * n - 1 - i;
  }
  return i;
}

template <int BPS>
__device__ __forceinline__ int luma_at(const uint8_t *__restrict__ f, int w, int x, int y) {
  const long long i = (long long)y * w + x;
  if (BPS == 1) return __ldg(f + i);
  return __ldg(reinterpret_cast<const uint16_t *>(f) + i);
}

template <int BPS>
__global__ void __launch_bounds__(256)
    k_fssim_decimate(FGeom g, const uint8_t *__restrict__ ref, const uint8_t *__restrict__ dis,
                     float *__restrict__ D) {
  const int x = blockIdx.x * 32 + threadIdx.x, y = blockIdx.y * 8 + threadIdx.y;
  const int frame = blockIdx.z;
  if (x >= g.wd || y >= g.hd) return;
  const uint8_t *fr[2] = {ref + frame * g.frame_bytes, dis + frame * g.frame_bytes};
  float *out = D + (long long)frame * 2 * g.plane + (long long)y * g.pitch + x;
  if (g.scale == 1) {
#pragma unroll
    for (int img = 0; img < 2; ++img)
      out[img * g.plane] = __fmul_rn((float)luma_at<BPS>(fr[img], g.w, x, y), g.norm);
    return;
  }
  const int lo = -(g.scale / 2), hi = g.scale - 1 - g.scale / 2;
  const int x0 = x * g.scale + lo, y0 = y * g.scale + lo;
  // windows wholly inside the frame need no mirroring (all but the edges)
  const bool inner = x0 >= 0 && y0 >= 0 && x * g.scale + hi < g.w && y * g.scale + hi < g.h;
  const float two52 = 4503599627370496.0f;  // 2^52
#pragma unroll
  for (int img = 0; img < 2; ++img) {
    long long acc = 0;
    if (inner) {
      const uint8_t *f = fr[img];
#pragma unroll 1
      for (int yy = y0; yy < y0 + g.scale; ++yy) {
#pragma unroll 4
        for (int xx = x0; xx < x0 + g.scale; ++xx) {
          const float smp = __fmul_rn((float)luma_at<BPS>(f, g.w, xx, yy), g.norm);  // exact
          acc += __float2ll_rn(__fmul_rn(__fmul_rn(smp, g.wt), two52));   // exact integer
        }
      }
    } else {
#pragma unroll 1
      for (int dy = lo; dy <= hi; ++dy) {
        const int yy = mirror(y * g.scale + dy, g.h);
#pragma unroll 1
        for (int dx = lo; dx <= hi; ++dx) {
          const int xx = mirror(x * g.scale + dx, g.w);
          const float smp = __fmul_rn((float)luma_at<BPS>(fr[img], g.w, xx, yy), g.norm);
          acc += __float2ll_rn(__fmul_rn(__fmul_rn(smp, g.wt), two52));
        }
      }
    }
    out[img * g.plane] = __fmul_rn(__ll2float_rn(acc), 1.0f / two52);   // exact scaling
  }
}

__global__ void __launch_bounds__(256)
    k_fssim_map(FGeom g, const float *__restrict__ D, double *__restrict__ part) {
  __shared__ float a[kTileI][kTileI + 1], b[kTileI][kTileI + 1];
  __shared__ float hs[5][kTileI][kTileO + 1];
  __shared__ double red[256];
  const int frame = blockIdx.z;
  const int ox0 = blockIdx.x * kTileO, oy0 = blockIdx.y * kTileO;
  const float *pa = D + (long long)frame * 2 * g.plane;
  const float *pb = pa + g.plane;
  const int t = threadIdx.x;
  // per-tile offset: the reference sample at the tile origin (same for both)
  const float off = pa[(long long)oy0 * g.pitch + ox0];
  for (int i = t; i < kTileI * kTileI; i += 256) {
    const int r = i / kTileI, c = i % kTileI;
    const int y = min(oy0 + r, g.hd - 1), x = min(ox0 + c, g.wd - 1);
    a[r][c] = __fsub_rn(pa[(long long)y * g.pitch + x], off);
    b[r][c] = __fsub_rn(pb[(long long)y * g.pitch + x], off);
  }
  __syncthreads();
  // horizontal Gaussian sums for every input row and output column
  for (int i = t; i < kTileI * kTileO; i += 256) {
    const int r = i / kTileO, c = i % kTileO;
    float s0 = 0, s1 = 0, s2 = 0, s3 = 0, s4 = 0;
#pragma unroll
    for (int k = 0; k < kWin; ++k) {
      const float p = a[r][c + k], q = b[r][c + k], w = g.gauss[k];
      s0 = __fmaf_rn(w, p, s0);
      s1 = __fmaf_rn(w, q, s1);
      s2 = __fmaf_rn(w, __fmul_rn(p, p), s2);
      s3 = __fmaf_rn(w, __fmul_rn(q, q), s3);
      s4 = __fmaf_rn(w, __fmul_rn(p, q), s4);
    }
    hs[0][r][c] = s0; hs[1][r][c] = s1; hs[2][r][c] = s2; hs[3][r][c] = s3; hs[4][r][c] = s4;
  }
  __syncthreads();
  // vertical sums and the SSIM term of one output pixel per thread
  const int oc = t % kTileO, orow = t / kTileO;
  const int ox = ox0 + oc, oy = oy0 + orow;
  float v = 0.0f;
  if (ox < g.ow && oy < g.oh) {
    float m[5] = {0, 0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < kWin; ++k)
#pragma unroll
      for (int q = 0; q < 5; ++q) m[q] = __fmaf_rn(g.gauss[k], hs[q][orow + k][oc], m[q]);
    const float m1 = m[0], m2 = m[1];
    const float v1 = __fsub_rn(m[2], __fmul_rn(m1, m1));
    const float v2 = __fsub_rn(m[3], __fmul_rn(m2, m2));
    const float cv = __fsub_rn(m[4], __fmul_rn(m1, m2));
    const float mu1 = __fadd_rn(m1, off), mu2 = __fadd_rn(m2, off);
    const float num = __fmul_rn(__fadd_rn(__fmul_rn(2.0f, __fmul_rn(mu1, mu2)), g.C1),
                                __fadd_rn(__fmul_rn(2.0f, cv), g.C2));
    const float den = __fmul_rn(
        __fadd_rn(__fadd_rn(__fmul_rn(mu1, mu1), __fmul_rn(mu2, mu2)), g.C1),
        __fadd_rn(__fadd_rn(v1, v2), g.C2));
    v = __fdiv_rn(num, den);
  }
  red[t] = (double)v;
  __syncthreads();
#pragma unroll
  for (int s = 128; s > 0; s >>= 1) {
    if (t < s) red[t] = __dadd_rn(red[t], red[t + s]);
    __syncthreads();
  }
  if (t == 0)
    part[(long long)frame * g.tiles_x * g.tiles_y + blockIdx.y * g.tiles_x + blockIdx.x] = red[0];
}

__global__ void k_fssim_final(FGeom g, const double *__restrict__ part, double *__restrict__ out) {
  const int frame = blockIdx.x;
  if (threadIdx.x != 0) return;
  const double *p = part + (long long)frame * g.tiles_x * g.tiles_y;
  double s = 0.0;
  for (int i = 0; i < g.tiles_x * g.tiles_y; ++i) s += p[i];
  out[frame] = s / ((double)g.ow * (double)g.oh);
}

}  // namespace

using namespace ss2;

struct ss2_fssim {
  FGeom g;
  int batch, device;
  float *d_dec = nullptr;      // 2 planes per frame
  double *d_part = nullptr, *d_scores = nullptr, *h_scores = nullptr;
  size_t h_cap = 0;
  // per-kernel event timing (ss2_fssim_profile_begin / _end)
  bool prof = false;
  std::vector<cudaEvent_t> ev_pool;
  std::vector<std::pair<int, int>> ev_used;   // (kernel class, index of start event)
};

static void fssim_free(ss2_fssim *c) {
  if (!c) return;
  for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
  cudaFree(c->d_dec);
  cudaFree(c->d_part);
  cudaFree(c->d_scores);
  if (c->h_scores) cudaFreeHost(c->h_scores);
  delete c;
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
  g.tiles_x = (g.ow + kTileO - 1) / kTileO;
  g.tiles_y = (g.oh + kTileO - 1) / kTileO;
  g.wt = 1.0f / (float)(g.scale * g.scale);
  g.norm = 1.0f / (float)(1 << (bitdepth - 8));
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
      cudaMalloc(&c->d_scores, B * sizeof(double)) != cudaSuccess) {
    cudaGetLastError();
    fail(SS2_ENOMEM, "float_ssim workspace allocation failed");
    fssim_free(c);
    return nullptr;
  }
  return c;
}

SS2_API void ss2_fssim_destroy(ss2_fssim *ctx) { fssim_free(ctx); }

SS2_API int ss2_fssim_scale(const ss2_fssim *ctx) { return ctx ? ctx->g.scale : 0; }

// Records the start (start = true) or end event of one launch of kernel
// class cls while profiling.
static cudaError_t fssim_mark(ss2_fssim *c, int cls, bool start, cudaStream_t st) {
  if (!c->prof) return cudaSuccess;
  size_t idx;
  if (start) {
    idx = c->ev_used.size() * 2;
    while (c->ev_pool.size() < idx + 2) {
      cudaEvent_t e;
      cudaError_t r = cudaEventCreate(&e);
      if (r != cudaSuccess) return r;
      c->ev_pool.push_back(e);
    }
    c->ev_used.push_back({cls, (int)idx});
  } else {
    idx = (size_t)c->ev_used.back().second + 1;
  }
  return cudaEventRecord(c->ev_pool[idx], st);
}

SS2_API int ss2_fssim_profile_begin(ss2_fssim *ctx) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  ctx->prof = true;
  ctx->ev_used.clear();
  return 0;
}

SS2_API int ss2_fssim_profile_end(ss2_fssim *ctx, double *ms, int *launches) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  double t[3] = {0, 0, 0};
  int n[3] = {0, 0, 0};
  for (const auto &u : ctx->ev_used) {
    cudaError_t e = cudaEventSynchronize(ctx->ev_pool[u.second + 1]);
    float dt = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&dt, ctx->ev_pool[u.second],
                                                   ctx->ev_pool[u.second + 1]);
    if (e != cudaSuccess) {
      ctx->prof = false;
      ctx->ev_used.clear();
      return cuda_fail(e, "float_ssim profile events");
    }
    t[u.first] += dt;
    n[u.first] += 1;
  }
  ctx->prof = false;
  ctx->ev_used.clear();
  for (int i = 0; i < 3; ++i) {
    if (ms) ms[i] = t[i];
    if (launches) launches[i] = n[i];
  }
  return 0;
}

static cudaError_t fssim_launch_decimate(const FGeom &g, const uint8_t *ref, const uint8_t *dis,
                                         float *D, int nb, cudaStream_t st) {
  dim3 grid((g.wd + 31) / 32, (g.hd + 7) / 8, nb), block(32, 8);
  if (g.bps == 1) k_fssim_decimate<1><<<grid, block, 0, st>>>(g, ref, dis, D);
  else k_fssim_decimate<2><<<grid, block, 0, st>>>(g, ref, dis, D);
  return cudaGetLastError();
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
    cudaError_t e = fssim_mark(ctx, 0, true, st);
    if (e == cudaSuccess)
      e = fssim_launch_decimate(g, r8 + f0 * g.frame_bytes, d8 + f0 * g.frame_bytes, ctx->d_dec,
                                nb, st);
    if (e == cudaSuccess) e = fssim_mark(ctx, 0, false, st);
    if (e == cudaSuccess) e = fssim_mark(ctx, 1, true, st);
    if (e == cudaSuccess) {
      k_fssim_map<<<dim3(g.tiles_x, g.tiles_y, nb), 256, 0, st>>>(g, ctx->d_dec, ctx->d_part);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = fssim_mark(ctx, 1, false, st);
    if (e == cudaSuccess) e = fssim_mark(ctx, 2, true, st);
    if (e == cudaSuccess) {
      k_fssim_final<<<nb, 32, 0, st>>>(g, ctx->d_part, ctx->d_scores);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = fssim_mark(ctx, 2, false, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ctx->h_scores + f0, ctx->d_scores, nb * sizeof(double),
                          cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "float_ssim launch");
  }
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  std::memcpy(scores, ctx->h_scores, (size_t)n_frames * sizeof(double));
  return 0;
}

SS2_API int ss2_fssim_debug_decimated(ss2_fssim *ctx, const void *ref, const void *dis,
                                      float *planes, void *stream) {
  if (!ctx || !ref || !dis || !planes) return fail(SS2_EINVAL, "NULL argument");
  const FGeom &g = ctx->g;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = fssim_launch_decimate(g, (const uint8_t *)ref, (const uint8_t *)dis,
                                        ctx->d_dec, 1, st);
  for (int p = 0; p < 2 && e == cudaSuccess; ++p)
    e = cudaMemcpy2DAsync(planes + (size_t)p * g.wd * g.hd, g.wd * sizeof(float),
                          ctx->d_dec + p * g.plane, g.pitch * sizeof(float), g.wd * sizeof(float),
                          g.hd, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "float_ssim decimation");
  return 0;
}
