// api.cu — the C ABI of libss2 (include/ss2.h): argument checks, the
// context and its device workspace, the constant tables the kernels read,
// and the order of launches for a batch of frames.
//
// Control crosses to the device once per batch of frames (the launches) and
// back once per call (the 8-byte-per-frame score read-back and one stream
// synchronisation), as "Research-1363: Device-resident ssimulacra2 and a
// single-wait MS-SSIM on SYCL" asks in its Question and Finding 6.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cerrno>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "../../include/ss2.h"
#include "ss2_host.h"
#include "ss2_impl.h"
#include "ss2_kernels.h"
#include "ss2_tma.cuh"

#define SS2_API extern "C" __attribute__((visibility("default")))

using namespace ss2;

// ---------------------------------------------------------------------------
// Errors
// ---------------------------------------------------------------------------

static thread_local int t_err = 0;
static thread_local char t_msg[512] = "";

int ss2::fail(int code, const char *fmt, ...) {
  t_err = code;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return code;
}

int ss2::cuda_fail(cudaError_t e, const char *what) {
  return fail(SS2_EIO, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define CU(call, what)                     \
  do {                                     \
    cudaError_t e_ = (call);               \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

SS2_API int ss2_last_error(void) { return t_err; }
SS2_API const char *ss2_last_error_string(void) { return t_msg; }

// ---------------------------------------------------------------------------
// Host-built constant tables (the library's own; nothing is shared with any
// other implementation).
// ---------------------------------------------------------------------------

// sRGB decoding (IEC 61966-2-1) in fp64.
static double srgb_to_linear(double v);

// (T[i], T[i+1] - T[i]) for i < N, then (T[N], 0): the interpolation at
// t = N with index N gives T[N] + 0 * 0 = T[N], which is what index N - 1
// with weight 1 gives (T[N] - T[N-1] is exact, both lying in [1/2, 1]).
void ss2::build_eotf_pairs(float *P) {
  float T[kEotfN + 1];
  build_eotf(T);
  for (int i = 0; i < kEotfN; ++i) {
    P[2 * i] = T[i];
    P[2 * i + 1] = T[i + 1] - T[i];
  }
  P[2 * kEotfN] = T[kEotfN];
  P[2 * kEotfN + 1] = 0.0f;
}

// 8-bit samples read their normalisations from tables (256 entries each);
// deeper ones divide without a table on the device.
int ss2::norm_entries(int depth) { return depth == 8 ? 256 : 0; }

// (v - 16k) / 219k and (v - 128k) / 224k, k = 2^(depth-8), as float
// quotients of exactly representable operands (correctly rounded).
void ss2::build_norm(int depth, float *yn, float *cn) {
  const int k = 1 << (depth - 8), n = norm_entries(depth);
  const float dy = (float)(219 * k), dc = (float)(224 * k);
  for (int v = 0; v < n; ++v) {
    yn[v] = (float)(v - 16 * k) / dy;
    cn[v] = (float)(v - 128 * k) / dc;
  }
}

static double srgb_to_linear(double v) {
  return v <= 0.04045 ? v / 12.92 : std::pow((v + 0.055) / 1.055, 2.4);
}

void ss2::build_eotf(float *T) {
  for (int i = 0; i <= kEotfN; ++i) T[i] = (float)srgb_to_linear((double)i / kEotfN);
}

// Recursive Gaussian (sigma = 1.5) as three odd cosine harmonics on |m| <= R:
// h[m] = sum_k a_k cos(w_k m), w_k = (2k+1) pi / (2 (R+1)).  The a_k solve
// the least-squares fit to the sampled Gaussian density under sum_m h[m] = 1
// (Lagrange system, Gauss-Jordan with partial pivoting).  The resonator of
// harmonic k runs Y[n+1] = 2 cos(w_k) Y[n] - Y[n-1] + a_k cos(w_k R)
// (x[n+R+1] + x[n-R-1]).
static void build_iir(float *c2, float *gk) {
  const double kPi = 3.14159265358979323846, sigma = 1.5;
  const int R = kIirR;
  double w[3];
  for (int k = 0; k < 3; ++k) w[k] = (2 * k + 1) * kPi / (2.0 * (R + 1));
  double A[4][5] = {};
  for (int m = -R; m <= R; ++m) {
    const double gm = std::exp(-(double)m * m / (2.0 * sigma * sigma)) / (sigma * std::sqrt(2.0 * kPi));
    double cs[3];
    for (int k = 0; k < 3; ++k) cs[k] = std::cos(w[k] * m);
    for (int r = 0; r < 3; ++r) {
      for (int k = 0; k < 3; ++k) A[r][k] += cs[r] * cs[k];
      A[r][3] += cs[r];
      A[r][4] += cs[r] * gm;
    }
  }
  for (int k = 0; k < 3; ++k) A[3][k] = A[k][3];
  A[3][4] = 1.0;
  for (int col = 0; col < 4; ++col) {
    int best = col;
    for (int r = col + 1; r < 4; ++r)
      if (std::fabs(A[r][col]) > std::fabs(A[best][col])) best = r;
    for (int j = 0; j < 5; ++j) std::swap(A[col][j], A[best][j]);
    for (int r = col + 1; r < 4; ++r) {
      const double f = A[r][col] / A[col][col];
      for (int j = col; j < 5; ++j) A[r][j] -= f * A[col][j];
    }
  }
  double a[4];
  for (int r = 3; r >= 0; --r) {
    double acc = A[r][4];
    for (int j = r + 1; j < 4; ++j) acc -= A[r][j] * a[j];
    a[r] = acc / A[r][r];
  }
  for (int k = 0; k < 3; ++k) {
    c2[k] = (float)(2.0 * std::cos(w[k]));
    gk[k] = (float)(a[k] * std::cos(w[k] * R));
  }
}

// BT.709 (Kr = 0.2126, Kb = 0.0722) limited-range decoding coefficients.
static void build_yuv(float *k) {
  const double kr = 0.2126, kb = 0.0722, kg = 1.0 - kr - kb;
  k[0] = (float)(2.0 * (1.0 - kr));           // Cr -> R'
  k[1] = (float)(2.0 * kb * (1.0 - kb) / kg); // Cb -> G' (subtracted)
  k[2] = (float)(2.0 * kr * (1.0 - kr) / kg); // Cr -> G' (subtracted)
  k[3] = (float)(2.0 * (1.0 - kb));           // Cb -> B'
}

void ss2::default_params(double *p) {
  std::memset(p, 0, sizeof(double) * kNParams);
  for (int i = 0; i < kNValues; ++i) p[kPWeights + i] = 1.0 / 108.0;  // placeholder
  p[kPPoly + 0] = 100.0;   // placeholder map: score = 100 - 100 P
  p[kPPoly + 1] = -100.0;
  p[kPPower + 0] = 1.0;
  p[kPPower + 1] = 1.0;
  // XYB opsin mixing (JPEG XL, ISO/IEC 18181-1)
  const double m[9] = {0.30, 0.622, 0.078, 0.23, 0.692, 0.078,
                       0.24342268924547819, 0.20476744424496821, 0.55180986650955360};
  for (int i = 0; i < 9; ++i) p[kPOpsin + i] = m[i];
  for (int i = 0; i < 3; ++i) p[kPBias + i] = 0.0037930732552754493;
  p[kPAffine + 0] = 1.0;  // identity make-positive affine (placeholder)
  p[kPAffine + 3] = 1.0;
  p[kPC2] = 0.0009;
}

// ---------------------------------------------------------------------------
// Context
// ---------------------------------------------------------------------------

// A lane is one pass of the pipeline in flight: a workspace for `batch`
// frames and an internal stream.  Batches alternate between the two lanes,
// so the memory-bound pass of one batch can run beside the arithmetic-bound
// passes of the other.
constexpr int kLanes = 2;

struct Lane {
  float *X = nullptr, *H = nullptr;
  float2 *part = nullptr;
  double *values = nullptr, *scores = nullptr;
  PlaneMaps maps;
  cudaStream_t st = nullptr;
  cudaEvent_t ev_done = nullptr;
  // host-input path (allocated on first use): ref then dis frames of a batch
  uint8_t *in = nullptr;
  cudaEvent_t ev_copied = nullptr, ev_consumed = nullptr;
};

// The launch sequence of one device-input call, captured as a CUDA graph and
// replayed by one launch while later calls repeat it: the same frame
// pointers, count and outputs (the read-back destinations are baked in) and
// the same timing state.  With per-kernel timing on, each launch is
// bracketed by external event-record nodes whose times are read after the
// call's stream synchronisation.
struct CallKey {
  const void *ref = nullptr, *dis = nullptr;
  int n = 0;
  bool values = false, timed = false;
  const double *h_scores = nullptr, *h_values = nullptr;
  bool operator==(const CallKey &o) const {
    return ref == o.ref && dis == o.dis && n == o.n && values == o.values &&
           timed == o.timed && h_scores == o.h_scores && h_values == o.h_values;
  }
};

struct CallGraph {
  cudaGraphExec_t exec = nullptr;
  CallKey key;
  std::vector<cudaEvent_t> ev;  // start, end of each timed launch
  std::vector<int> cls;         // its kernel class
  void reset() {
    if (exec) cudaGraphExecDestroy(exec);
    exec = nullptr;
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
    cls.clear();
  }
};

struct ss2_ctx {
  Geom g;
  Pix px;
  int batch;
  int device;
  double params[kNParams];
  Lane lane[kLanes];
  double *d_params = nullptr;
  float *d_tabs = nullptr;         // EOTF pairs, then the two normalisation tables
  PyrTabs tabs;
  int *d_err = nullptr;            // error bits raised by kernels (bounded waits)
  cudaEvent_t ev_fork = nullptr;
  size_t ws_bytes = 0;
  // pinned read-back staging
  double *h_scores = nullptr;
  double *h_values = nullptr;
  int *h_err = nullptr;
  size_t h_cap = 0;  // frames
  KernelTimer timer;  // per-kernel event timing (ss2_profile_begin / ss2_profile_end)
  cudaStream_t copy_stream = nullptr;   // host-input path uploads
  // device-input calls as CUDA graphs (ss2_set_graphs, off by default): a
  // context's first call runs eagerly (one-time kernel attributes are set
  // outside any capture)
  CallGraph graph;
  cudaStream_t cap_stream = nullptr;    // capture happens here, never on the caller's stream
  bool graphs = false, warm = false, capturing = false;
};

static int chroma_shift(int chroma, int *sx, int *sy) {
  switch (chroma) {
    case SS2_CHROMA_420: *sx = 1; *sy = 1; return 0;
    case SS2_CHROMA_422: *sx = 1; *sy = 0; return 0;
    case SS2_CHROMA_444: *sx = 0; *sy = 0; return 0;
    default: return -1;
  }
}

int ss2::check_geometry(int w, int h, int depth, int chroma) {
  int sx = 0, sy = 0;
  if (w < 8 || h < 8) return fail(SS2_EINVAL, "frame %dx%d is below the 8x8 minimum", w, h);
  if (w > SS2_MAX_DIM || h > SS2_MAX_DIM)
    return fail(SS2_EINVAL, "frame %dx%d is above the %d limit", w, h, SS2_MAX_DIM);
  if (depth < 8 || depth > 16) return fail(SS2_EINVAL, "bit depth %d is outside 8..16", depth);
  if (chroma_shift(chroma, &sx, &sy))
    return fail(SS2_EINVAL, "chroma %d is not one of 420, 422, 444", chroma);
  if (sx && (w & 1)) return fail(SS2_EINVAL, "odd width %d with subsampled chroma %d", w, chroma);
  return 0;
}

void ss2::make_geom(int w, int h, int depth, int chroma, Geom &g) {
  std::memset(&g, 0, sizeof(g));
  g.w = w; g.h = h; g.depth = depth; g.chroma = chroma;
  chroma_shift(chroma, &g.sx, &g.sy);
  g.cw = (w + g.sx) >> g.sx;
  g.ch = (h + g.sy) >> g.sy;
  g.bps = depth > 8 ? 2 : 1;
  g.frame_bytes = ((long long)w * h + 2LL * g.cw * g.ch) * g.bps;
  int sw = w, sh = h, n = 0;
  while (n < kMaxScales && sw >= 8 && sh >= 8) {
    g.ws[n] = sw; g.hs[n] = sh;
    g.pitch[n] = (sw + 31) & ~31;
    g.nw[n] = (sw + 31) / 32;
    g.plane[n] = (long long)g.pitch[n] * sh;
    ++n;
    sw = (sw + 1) / 2; sh = (sh + 1) / 2;
  }
  g.nscales = n;
  long long xo = 0, ho = 0;
  int po = 0;
  g.hunit_off[0] = 0;
  g.vwarp_off[0] = 0;
  for (int s = 0; s < n; ++s) {
    g.xoff[s] = xo; xo += 6 * g.plane[s];
    g.hoff[s] = ho; ho += (long long)3 * kNq * g.plane[s];
    g.poff[s] = po; po += 3 * kNSum * g.nw[s];
    g.hunit_off[s + 1] = g.hunit_off[s] + 3 * ((g.hs[s] + kBoxRows - 1) / kBoxRows);
    g.vwarp_off[s + 1] = g.vwarp_off[s] + 3 * g.nw[s];
  }
  for (int s = n; s < kMaxScales; ++s) {
    g.hunit_off[s + 1] = g.hunit_off[s];
    g.vwarp_off[s + 1] = g.vwarp_off[s];
  }
  g.x_fs = xo; g.h_fs = ho; g.p_fs = po;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// One tiled map over fp32 data of the given rank: dims[0] is the innermost
// extent, strides[i] the byte stride of dims[i + 1]; zero fill outside the
// tensor.
static int encode_tiled(CUtensorMap *m, float *base, int rank, const cuuint64_t *dims,
                        const cuuint64_t *strides, const cuuint32_t *box,
                        CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return fail(SS2_EIO, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, base, dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SS2_EIO, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return 0;
}

// (column, row, plane, frame) over a stack of planes, boxes of bc x br x bp.
static int encode_stack(CUtensorMap *m, float *base, int ws, int hs, int nplanes, int batch,
                        long long pitch, long long plane, long long frame_stride, int bc, int br,
                        int bp, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  const cuuint64_t dims[4] = {(cuuint64_t)ws, (cuuint64_t)hs, (cuuint64_t)nplanes,
                              (cuuint64_t)batch};
  const cuuint64_t strides[3] = {(cuuint64_t)pitch * 4, (cuuint64_t)plane * 4,
                                 (cuuint64_t)frame_stride * 4};
  const cuuint32_t box[4] = {(cuuint32_t)bc, (cuuint32_t)br, (cuuint32_t)bp, 1};
  return encode_tiled(m, base, 4, dims, strides, box, swizzle);
}

// (float of the quad row, row, channel, frame) over the interleaved quads of
// mu1, mu2, s11, s22 (a quad row is 4 x pitch floats, a channel 4 x plane):
// boxes of bf floats x br rows.
static int encode_quads(CUtensorMap *m, float *base, int ws, int hs, int batch, long long pitch,
                        long long plane, long long frame_stride, int bf, int br,
                        CUtensorMapSwizzle swizzle) {
  const cuuint64_t dims[4] = {4 * (cuuint64_t)ws, (cuuint64_t)hs, 3, (cuuint64_t)batch};
  const cuuint64_t strides[3] = {(cuuint64_t)pitch * 16, (cuuint64_t)plane * 16,
                                 (cuuint64_t)frame_stride * 4};
  const cuuint32_t box[4] = {(cuuint32_t)bf, (cuuint32_t)br, 1, 1};
  return encode_tiled(m, base, 4, dims, strides, box, swizzle);
}

int ss2::encode_maps(const Geom &g, float *X, float *H, int batch, PlaneMaps &m) {
  std::memset(&m, 0, sizeof(m));
  for (int s = 0; s < g.nscales; ++s) {
    float *xb = X + g.xoff[s], *hb = H + g.hoff[s], *sb = hb + 12 * g.plane[s];
    const int ws = g.ws[s], hs = g.hs[s];
    const long long pitch = g.pitch[s], plane = g.plane[s];
    // the horizontal pass's lanes own one row each: its boxes are swizzled
    // by their row width (8 floats = 32 bytes for XYB and s12, 8 quads =
    // 128 bytes for the quads) so that those lanes read and write 16-byte
    // units without bank conflicts; the vertical pass loads rows of 32
    // quads, unswizzled (its lanes read consecutive 16-byte units)
    if (encode_stack(&m.h.x[s], xb, ws, hs, 6, batch, pitch, plane, g.x_fs, kBoxCols, kBoxRows,
                     1, CU_TENSOR_MAP_SWIZZLE_32B) ||
        encode_quads(&m.h.q4[s], hb, ws, hs, batch, pitch, plane, g.h_fs, 4 * kBoxCols,
                     kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        encode_stack(&m.h.s1[s], sb, ws, hs, 3, batch, pitch, plane, g.h_fs, kBoxCols, kBoxRows,
                     1, CU_TENSOR_MAP_SWIZZLE_32B) ||
        encode_quads(&m.v.vq4[s], hb, ws, hs, batch, pitch, plane, g.h_fs, 4 * kVCols, kVRows,
                     CU_TENSOR_MAP_SWIZZLE_NONE) ||
        encode_stack(&m.v.vs1[s], sb, ws, hs, 3, batch, pitch, plane, g.h_fs, kVCols, kVRows, 1))
      return t_err;
  }
  return 0;
}

size_t ss2::per_frame_bytes(const Geom &g) {
  return (size_t)(g.x_fs + g.h_fs) * sizeof(float) + (size_t)g.p_fs * sizeof(float2) +
         (kNValues + 1) * sizeof(double);
}

// Frames per pass: enough column walkers at scale 0 to fill the GPU (about
// 160k threads, 3 per column), within 16 GB per lane workspace.
// About 60 M pixels per pass (7 frames at 3840x2160, 29 at 1920x1080): the
// best measured throughput at both sizes.  2 to 64 frames, and at most 16 GB
// of workspace per lane.
static int default_batch(const Geom &g) {
  const long long px = (long long)g.w * g.h;
  long long b = (60000000LL + px / 2) / px;
  b = std::max(2LL, std::min(64LL, b));
  const long long cap = (16LL << 30) / (long long)per_frame_bytes(g);
  b = std::max(1LL, std::min(b, cap));
  return (int)b;
}

// A positive finite float as X 2^e, X an integer below 2^24.
static void split_float(float v, uint64_t &X, int &e) {
  uint32_t b;
  std::memcpy(&b, &v, sizeof(b));
  const uint32_t be = (b >> 23) & 0xffu, m = b & 0x7fffffu;
  X = be ? (m | 0x800000u) : m;
  e = be ? (int)be - 150 : -149;
}

// Sign of (M 2^f)^3 - X 2^g, exact in 128-bit integers (M < 2^26, X < 2^24).
static int cube_vs(uint64_t M, int f, uint64_t X, int g) {
  const unsigned __int128 c = (unsigned __int128)(M * M) * M;  // below 2^78
  const int d = 3 * f - g;
  if (d >= 0) {
    if (d >= 24) return 1;  // c >= 1 and X < 2^24
    const unsigned __int128 l = c << d;
    return l > X ? 1 : (l < X ? -1 : 0);
  }
  if (-d >= 104) return -1;  // X >= 1: X 2^-d >= 2^104 > c
  const unsigned __int128 r = (unsigned __int128)X << (-d);
  return c > r ? 1 : (c < r ? -1 : 0);
}

// Correctly rounded cube root of a finite float on the host (for the three
// cbrt(bias_i) the XYB conversion subtracts): the double cube root rounded
// to float is an ulp or so off at most, and the exact comparisons of x with
// the cubes of the midpoints to the neighbouring floats move it to the
// nearest one (below a power of two the lower neighbour is half as far).
static float cbrt_rn_host(float x) {
  if (x == 0.0f || !std::isfinite(x)) return x;
  if (x < 0.0f) return -cbrt_rn_host(-x);
  uint64_t X;
  int g;
  split_float(x, X, g);
  float y = (float)std::cbrt((double)x);
  for (int it = 0; it < 8; ++it) {
    uint64_t Y;
    int e;
    split_float(y, Y, e);
    if (cube_vs(2 * Y + 1, e - 1, X, g) < 0) {  // x beyond the upper midpoint's cube
      y = std::nextafter(y, HUGE_VALF);
      continue;
    }
    const bool at_floor = Y == 0x800000u && e > -149;
    if (cube_vs(at_floor ? 4 * Y - 1 : 2 * Y - 1, at_floor ? e - 2 : e - 1, X, g) > 0) {
      y = std::nextafter(y, 0.0f);  // x below the lower midpoint's cube
      continue;
    }
    break;
  }
  return y;
}

void ss2::build_pix(const double *params, Pix &p) {
  build_yuv(p.yuv);
  for (int i = 0; i < 9; ++i) p.opsin[i] = (float)params[kPOpsin + i];
  for (int i = 0; i < 3; ++i) p.bias[i] = (float)params[kPBias + i];
  for (int i = 0; i < 3; ++i) p.cbias[i] = cbrt_rn_host(p.bias[i]);
  p.sx = (float)params[kPAffine + 0];
  p.ox = (float)params[kPAffine + 1];
  p.oy = (float)params[kPAffine + 2];
  p.sb = (float)params[kPAffine + 3];
  p.ob = (float)params[kPAffine + 4];
  p.c2 = (float)params[kPC2];
  build_iir(p.iir_c2, p.iir_g);
}

static void set_pix(ss2_ctx *c) { build_pix(c->params, c->px); }

static void free_ctx(ss2_ctx *c) {
  if (!c) return;
  for (Lane &L : c->lane) {
    cudaFree(L.X); cudaFree(L.H); cudaFree(L.part); cudaFree(L.values); cudaFree(L.scores);
    cudaFree(L.in);
    if (L.st) cudaStreamDestroy(L.st);
    if (L.ev_done) cudaEventDestroy(L.ev_done);
    if (L.ev_copied) cudaEventDestroy(L.ev_copied);
    if (L.ev_consumed) cudaEventDestroy(L.ev_consumed);
  }
  cudaFree(c->d_params); cudaFree(c->d_tabs); cudaFree(c->d_err);
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  if (c->h_err) cudaFreeHost(c->h_err);
  if (c->h_scores) cudaFreeHost(c->h_scores);
  if (c->h_values) cudaFreeHost(c->h_values);
  if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
  c->graph.reset();
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  delete c;
}

int ss2::check_device(int *dev) {
  int n = 0;
  cudaError_t e = cudaGetDeviceCount(&n);
  if (e != cudaSuccess || n == 0) {
    cudaGetLastError();
    return fail(SS2_ENOTSUP, "no CUDA device (%s)", cudaGetErrorString(e));
  }
  CU(cudaGetDevice(dev), "cudaGetDevice");
  cudaDeviceProp prop;
  CU(cudaGetDeviceProperties(&prop, *dev), "cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3)
    return fail(SS2_ENOTSUP, "device %s is sm_%d%d; libss2 is built for sm_103a", prop.name,
                prop.major, prop.minor);
  return 0;
}

// Host-side fault injection for the failure-path tests: SS2_FAULT holds a
// comma-separated list of "alloc", "launch", "memcpy"; the named step then
// fails before it touches the device.
static bool injected(const char *kind) {
  const char *f = std::getenv("SS2_FAULT");
  if (!f || !*f) return false;
  const size_t n = std::strlen(kind);
  for (const char *p = f; (p = std::strstr(p, kind)) != nullptr; p += n) {
    const bool starts = p == f || p[-1] == ',';
    const bool ends = p[n] == '\0' || p[n] == ',';
    if (starts && ends) return true;
  }
  return false;
}

static int dev_alloc(void **p, size_t bytes, size_t *total) {
  if (injected("alloc")) {
    *p = nullptr;
    return fail(SS2_ENOMEM, "cudaMalloc of %zu bytes failed (injected by SS2_FAULT=alloc)",
                bytes);
  }
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return fail(SS2_ENOMEM, "cudaMalloc of %zu bytes failed (%s)", bytes, cudaGetErrorString(e));
  }
  *total += bytes;
  return 0;
}

static int ensure_host_cap(ss2_ctx *c, size_t frames) {
  if (frames <= c->h_cap) return 0;
  if (c->h_scores) cudaFreeHost(c->h_scores);
  if (c->h_values) cudaFreeHost(c->h_values);
  c->h_scores = nullptr;
  c->h_values = nullptr;
  c->h_cap = 0;
  size_t cap = std::max(frames, (size_t)c->batch);
  if (cudaMallocHost((void **)&c->h_scores, cap * sizeof(double)) != cudaSuccess ||
      cudaMallocHost((void **)&c->h_values, cap * kNValues * sizeof(double)) != cudaSuccess) {
    cudaGetLastError();
    return fail(SS2_ENOMEM, "pinned allocation for %zu frames failed", cap);
  }
  c->h_cap = cap;
  return 0;
}

static ss2_ctx *create(int w, int h, int depth, int chroma, int batch) {
  if (check_geometry(w, h, depth, chroma)) return nullptr;
  if (batch != 0 && (batch < 1 || batch > 1024)) {
    fail(SS2_EINVAL, "batch %d is outside 1..1024", batch);
    return nullptr;
  }
  int dev = 0;
  if (check_device(&dev)) return nullptr;
  ss2_ctx *c = new (std::nothrow) ss2_ctx();
  if (!c) {
    fail(SS2_ENOMEM, "host allocation failed");
    return nullptr;
  }
  c->device = dev;
  make_geom(w, h, depth, chroma, c->g);
  c->batch = batch ? batch : default_batch(c->g);
  default_params(c->params);
  set_pix(c);
  const Geom &g = c->g;
  const size_t B = (size_t)c->batch;
  size_t tot = 0;
  for (Lane &L : c->lane) {
    if (dev_alloc((void **)&L.X, B * g.x_fs * sizeof(float), &tot) ||
        dev_alloc((void **)&L.H, B * g.h_fs * sizeof(float), &tot) ||
        dev_alloc((void **)&L.part, B * g.p_fs * sizeof(float2), &tot) ||
        dev_alloc((void **)&L.values, B * kNValues * sizeof(double), &tot) ||
        dev_alloc((void **)&L.scores, B * sizeof(double), &tot) ||
        encode_maps(g, L.X, L.H, c->batch, L.maps)) {
      free_ctx(c);
      return nullptr;
    }
    cudaError_t e = cudaStreamCreateWithFlags(&L.st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&L.ev_done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      cuda_fail(e, "lane stream");
      free_ctx(c);
      return nullptr;
    }
  }
  if (cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming) != cudaSuccess) {
    cuda_fail(cudaGetLastError(), "fork event");
    free_ctx(c);
    return nullptr;
  }
  if (dev_alloc((void **)&c->d_params, kNParams * sizeof(double), &tot) ||
      dev_alloc((void **)&c->d_tabs,
                (2 * kEotfPairs + 2 * norm_entries(depth)) * sizeof(float), &tot) ||
      dev_alloc((void **)&c->d_err, sizeof(int), &tot)) {
    free_ctx(c);
    return nullptr;
  }
  c->ws_bytes = tot;
  const int nn = norm_entries(depth);
  std::vector<float> tab((size_t)2 * kEotfPairs + 2 * (size_t)nn);
  build_eotf_pairs(tab.data());
  build_norm(depth, tab.data() + 2 * kEotfPairs, tab.data() + 2 * kEotfPairs + nn);
  c->tabs.eotf = reinterpret_cast<const float2 *>(c->d_tabs);
  c->tabs.ynorm = nn ? c->d_tabs + 2 * kEotfPairs : nullptr;
  c->tabs.cnorm = nn ? c->d_tabs + 2 * kEotfPairs + nn : nullptr;
  c->tabs.rdy = 1.0f / (float)(219 << (depth - 8));
  c->tabs.rdc = 1.0f / (float)(224 << (depth - 8));
  cudaError_t e = cudaMemcpy(c->d_tabs, tab.data(), tab.size() * sizeof(float),
                             cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(c->d_params, c->params, sizeof(c->params), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(c->d_err, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaMallocHost((void **)&c->h_err, sizeof(int));
  // The copies and the memset are ordered on the legacy default stream only
  // (a copy from pageable memory may still be in flight when cudaMemcpy
  // returns); the scoring calls run on non-blocking streams, so they are
  // waited for here.
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cuda_fail(e, "uploading constant tables");
    free_ctx(c);
    return nullptr;
  }
  if (ensure_host_cap(c, (size_t)c->batch)) {
    free_ctx(c);
    return nullptr;
  }
  return c;
}

SS2_API ss2_ctx *ss2_create(int width, int height, int bitdepth, int chroma) {
  return create(width, height, bitdepth, chroma, 0);
}

SS2_API ss2_ctx *ss2_create_batch(int width, int height, int bitdepth, int chroma,
                                  int max_batch) {
  if (max_batch == 0) {
    fail(SS2_EINVAL, "batch 0 is outside 1..1024");
    return nullptr;
  }
  return create(width, height, bitdepth, chroma, max_batch);
}

SS2_API void ss2_destroy(ss2_ctx *ctx) { free_ctx(ctx); }

SS2_API size_t ss2_frame_bytes(const ss2_ctx *ctx) {
  return ctx ? (size_t)ctx->g.frame_bytes : 0;
}

SS2_API int ss2_batch(const ss2_ctx *ctx) { return ctx ? ctx->batch : 0; }

SS2_API size_t ss2_workspace_bytes(const ss2_ctx *ctx) { return ctx ? ctx->ws_bytes : 0; }

SS2_API int ss2_default_params(double *params, int n_params) {
  if (!params || n_params != kNParams)
    return fail(SS2_EINVAL, "parameter vector must hold %d doubles", kNParams);
  default_params(params);
  return 0;
}

SS2_API int ss2_set_params(ss2_ctx *ctx, const double *params, int n_params) {
  if (!ctx || !params || n_params != kNParams)
    return fail(SS2_EINVAL, "ss2_set_params needs a context and %d doubles", kNParams);
  for (int i = 0; i < kNParams; ++i)
    if (!std::isfinite(params[i])) return fail(SS2_EINVAL, "parameter %d is not finite", i);
  for (int i = 0; i < 3; ++i)
    if (!((float)params[kPBias + i] > 0.0f))
      return fail(SS2_EINVAL, "opsin bias %d must be positive", i);
  std::memcpy(ctx->params, params, sizeof(ctx->params));
  set_pix(ctx);
  ctx->graph.reset();  // the kernels' parameter block is baked into the graph
  CU(cudaMemcpy(ctx->d_params, ctx->params, sizeof(ctx->params), cudaMemcpyHostToDevice),
     "uploading parameters");
  // in place before any later call on a non-blocking stream reads them
  CU(cudaDeviceSynchronize(), "uploading parameters");
  return 0;
}

SS2_API int ss2_host_tables(float *eotf, float *iir) {
  if (eotf) build_eotf(eotf);
  if (iir) build_iir(iir, iir + 3);
  return 0;
}

// ---------------------------------------------------------------------------
// Per-kernel timing: when enabled, every launch is bracketed by a pair of
// events on the launching stream.
// ---------------------------------------------------------------------------

enum { kKPyramid = 0, kKHblur = 1, kKVblur = 2, kKFinalize = 3, kKClasses = 4 };

// Inside a graph capture the events become external event-record nodes of
// the graph (created per captured launch, owned by the graph).
static cudaError_t timed_mark(ss2_ctx *c, int cls, bool start, cudaStream_t st) {
  if (!c->capturing) return c->timer.mark(cls, start, st);
  if (!c->timer.on()) return cudaSuccess;
  cudaEvent_t e;
  cudaError_t r = cudaEventCreate(&e);
  if (r != cudaSuccess) return r;
  c->graph.ev.push_back(e);
  if (start) c->graph.cls.push_back(cls);
  return cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
}

#define TIMED(c, cls, st, launch, what)                  \
  do {                                                    \
    CU(timed_mark(c, cls, true, st), "event");            \
    CU(launch, what);                                     \
    CU(timed_mark(c, cls, false, st), "event");           \
  } while (0)

SS2_API int ss2_set_graphs(ss2_ctx *ctx, int enable) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  ctx->graphs = enable != 0;
  if (!ctx->graphs) ctx->graph.reset();
  return 0;
}

SS2_API int ss2_profile_begin(ss2_ctx *ctx) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  ctx->timer.begin();
  return 0;
}

SS2_API int ss2_profile_end(ss2_ctx *ctx, double *ms, int *launches) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  CU(ctx->timer.finish(kKClasses, ms, launches), "profile events");
  return 0;
}

// ---------------------------------------------------------------------------
// One pass of the pipeline over nb frames already on the device.
// ---------------------------------------------------------------------------

static int run_batch(ss2_ctx *c, Lane &L, const uint8_t *ref, const uint8_t *dis, int nb,
                     cudaEvent_t after_pyramid) {
  const Geom &g = c->g;
  cudaStream_t st = L.st;
  if (injected("launch")) return fail(SS2_EIO, "kernel launch failed (injected by SS2_FAULT=launch)");
  TIMED(c, kKPyramid, st, launch_pyramid(g, c->px, c->tabs, ref, dis, L.X, nb, st),
        "k_pyramid launch");
  if (after_pyramid) CU(cudaEventRecord(after_pyramid, st), "event record");
  TIMED(c, kKHblur, st, launch_hblur(g, c->px, L.maps, c->d_err, nb, st), "k_hblur launch");
  TIMED(c, kKVblur, st, launch_vblur(g, c->px, L.maps, L.X, L.part, c->d_err, nb, st),
        "k_vblur launch");
  TIMED(c, kKFinalize, st,
        launch_finalize(g, L.part, c->d_params, L.values, L.scores, nb, st),
        "k_finalize launch");
  return 0;
}

// Batches of a call: as few as the workspace allows, of near-equal size.
static void batch_plan(int n, int cap, int *nbatches, int *base, int *extra) {
  *nbatches = (n + cap - 1) / cap;
  *base = n / *nbatches;
  *extra = n % *nbatches;   // the first `extra` batches take one more frame
}

// The lanes' streams start after the work already on the caller's stream...
static int fork_lanes(ss2_ctx *c, cudaStream_t st) {
  CU(cudaEventRecord(c->ev_fork, st), "fork event");
  for (Lane &L : c->lane) CU(cudaStreamWaitEvent(L.st, c->ev_fork, 0), "fork wait");
  return 0;
}

// ...and the caller's stream continues after the lanes' work.
static int join_lanes(ss2_ctx *c, cudaStream_t st) {
  for (Lane &L : c->lane) {
    CU(cudaEventRecord(L.ev_done, L.st), "join event");
    CU(cudaStreamWaitEvent(st, L.ev_done, 0), "join wait");
  }
  return 0;
}

// Reads the kernels' error word after the stream's work (enqueue before the
// stream synchronisation, check after it).
static int enqueue_err_readback(ss2_ctx *c, cudaStream_t st) {
  CU(cudaMemcpyAsync(c->h_err, c->d_err, sizeof(int), cudaMemcpyDeviceToHost, st),
     "error word read-back");
  return 0;
}

static int check_err_word(ss2_ctx *c, cudaStream_t st) {
  if (*c->h_err == 0) return 0;
  const int bits = *c->h_err;
  *c->h_err = 0;
  cudaMemsetAsync(c->d_err, 0, sizeof(int), st);
  cudaStreamSynchronize(st);
  return fail(SS2_EIO, "a kernel gave up waiting for a TMA transfer (error bits 0x%x)", bits);
}

static int check_call(ss2_ctx *ctx, const void *ref, const void *dis, int n) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  if (n < 0) return fail(SS2_EINVAL, "negative frame count %d", n);
  if (n > 0 && (!ref || !dis)) return fail(SS2_EINVAL, "NULL frame pointer");
  return 0;
}

// After a failure part of a call's work may still be queued on the lanes:
// wait for it so that the context can be reused or destroyed safely.
static int drain(ss2_ctx *c, int rc) {
  for (Lane &L : c->lane)
    if (L.st) cudaStreamSynchronize(L.st);
  if (c->copy_stream) cudaStreamSynchronize(c->copy_stream);
  return rc;
}

static int read_back(ss2_ctx *c, double *dst, const double *src, size_t n, cudaStream_t st) {
  if (injected("memcpy"))
    return fail(SS2_EIO, "device-to-host copy failed (injected by SS2_FAULT=memcpy)");
  CU(cudaMemcpyAsync(dst, src, n * sizeof(double), cudaMemcpyDeviceToHost, st), "read-back");
  return 0;
}

// Enqueues a device-input call on st: the lanes fork from st, run the
// batches and read back, and st joins them and reads the error word.
static int enqueue_call(ss2_ctx *ctx, cudaStream_t st, const uint8_t *r8, const uint8_t *d8,
                        int n, bool values) {
  const long long fb = ctx->g.frame_bytes;
  int nbat, base, extra;
  batch_plan(n, ctx->batch, &nbat, &base, &extra);
  if (fork_lanes(ctx, st)) return t_err;
  for (int b = 0, f0 = 0; b < nbat; ++b) {
    const int nb = base + (b < extra ? 1 : 0);
    Lane &L = ctx->lane[b % kLanes];
    if (run_batch(ctx, L, r8 + f0 * fb, d8 + f0 * fb, nb, nullptr) ||
        read_back(ctx, ctx->h_scores + f0, L.scores, (size_t)nb, L.st) ||
        (values && read_back(ctx, ctx->h_values + (size_t)f0 * kNValues, L.values,
                             (size_t)nb * kNValues, L.st)))
      return t_err;
    f0 += nb;
  }
  if (join_lanes(ctx, st) || enqueue_err_readback(ctx, st)) return t_err;
  return 0;
}

// Captures the call into ctx->graph (on the context's own stream: the
// caller's may be the legacy default stream, which cannot be captured).
static int capture_call(ss2_ctx *ctx, const CallKey &key, const uint8_t *r8, const uint8_t *d8,
                        int n, bool values) {
  ctx->graph.reset();
  if (!ctx->cap_stream)
    CU(cudaStreamCreateWithFlags(&ctx->cap_stream, cudaStreamNonBlocking), "capture stream");
  CU(cudaStreamBeginCapture(ctx->cap_stream, cudaStreamCaptureModeRelaxed), "begin capture");
  ctx->capturing = true;
  const int rc = enqueue_call(ctx, ctx->cap_stream, r8, d8, n, values);
  ctx->capturing = false;
  // a failure after the fork leaves the lanes in the capture: join them so
  // that ending it releases every stream
  if (rc) join_lanes(ctx, ctx->cap_stream);
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(ctx->cap_stream, &graph);
  if (rc || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    ctx->graph.reset();
    cudaGetLastError();
    return rc ? rc : cuda_fail(e, "end capture");
  }
  const cudaError_t ei = cudaGraphInstantiate(&ctx->graph.exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess) {
    ctx->graph.exec = nullptr;
    ctx->graph.reset();
    cudaGetLastError();
    return cuda_fail(ei, "graph instantiation");
  }
  ctx->graph.key = key;
  return 0;
}

static int score_device(ss2_ctx *ctx, const void *ref, const void *dis, int n, double *scores,
                        double *values, void *stream) {
  if (check_call(ctx, ref, dis, n)) return t_err;
  if (n == 0) return 0;
  if (!scores && !values) return fail(SS2_EINVAL, "no output array");
  if (ensure_host_cap(ctx, (size_t)n)) return t_err;
  CU(cudaSetDevice(ctx->device), "cudaSetDevice");
  cudaStream_t st = (cudaStream_t)stream;
  const uint8_t *r8 = (const uint8_t *)ref, *d8 = (const uint8_t *)dis;
  bool replayed = false;
  if (ctx->graphs && ctx->warm) {
    CallKey key;
    key.ref = ref;
    key.dis = dis;
    key.n = n;
    key.values = values != nullptr;
    key.timed = ctx->timer.on();
    key.h_scores = ctx->h_scores;
    key.h_values = ctx->h_values;
    // a capture that fails (an injected fault, a call the capture refuses)
    // leaves the context on eager launches, which report the failure
    if (!(ctx->graph.exec && ctx->graph.key == key) &&
        capture_call(ctx, key, r8, d8, n, values != nullptr))
      ctx->graphs = false;
    if (ctx->graphs) {
      CU(cudaGraphLaunch(ctx->graph.exec, st), "graph launch");
      replayed = true;
    }
  }
  if (!replayed) {
    if (enqueue_call(ctx, st, r8, d8, n, values != nullptr)) return drain(ctx, t_err);
    ctx->warm = true;
  }
  CU(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  if (replayed && ctx->graph.key.timed) {
    for (size_t i = 0; i < ctx->graph.cls.size(); ++i) {
      float dt = 0.0f;
      CU(cudaEventElapsedTime(&dt, ctx->graph.ev[2 * i], ctx->graph.ev[2 * i + 1]),
         "graph timing events");
      ctx->timer.add(ctx->graph.cls[i], dt);
    }
  }
  if (check_err_word(ctx, st)) return t_err;
  if (scores) std::memcpy(scores, ctx->h_scores, (size_t)n * sizeof(double));
  if (values) std::memcpy(values, ctx->h_values, (size_t)n * kNValues * sizeof(double));
  return 0;
}

SS2_API int ss2_score_frames(ss2_ctx *ctx, const void *ref, const void *dis, int n_frames,
                             double *scores, void *stream) {
  if (n_frames > 0 && !scores) return fail(SS2_EINVAL, "NULL scores array");
  return score_device(ctx, ref, dis, n_frames, scores, nullptr, stream);
}

SS2_API int ss2_values(ss2_ctx *ctx, const void *ref, const void *dis, int n_frames,
                       double *values, double *scores, void *stream) {
  if (n_frames > 0 && !values) return fail(SS2_EINVAL, "NULL values array");
  return score_device(ctx, ref, dis, n_frames, scores, values, stream);
}

static int ensure_upload_slots(ss2_ctx *c) {
  if (c->lane[0].in) return 0;
  const size_t bytes = 2 * (size_t)c->batch * (size_t)c->g.frame_bytes;  // ref + dis
  size_t tot = 0;
  for (Lane &L : c->lane) {
    if (dev_alloc((void **)&L.in, bytes, &tot)) return t_err;
    CU(cudaEventCreateWithFlags(&L.ev_copied, cudaEventDisableTiming), "event");
    CU(cudaEventCreateWithFlags(&L.ev_consumed, cudaEventDisableTiming), "event");
  }
  c->ws_bytes += tot;
  CU(cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking), "copy stream");
  return 0;
}

SS2_API int ss2_score_frames_host(ss2_ctx *ctx, const void *ref_host, const void *dis_host,
                                  int n_frames, double *scores, void *stream) {
  if (check_call(ctx, ref_host, dis_host, n_frames)) return t_err;
  if (n_frames == 0) return 0;
  if (!scores) return fail(SS2_EINVAL, "NULL scores array");
  if (ensure_host_cap(ctx, (size_t)n_frames)) return t_err;
  CU(cudaSetDevice(ctx->device), "cudaSetDevice");
  if (ensure_upload_slots(ctx)) return t_err;
  cudaStream_t st = (cudaStream_t)stream;
  const long long fb = ctx->g.frame_bytes;
  const size_t half = (size_t)ctx->batch * (size_t)fb;
  const uint8_t *r8 = (const uint8_t *)ref_host, *d8 = (const uint8_t *)dis_host;
  // Nothing overlaps the first batch's upload, so the first batch is a
  // quarter of a full one (rounded up); the rest are planned as usual.
  const int first = std::min(n_frames, (ctx->batch + 3) / 4);
  int nbat = 0, base = 0, extra = 0;
  if (n_frames > first) batch_plan(n_frames - first, ctx->batch, &nbat, &base, &extra);
  if (fork_lanes(ctx, st)) return t_err;
  for (int b = 0, f0 = 0; b <= nbat; ++b) {
    const int nb = b == 0 ? first : base + (b - 1 < extra ? 1 : 0);
    Lane &L = ctx->lane[b % kLanes];
    uint8_t *dref = L.in, *ddis = L.in + half;
    // slot fence: the upload waits for the kernel that last read this lane's slot
    CU(cudaStreamWaitEvent(ctx->copy_stream, L.ev_consumed, 0), "slot fence");
    CU(cudaMemcpyAsync(dref, r8 + f0 * fb, (size_t)nb * fb, cudaMemcpyHostToDevice,
                       ctx->copy_stream),
       "ref upload");
    CU(cudaMemcpyAsync(ddis, d8 + f0 * fb, (size_t)nb * fb, cudaMemcpyHostToDevice,
                       ctx->copy_stream),
       "dis upload");
    CU(cudaEventRecord(L.ev_copied, ctx->copy_stream), "event record");
    CU(cudaStreamWaitEvent(L.st, L.ev_copied, 0), "upload wait");
    if (run_batch(ctx, L, dref, ddis, nb, L.ev_consumed) ||
        read_back(ctx, ctx->h_scores + f0, L.scores, (size_t)nb, L.st))
      return drain(ctx, t_err);
    f0 += nb;
  }
  if (join_lanes(ctx, st) || enqueue_err_readback(ctx, st)) return drain(ctx, t_err);
  CU(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  if (check_err_word(ctx, st)) return t_err;
  std::memcpy(scores, ctx->h_scores, (size_t)n_frames * sizeof(double));
  return 0;
}

SS2_API int ss2_debug_planes(ss2_ctx *ctx, const void *ref, const void *dis, int scale,
                             float *xyb, float *hblur, void *stream) {
  if (check_call(ctx, ref, dis, 1)) return t_err;
  if (scale < 0 || scale >= ctx->g.nscales)
    return fail(SS2_EINVAL, "scale %d is not computed for this geometry", scale);
  CU(cudaSetDevice(ctx->device), "cudaSetDevice");
  cudaStream_t st = (cudaStream_t)stream;
  const Geom &g = ctx->g;
  Lane &L = ctx->lane[0];
  CU(launch_pyramid(g, ctx->px, ctx->tabs, (const uint8_t *)ref, (const uint8_t *)dis, L.X,
                    1, st),
     "k_pyramid launch");
  CU(launch_hblur(g, ctx->px, L.maps, ctx->d_err, 1, st), "k_hblur launch");
  const size_t ws = g.ws[scale], hs = g.hs[scale];
  const size_t pitch_b = (size_t)g.pitch[scale] * sizeof(float);
  if (xyb)
    for (int p = 0; p < 6; ++p)
      CU(cudaMemcpy2DAsync(xyb + p * ws * hs, ws * sizeof(float),
                           L.X + g.xoff[scale] + p * g.plane[scale], pitch_b,
                           ws * sizeof(float), hs, cudaMemcpyDeviceToHost, st),
         "plane read-back");
  // blurred planes, per channel c: mu1, mu2, s11, s22 interleaved as quads
  // (de-interleaved on the host below), then s12
  std::vector<float> quads;
  if (hblur) {
    const size_t plane = (size_t)g.plane[scale];
    quads.resize(3 * 4 * plane);
    CU(cudaMemcpyAsync(quads.data(), L.H + g.hoff[scale], quads.size() * sizeof(float),
                       cudaMemcpyDeviceToHost, st),
       "quad read-back");
    for (int c = 0; c < 3; ++c)
      CU(cudaMemcpy2DAsync(hblur + (c * kNq + 4) * ws * hs, ws * sizeof(float),
                           L.H + g.hoff[scale] + (12 + c) * plane, pitch_b,
                           ws * sizeof(float), hs, cudaMemcpyDeviceToHost, st),
         "plane read-back");
  }
  if (enqueue_err_readback(ctx, st)) return t_err;
  CU(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  if (hblur) {
    const size_t pitch = (size_t)g.pitch[scale], plane = (size_t)g.plane[scale];
    for (int c = 0; c < 3; ++c)
      for (int q = 0; q < 4; ++q)
        for (size_t y = 0; y < hs; ++y)
          for (size_t x = 0; x < ws; ++x)
            hblur[(c * kNq + q) * ws * hs + y * ws + x] =
                quads[c * 4 * plane + (y * pitch + x) * 4 + q];
  }
  return check_err_word(ctx, st);
}

SS2_API int ss2_debug_linear(ss2_ctx *ctx, const void *ref, const void *dis, int scale,
                             float *lin, void *stream) {
  if (check_call(ctx, ref, dis, 1)) return t_err;
  if (scale < 0 || scale >= ctx->g.nscales)
    return fail(SS2_EINVAL, "scale %d is not computed for this geometry", scale);
  if (!lin) return fail(SS2_EINVAL, "NULL output");
  CU(cudaSetDevice(ctx->device), "cudaSetDevice");
  cudaStream_t st = (cudaStream_t)stream;
  const Geom &g = ctx->g;
  const size_t n = (size_t)6 * g.ws[scale] * g.hs[scale];
  float *d_lin = nullptr;
  CU(cudaMalloc(&d_lin, n * sizeof(float)), "cudaMalloc");
  cudaError_t e = launch_pyramid(g, ctx->px, ctx->tabs, (const uint8_t *)ref,
                                 (const uint8_t *)dis, ctx->lane[0].X, 1, st, d_lin, scale);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(lin, d_lin, n * sizeof(float), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(d_lin);
  if (e != cudaSuccess) return cuda_fail(e, "linear RGB read-back");
  return 0;
}

SS2_API int ss2_debug_cbrt(const float *x, float *y, long long n, void *stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return fail(SS2_EINVAL, "bad cbrt arguments");
  int dev = 0;
  if (check_device(&dev)) return t_err;
  cudaStream_t st = (cudaStream_t)stream;
  CU(launch_cbrt(x, y, n, st), "k_cbrt launch");
  CU(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  return 0;
}

SS2_API int ss2_debug_cbrt_host(const float *x, float *y, long long n) {
  if (n < 0 || (n > 0 && (!x || !y))) return fail(SS2_EINVAL, "bad cbrt arguments");
  for (long long i = 0; i < n; ++i) y[i] = cbrt_rn_host(x[i]);
  return 0;
}

SS2_API int ss2_debug_wait_probe(unsigned spins, void *stream) {
  int dev = 0;
  if (check_device(&dev)) return t_err;
  int *d_flag = nullptr;
  CU(cudaMalloc(&d_flag, sizeof(int)), "cudaMalloc");
  int h_flag = 0;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(d_flag, 0, sizeof(int), st);
  if (e == cudaSuccess) e = launch_wait_probe(spins, d_flag, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&h_flag, d_flag, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(d_flag);
  if (e != cudaSuccess) return cuda_fail(e, "wait probe");
  if (h_flag & kErrTmaTimeout)
    return fail(SS2_EIO, "the probe kernel gave up waiting on its barrier after %u polls", spins);
  return 0;
}
