// noalloc.cu — ss2_score_frames_noalloc: scoring without any allocation.
//
// Some callers cannot allocate device memory at scoring time: code running
// under an allocator that must not be re-entered (a custom caching allocator
// or a memory-pool callback that asks for a score), processes whose device
// memory budget is fixed up front, and plug-ins that are handed device
// buffers by a host application that forbids them from calling cudaMalloc.
// They cannot create an ss2_ctx, whose workspace is cudaMalloc'd.
//
// This entry point runs the same four kernels as ss2_score_frames, one batch
// of frames at a time, with every intermediate plane, partial sum and pooled
// value placed in one file-scope device array of fixed size (kScratchBytes,
// 64 MiB).  Every GPU that loads the library holds that array until the
// process exits.  The caller passes the device input frames and a device
// array for the scores; nothing is read back and nothing is allocated:
// no cudaMalloc, cudaFree, pinned memory or allocating library routine.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and copies the constant
// tables (sRGB EOTF table and the default parameter vector) into the
// array's head with synchronous copies.  Make that first call before any
// stream capture on the device.  Later calls enqueue kernels only.
//
// Sharing: all calls on a device share the one array, which keeps the last
// call's contents.  Each call clears the array's error word on its stream
// before its kernels run, and its kernels write every other scratch word
// before reading it.  Calls whose work overlaps on the GPU (different
// streams, or different host threads without ordering) race on the array and
// corrupt each other's scores; order them on one stream.
//
// Failure signal: the blur kernels' bounded waits raise a bit in that error
// word when a copy never arrives.  Nothing is read back, so the host cannot
// see it; instead k_finalize writes NaN to every score of its batch when the
// word is set, which marks the failed batch and every later batch of the
// call.
//
// Device reset: the set-up is cached per device for the life of the
// process.  After cudaDeviceReset the array's contents (the constant tables)
// are gone, so this entry point must not be used in a process that has
// reset a device it ran on.
//
// Parameters: the library defaults (see ss2_default_params).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/ss2.h"
#include "ss2_host.h"
#include "ss2_impl.h"
#include "ss2_kernels.h"

#define SS2_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;   // 64 MiB
constexpr size_t kAlign = 256;
constexpr size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// head of the array: constant tables written once at set-up
constexpr size_t kEotfOff = 0;
constexpr size_t kParamsOff = align_up(kEotfOff + sizeof(float) * 2 * ss2::kEotfPairs);
constexpr size_t kErrOff = align_up(kParamsOff + sizeof(double) * ss2::kNParams);
constexpr size_t kHeadBytes = align_up(kErrOff + sizeof(int));

constexpr int kMaxDevices = 64;

std::mutex g_setup_mutex;
unsigned char *g_dev_ptr[kMaxDevices] = {};   // device address of g_scratch per device

// Test hook (ss2_debug_noalloc_timeout): when non-zero, each call runs a
// bounded wait that nothing completes, with this poll limit, against the
// call's error word, so that the failure signal can be checked.
std::atomic<unsigned> g_timeout_probe_spins{0};

}  // namespace

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

using namespace ss2;

// Device address of g_scratch on the current device, with the constant
// tables in place (first call per device does the set-up).
static int scratch_for_device(int dev, unsigned char **out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(SS2_ENOTSUP, "device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_dev_ptr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    float table[2 * kEotfPairs];
    double params[kNParams];
    build_eotf_pairs(table);
    default_params(params);
    unsigned char *base = static_cast<unsigned char *>(p);
    e = cudaMemcpy(base + kEotfOff, table, sizeof(table), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(base + kParamsOff, params, sizeof(params), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(base + kErrOff, 0, sizeof(int));
    // ordered on the legacy stream only: wait before the caller's stream runs
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "scratch set-up copy");
    g_dev_ptr[dev] = base;
  }
  *out = g_dev_ptr[dev];
  return 0;
}

SS2_API int ss2_score_frames_noalloc(int width, int height, int bitdepth, int chroma,
                                     const void *ref, const void *dis, int n_frames,
                                     double *scores, void *stream) {
  if (check_geometry(width, height, bitdepth, chroma)) return SS2_EINVAL;
  if (n_frames < 0) return fail(SS2_EINVAL, "negative frame count %d", n_frames);
  if (n_frames > 0 && (!ref || !dis || !scores))
    return fail(SS2_EINVAL, "NULL frame or score pointer");
  Geom g;
  make_geom(width, height, bitdepth, chroma, g);
  // per frame: XYB planes, blurred planes, partial pairs, 108 pooled values
  const size_t x_bytes = align_up((size_t)g.x_fs * sizeof(float));
  const size_t h_bytes = align_up((size_t)g.h_fs * sizeof(float));
  const size_t p_bytes = align_up((size_t)g.p_fs * sizeof(float2));
  const size_t v_bytes = align_up((size_t)kNValues * sizeof(double));
  const size_t per_frame = x_bytes + h_bytes + p_bytes + v_bytes;
  const size_t avail = kScratchBytes - kHeadBytes;
  if (per_frame > avail)
    return fail(SS2_EINVAL,
                "%dx%d needs %zu bytes of scratch per frame; the allocation-free entry point "
                "holds %zu bytes (64 MiB), about 600k pixels per frame",
                width, height, per_frame, avail);
  if (n_frames == 0) return 0;
  int dev = 0;
  if (check_device(&dev)) return ss2_last_error();
  unsigned char *base = nullptr;
  if (scratch_for_device(dev, &base)) return ss2_last_error();

  const int nb_max = (int)std::min<size_t>(avail / per_frame, 1024);
  unsigned char *work = base + kHeadBytes;
  float *X = reinterpret_cast<float *>(work);
  float *H = reinterpret_cast<float *>(work + nb_max * x_bytes);
  float2 *part = reinterpret_cast<float2 *>(work + nb_max * (x_bytes + h_bytes));
  double *values = reinterpret_cast<double *>(work + nb_max * (x_bytes + h_bytes + p_bytes));
  PyrTabs tabs;
  tabs.eotf = reinterpret_cast<const float2 *>(base + kEotfOff);
  tabs.ynorm = nullptr;   // normalisation without tables on the device
  tabs.cnorm = nullptr;
  tabs.rdy = 1.0f / (float)(219 << (bitdepth - 8));
  tabs.rdc = 1.0f / (float)(224 << (bitdepth - 8));
  const double *params = reinterpret_cast<const double *>(base + kParamsOff);
  // the kernels index frames by g.x_fs / g.h_fs / g.p_fs; use the padded strides
  g.x_fs = (long long)(x_bytes / sizeof(float));
  g.h_fs = (long long)(h_bytes / sizeof(float));
  g.p_fs = (int)(p_bytes / sizeof(float2));

  double pdef[kNParams];
  default_params(pdef);
  Pix px;
  build_pix(pdef, px);
  PlaneMaps maps;
  if (encode_maps(g, X, H, nb_max, maps)) return ss2_last_error();
  int *err = reinterpret_cast<int *>(base + kErrOff);
  cudaStream_t st = (cudaStream_t)stream;
  // a word left set by an earlier call must not mark this call's scores
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), st);
  if (e != cudaSuccess) return cuda_fail(e, "error word reset");
  const unsigned probe = g_timeout_probe_spins.load();
  if (probe) {
    e = launch_wait_probe(probe, err, st);
    if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
  }
  const uint8_t *r8 = static_cast<const uint8_t *>(ref), *d8 = static_cast<const uint8_t *>(dis);
  for (int f0 = 0; f0 < n_frames; f0 += nb_max) {
    const int nb = std::min(nb_max, n_frames - f0);
    const long long off = (long long)f0 * g.frame_bytes;
    e = launch_pyramid(g, px, tabs, r8 + off, d8 + off, X, nb, st);
    if (e == cudaSuccess) e = launch_hblur(g, px, maps, err, nb, st);
    if (e == cudaSuccess) e = launch_vblur(g, px, maps, X, part, err, nb, st);
    if (e == cudaSuccess) e = launch_finalize(g, part, params, values, scores + f0, nb, st, err);
    if (e != cudaSuccess) return cuda_fail(e, "allocation-free scoring launch");
  }
  return 0;
}

SS2_API int ss2_debug_noalloc_timeout(unsigned spins) {
  g_timeout_probe_spins.store(spins);
  return 0;
}
