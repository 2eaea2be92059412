// ss2_host.h — host-side helpers of libss2 shared by its entry points:
// error reporting, argument checks, workspace geometry and the constant
// tables the kernels read.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <utility>
#include <vector>

#include "ss2_impl.h"

namespace ss2 {

// Records code and message as the calling thread's last failure; returns code.
int fail(int code, const char *fmt, ...);
int cuda_fail(cudaError_t e, const char *what);

int check_geometry(int w, int h, int depth, int chroma);  // 0 or -EINVAL
int check_device(int *dev);                               // 0 or -ENOTSUP / -EIO
void make_geom(int w, int h, int depth, int chroma, Geom &g);
size_t per_frame_bytes(const Geom &g);                    // workspace bytes per frame

// TMA descriptors of the XYB and blurred-plane stacks of a workspace holding
// `batch` frames (X, H: device bases of the frame blocks).
int encode_maps(const Geom &g, float *X, float *H, int batch, PlaneMaps &maps);

void default_params(double *params);                      // kNParams doubles
void build_pix(const double *params, Pix &p);
void build_eotf(float *table);                            // kEotfN + 1 floats
void build_eotf_pairs(float *pairs);                      // 2 * kEotfPairs floats
int norm_entries(int depth);                              // 256 (8-bit) or 0
void build_norm(int depth, float *ynorm, float *cnorm);   // norm_entries(depth) each

// Per-kernel CUDA-event timing of one context (the ss2*_profile_begin /
// _end entry points): while on, each launch is bracketed by a pair of events
// recorded on its own stream; finish() waits for them and adds the elapsed
// times per kernel class.  The events are created on first use and reused.
class KernelTimer {
 public:
  KernelTimer() = default;
  KernelTimer(const KernelTimer &) = delete;
  KernelTimer &operator=(const KernelTimer &) = delete;
  ~KernelTimer() {
    for (cudaEvent_t e : pool_) cudaEventDestroy(e);
  }

  void begin() {
    on_ = true;
    used_.clear();
    added_.clear();
  }

  bool on() const { return on_; }

  // Adds one launch of class cls timed outside the event pool (the timing
  // events of a replayed CUDA graph, read after its stream synchronised).
  void add(int cls, float ms) {
    if (on_) added_.push_back({cls, ms});
  }

  // Records the start (start = true) or end event of one launch of class cls.
  cudaError_t mark(int cls, bool start, cudaStream_t st) {
    if (!on_) return cudaSuccess;
    size_t idx;
    if (start) {
      idx = used_.size() * 2;
      while (pool_.size() < idx + 2) {
        cudaEvent_t e;
        const cudaError_t r = cudaEventCreate(&e);
        if (r != cudaSuccess) return r;
        pool_.push_back(e);
      }
      used_.push_back({cls, idx});
    } else {
      if (used_.empty()) return cudaErrorInvalidValue;
      idx = used_.back().second + 1;
    }
    return cudaEventRecord(pool_[idx], st);
  }

  // Sums per class into ms[0..ncls) and launches[0..ncls) (either may be
  // NULL) and stops timing, also on failure.
  cudaError_t finish(int ncls, double *ms, int *launches) {
    std::vector<double> t((size_t)ncls, 0.0);
    std::vector<int> n((size_t)ncls, 0);
    cudaError_t e = cudaSuccess;
    for (const auto &u : used_) {
      e = cudaEventSynchronize(pool_[u.second + 1]);
      float dt = 0.0f;
      if (e == cudaSuccess) e = cudaEventElapsedTime(&dt, pool_[u.second], pool_[u.second + 1]);
      if (e != cudaSuccess) break;
      if (u.first >= 0 && u.first < ncls) {
        t[(size_t)u.first] += dt;
        n[(size_t)u.first] += 1;
      }
    }
    for (const auto &a : added_)
      if (a.first >= 0 && a.first < ncls) {
        t[(size_t)a.first] += a.second;
        n[(size_t)a.first] += 1;
      }
    on_ = false;
    used_.clear();
    added_.clear();
    if (e != cudaSuccess) return e;
    for (int i = 0; i < ncls; ++i) {
      if (ms) ms[i] = t[(size_t)i];
      if (launches) launches[i] = n[(size_t)i];
    }
    return cudaSuccess;
  }

 private:
  bool on_ = false;
  std::vector<cudaEvent_t> pool_;
  std::vector<std::pair<int, size_t>> used_;  // (kernel class, index of the start event)
  std::vector<std::pair<int, float>> added_;  // (kernel class, milliseconds)
};

}  // namespace ss2
