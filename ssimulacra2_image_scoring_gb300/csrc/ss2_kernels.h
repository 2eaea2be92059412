// ss2_kernels.h — host-side launchers of the ssimulacra2 kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ss2_impl.h"

namespace ss2 {

// lin_dbg: NULL, or 6 planes of ws x hs floats of scale dbg_scale (ref R, G,
// B, dis R, G, B) that receive the linear RGB of that scale (parity tests).
cudaError_t launch_pyramid(const Geom &g, const Pix &px, const PyrTabs &tabs, const uint8_t *ref,
                           const uint8_t *dis, float *X, int nframes, cudaStream_t st,
                           float *lin_dbg = nullptr, int dbg_scale = -1);
cudaError_t launch_hblur(const Geom &g, const Pix &px, const PlaneMaps &maps, int *err,
                         int nframes, cudaStream_t st);
cudaError_t launch_vblur(const Geom &g, const Pix &px, const PlaneMaps &maps, const float *X,
                         float2 *part, int *err, int nframes, cudaStream_t st);
// err: NULL, or an error word; when it is non-zero at the time k_finalize
// runs, every score and value of the batch is written as NaN.
cudaError_t launch_finalize(const Geom &g, const float2 *part, const double *params,
                            double *values, double *scores, int nframes, cudaStream_t st,
                            const int *err = nullptr);

cudaError_t launch_cbrt(const float *x, float *y, long long n, cudaStream_t st);
cudaError_t launch_wait_probe(uint32_t spins, int *err, cudaStream_t st);

}  // namespace ss2
