// ss2_host.h — host-side helpers of libss2 shared by its entry points:
// error reporting, argument checks, workspace geometry and the constant
// tables the kernels read.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

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
void build_eotf_pairs(float *pairs);                      // 2 * kEotfN floats
int norm_entries(int depth);                              // 256 or 65536
void build_norm(int depth, float *ynorm, float *cnorm);   // norm_entries(depth) each

}  // namespace ss2
