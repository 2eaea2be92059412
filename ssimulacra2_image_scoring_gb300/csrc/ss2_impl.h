// ss2_impl.h — internal types shared by the host side of libss2 and its
// kernels: the geometry of a context's workspace and the per-pixel
// constants passed to every launch by value.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>

namespace ss2 {

constexpr int kMaxScales = 6;
constexpr int kNValues = 108;
constexpr int kNParams = 133;
constexpr int kEotfN = 4096;   // table intervals; the table has kEotfN + 1 entries
constexpr int kEotfPairs = kEotfN + 1;  // device (value, slope) pairs, the last (T[N], 0)
constexpr int kIirR = 4;       // recursive Gaussian support |m| <= R
constexpr int kReach = kIirR + 1;  // taps at n +- (R + 1)
constexpr int kNq = 5;         // blurred quantities per channel: mu1 mu2 s11 s22 s12
constexpr int kNSum = 6;       // d, d^4, art, art^4, det, det^4

// Parameter vector offsets (doubles), see include/ss2.h.
constexpr int kPWeights = 0, kPPoly = 108, kPPower = 112, kPOpsin = 115, kPBias = 124,
              kPAffine = 127, kPC2 = 132;

// Workspace geometry of one context.  Planes at scale s are fp32, row-major,
// pitch[s] floats per row (a multiple of 32), plane[s] = pitch[s] * hs[s].
//   X block of a frame:  6 planes per scale (ref X Y B, dis X Y B) at xoff[s]
//   H block of a frame: 15 planes per scale (channel-major, 5 quantities)
//   partials of a frame: float2 pairs, (channel * 6 + sum) * nw[s] + warp,
//                         at poff[s]
struct Geom {
  int w, h, depth, chroma, sx, sy, cw, ch, bps;
  int nscales;
  int ws[kMaxScales], hs[kMaxScales], pitch[kMaxScales], nw[kMaxScales];
  long long plane[kMaxScales];
  long long xoff[kMaxScales], hoff[kMaxScales];
  long long x_fs, h_fs;            // floats per frame
  int poff[kMaxScales];
  int p_fs;                        // float2 per frame
  long long frame_bytes;
  // flat work decomposition over the scales
  int hunit_off[kMaxScales + 1];   // prefix of 3 * ceil(hs[s] / 32) (horizontal warps)
  int vwarp_off[kMaxScales + 1];   // prefix of 3 * nw[s]            (vertical warps)
};

// TMA descriptors, one per scale.  x[s] views the XYB block as a 4-D tensor
// (column, row, plane 0..5, frame).  The horizontally blurred block of a
// scale holds, per channel c, the quantities mu1, mu2, s11, s22 interleaved
// (four floats per pixel: the "quad" rows, 4 x pitch floats each, channel c
// at c * 4 * plane) and then, per channel, the s12 plane (at 12 * plane +
// c * plane).  q4 / vq4 view the quads as a 4-D tensor (float of the quad
// row, row, channel, frame), s1 / vs1 the s12 planes as (column, row,
// channel, frame).
//   x, s1:  8-column x 32-row boxes (row walkers of the horizontal pass)
//   q4:     32-float (8-pixel) x 32-row boxes, 128-byte swizzled in shared
//           memory (one box row is one 128-byte line)
//   vq4:    128-float (32-pixel) x 8-row boxes, vs1: 32-column x 8-row
//           boxes (column walkers, one channel)
// Each pass gets only its own maps, which keeps the kernels' parameters
// under 4 KB.
struct HMaps {
  CUtensorMap x[kMaxScales];
  CUtensorMap q4[kMaxScales];
  CUtensorMap s1[kMaxScales];
};
struct VMaps {
  CUtensorMap vq4[kMaxScales];
  CUtensorMap vs1[kMaxScales];
};
struct PlaneMaps {
  HMaps h;
  VMaps v;
};
constexpr int kBoxCols = 8, kBoxRows = 32;      // horizontal pass box
constexpr int kVCols = 32, kVRows = 8;          // vertical pass box

// Tables the pyramid kernel reads.  eotf: 4097 (value, slope) pairs of the
// sRGB EOTF table, slope = T[i+1] - T[i] rounded to float, and a last pair
// (T[4096], 0) so that an input of exactly 1 needs no index clamp.
// ynorm / cnorm (8-bit samples only, else null): the limited-range
// normalisations (v - 16) / 219 and (v - 128) / 224 of every sample value v,
// each a correctly rounded float quotient.  rdy / rdc: RN(1 / (219 k)) and
// RN(1 / (224 k)), k = 2^(depth - 8), for the division-free normalisation
// of deeper samples (and of 8-bit ones when the tables are null).
struct PyrTabs {
  const float2 *eotf;
  const float *ynorm;
  const float *cnorm;
  float rdy, rdc;
};

// Per-pixel constants (fp32 pipeline), rounded from the parameter vector.
struct Pix {
  float yuv[4];        // cr->R', cb->G' (magnitude), cr->G' (magnitude), cb->B'
  float opsin[9];
  float bias[3];
  float cbias[3];      // cbrt(bias[i]), correctly rounded (set on the host)
  float sx, ox, oy, sb, ob;
  float c2;
  float iir_c2[3];     // 2 cos(w_k)
  float iir_g[3];      // a_k cos(w_k R)
};

}  // namespace ss2
