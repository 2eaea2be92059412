// ss2_device.cuh — device arithmetic for the ssimulacra2 kernels.
//
// Every fp32 operation of the pixel pipeline is written with an explicit
// round-to-nearest intrinsic (__fadd_rn, __fmul_rn, __fmaf_rn, __fdiv_rn) so
// that nothing is contracted or reassociated: "Research-1363: Device-resident
// ssimulacra2 and a single-wait MS-SSIM on SYCL", Finding 2 (contraction off,
// products in named temporaries, fma only in the YUV matrix) makes the
// pipeline up to the sums reproducible bit for bit.  The library is also
// compiled with -fmad=false.
//
// Double-float ("float pair") arithmetic follows Finding 4: the product of
// two floats is exact as a pair (two_prod, via fma), the quotient is two
// partial quotients, and sums of pairs renormalise after every addition.
// These are the classic error-free transformations of Dekker (1971) and
// Knuth (TAOCP vol. 2, 4.2.2): two_sum, quick_two_sum, two_prod.
#pragma once

#include <cstdint>

#include "ss2_impl.h"

namespace ss2 {

struct ff {
  float hi, lo;
};

// a + b = s + e exactly (Knuth two_sum).
__device__ __forceinline__ ff two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// a + b = s + e exactly when |a| >= |b| (Dekker quick_two_sum).
__device__ __forceinline__ ff quick_two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float e = __fsub_rn(b, __fsub_rn(s, a));
  return {s, e};
}

// a * b = p + e exactly (fma-based two_prod).
__device__ __forceinline__ ff two_prod(float a, float b) {
  float p = __fmul_rn(a, b);
  float e = __fmaf_rn(a, b, -p);
  return {p, e};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = two_sum(a.hi, b.hi);
  float e = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  return quick_two_sum(s.hi, e);
}

__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  ff p = two_prod(a.hi, b.hi);
  float c = __fmaf_rn(a.hi, b.lo, __fmul_rn(a.lo, b.hi));
  return quick_two_sum(p.hi, __fadd_rn(p.lo, c));
}

// a^2 as a pair without the final renormalisation: hi = fl(a.hi^2) and lo
// gathers that product's exact error and 2 a.hi a.lo in one fused rounding
// (a.lo^2, below 2^-46 a^2, is dropped).  If |a.lo| <= e |a.hi| then |lo| <= (2^-24 +
// 2.01 e) |hi|: from a quotient pair (e = 2^-23) the low word stays below
// 2^-20 |hi| after the two squarings of a fourth power, and each squaring
// adds about 2^-45 relative error.  The pair can be squared again or added
// to a sum (acc_add needs no normalised operand) without the three
// instructions of quick_two_sum.
__device__ __forceinline__ ff ff_sqr_lazy(ff a) {
  const ff p = two_prod(a.hi, a.hi);
  return {p.hi, __fmaf_rn(__fadd_rn(a.hi, a.hi), a.lo, p.lo)};
}

// Approximate reciprocal (relative error near 2^-23).  The .ftz form: every
// caller passes a normal operand whose reciprocal is normal (a variance sum
// plus C2 > 0, 1 + |x - mu| >= 1, 3 y^2 >= 2^-67), and for those the flush
// changes nothing while sparing the subnormal handling.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// a / b to within an ulp: the product a * (1/b) corrected by one
// Newton-Raphson step on its residual (Markstein, IBM J. Res. Dev. 34(1),
// 1990).  The quotient is faithful, so the residual a - q b it leaves is
// exactly representable and a second partial quotient recovers the rest.
// When a == b the corrected quotient is exactly 1.
__device__ __forceinline__ float div_newton(float a, float b, float rb) {
  const float q0 = __fmul_rn(a, rb);
  const float e = __fmaf_rn(-q0, b, a);
  return __fmaf_rn(e, rb, q0);
}

// a / b for a pair numerator and a float denominator: two partial quotients
// (Finding 4: "two correctly rounded partial quotients", here the first is
// faithful and the exact residual makes the pair accurate to about 2^-46).
__device__ __forceinline__ ff ff_div_f(ff a, float b) {
  const float rb = rcp_approx(b);
  const float q1 = div_newton(a.hi, b, rb);
  float r = __fmaf_rn(-q1, b, a.hi);
  r = __fadd_rn(r, a.lo);
  // |q2| is within an ulp of q1: the pair is usable without renormalising
  return {q1, __fmul_rn(r, rb)};
}

// a / b for pairs (same scheme, the denominator's low word enters the
// residual).
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  const float rb = rcp_approx(b.hi);
  const float q1 = div_newton(a.hi, b.hi, rb);
  float r = __fmaf_rn(-q1, b.hi, a.hi);
  r = __fadd_rn(r, a.lo);
  r = __fmaf_rn(-q1, b.lo, r);
  return {q1, __fmul_rn(r, rb)};
}

// ---------------------------------------------------------------------------
// Correctly rounded cube root (Finding 2 asks for the CPU's cube root exactly;
// the plain reading is cbrt rounded to nearest).  The exact decision below
// settles a guess that may be an ulp or two off, between it and its
// neighbours: the rounded
// result y satisfies (y - u/2)^3 < x < (y + u/2)^3 for the float spacing u
// around y, and each midpoint cube is compared with x in 128-bit integers.
// ---------------------------------------------------------------------------

// A positive finite float as X * 2^e, X an integer < 2^24.
__device__ __forceinline__ void float_parts(float v, uint32_t &X, int &e) {
  uint32_t b = __float_as_uint(v);
  uint32_t be = (b >> 23) & 0xffu;
  uint32_t m = b & 0x7fffffu;
  X = be ? (m | 0x800000u) : m;
  e = be ? (int)be - 150 : -149;
}

// Sign of (M 2^f)^3 - X 2^g, exact; M < 2^27, X < 2^24.
__device__ __forceinline__ int cube_cmp(uint32_t M, int f, uint32_t X, int g) {
  unsigned long long m2 = (unsigned long long)M * M;
  unsigned __int128 c = (unsigned __int128)m2 * M;   // < 2^81
  int d = 3 * f - g;
  if (d >= 0) {
    if (d >= 24) return 1;
    unsigned __int128 lhs = c << d;
    return lhs > X ? 1 : (lhs < X ? -1 : 0);
  }
  if (-d >= 104) return X ? -1 : 1;
  unsigned __int128 rhs = (unsigned __int128)X << (-d);
  return c > rhs ? 1 : (c < rhs ? -1 : 0);
}

// Exact rounding decision: moves y until x lies strictly between the cubes
// of the two midpoints around it.
__device__ __noinline__ float cbrt_round_exact(float x, float y) {
  uint32_t X;
  int g;
  float_parts(x, X, g);
#pragma unroll 1
  for (int it = 0; it < 4; ++it) {
    uint32_t Y;
    int e;
    float_parts(y, Y, e);
    if (cube_cmp(2u * Y + 1u, e - 1, X, g) < 0) {          // above upper midpoint
      y = __uint_as_float(__float_as_uint(y) + 1u);
      continue;
    }
    const bool floor_binade = (Y == 0x800000u) && (e > -149);
    const uint32_t Ml = floor_binade ? 4u * Y - 1u : 2u * Y - 1u;
    const int fl = floor_binade ? e - 2 : e - 1;
    if (cube_cmp(Ml, fl, X, g) > 0) {                       // below lower midpoint
      y = __uint_as_float(__float_as_uint(y) - 1u);
      continue;
    }
    break;
  }
  return y;
}

// Inputs below 2^-100 (zeros included): the first guess from CUDA's cbrtf,
// settled by the exact decision.  Out of line: it is rare, and inlining the
// library cube root at every call site would bloat the kernels' code.
__device__ __noinline__ float cbrt_tiny(float x) {
  return x == 0.0f ? x : cbrt_round_exact(x, cbrtf(x));
}

// log2 and 2^x approximations in the .ftz form: the cube root's fast path
// calls them only for x >= 2^-100, where neither operand nor result is
// subnormal.
__device__ __forceinline__ float lg2_approx(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Correctly rounded cbrt for x >= 0 finite, in two parts so that a caller
// with several cube roots can take one branch for all of their rare slow
// paths.  cbrt_fast:
//   1. y0 = 2^(log2(x) / 3) from the hardware approximations (within about
//      2^-20 relative).
//   2. The residual R = x - y0^3 to about 2^-43 x: y0^2 = p + e exactly
//      (fma), then x - y0 p and the y0 e term each in one fma (the product
//      exact inside it); R is below about 2^-19 x, so each of the two
//      roundings is below about 2^-44 x.
//   3. One Newton step y0 + R k, k = 1 / (3 y0^2), whose error is about
//      2^-41 y0: y.hi = fma(R, k, y0) rounds the step once, and y.lo =
//      fma(R, k, y0 - y.hi) is its rounding error to within 2^-24 of itself
//      (y0 - y.hi is exact by Sterbenz, the correction being below 2^-19 y0):
//      the root lies at y.hi + y.lo, give or take 2^-41 y0.
//   4. y.hi is the nearest float when y.lo is below half the float spacing
//      on its side of y.hi, with a margin that covers that 2^-41: one fma
//      decides it, y.hi + y.lo (1 + 2^-13) rounding back to y.hi (rounding
//      uses the spacing on the side y.lo points to, so the halved spacing
//      below a power of two is taken care of).
// It returns y.hi and whether that is settled; it is not for near-ties
// (about one input in 2^13) and x < 2^-100 (where the products' error terms
// underflow; zeros included), which cbrt_slow decides exactly (128-bit
// integer test, CUDA's cbrtf as the first guess for the tiny inputs).
__device__ __forceinline__ float cbrt_fast(float x, bool &settled) {
  const float y0 = ex2_approx(__fmul_rn(lg2_approx(x), 0.333333343f));
  const ff p = two_prod(y0, y0);
  float r = __fmaf_rn(-y0, p.hi, x);
  r = __fmaf_rn(-y0, p.lo, r);
  const float k = rcp_approx(__fmul_rn(3.0f, p.hi));
  const float hi = __fmaf_rn(r, k, y0);
  const ff y = {hi, __fmaf_rn(r, k, __fsub_rn(y0, hi))};
  // x >= 2^-100 (x is not negative here; zeros fail the test)
  settled = x >= 7.8886090522101181e-31f && __fmaf_rn(y.lo, 1.0001220703125f, y.hi) == y.hi;
  return y.hi;
}

__device__ __noinline__ float cbrt_slow(float x, float y) {
  if ((__float_as_uint(x) << 1) < (0x0d800000u << 1)) return cbrt_tiny(x);
  return cbrt_round_exact(x, y);
}

__device__ __forceinline__ float cbrt_cr(float x) {
  bool settled;
  const float y = cbrt_fast(x, settled);
  return settled ? y : cbrt_slow(x, y);
}

// ---------------------------------------------------------------------------
// Pixel pipeline pieces (one rounding per written operation).
// ---------------------------------------------------------------------------

__device__ __forceinline__ float clamp01(float v) {
  if (v < 0.0f) return 0.0f;
  if (v > 1.0f) return 1.0f;
  return v;
}

// clamp01(fma(a, b, c)) in one instruction (the .sat form clamps the
// rounded result to [0, 1]; a NaN, which the finite operands here never
// give, would become 0, and -0 is equivalent downstream: the EOTF maps both
// zeros to +0).
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float r;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// (float)n / d correctly rounded without a division, for d = 219 k or
// 224 k (k a power of two) and |n| <= 65536, from rd = RN(1 / d): the
// product, its exact fma residual and one correction.  Checked against the
// IEEE quotient for every such n and both divisors (the power-of-two k
// scales every step exactly); the limited-range normalisation of samples of
// any depth stays within that range.
__device__ __forceinline__ float norm_div(int n, float d, float rd) {
  const float nf = (float)n;
  const float q0 = __fmul_rn(nf, rd);
  return __fmaf_rn(__fmaf_rn(-q0, d, nf), rd, q0);
}

// Linear interpolation in the sRGB EOTF table (uniform grid, 4096 intervals),
// stored as (T[i], T[i+1] - T[i]) pairs plus a last pair (T[4096], 0): for
// v in [0, 1] the index is at most 4096 and needs no clamp.
__device__ __forceinline__ float eotf_lookup(const float2 *__restrict__ P, float v) {
  float t = __fmul_rn(v, (float)kEotfN);
  int i = (int)t;
  float f = __fsub_rn(t, (float)i);
  const float2 e = __ldg(P + i);
  return __fmaf_rn(f, e.y, e.x);
}

// Linear RGB -> XYB with the make-positive affine.  The three cube roots
// share one branch to their rare slow paths.
__device__ __forceinline__ void pixel_xyb(const Pix &p, const float cb[3], float r,
                                          float g, float b, float &X, float &Y,
                                          float &B) {
  float m[3], root[3];
  bool ok[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    float t0 = __fmul_rn(p.opsin[3 * i + 0], r);
    float t1 = __fmul_rn(p.opsin[3 * i + 1], g);
    float t2 = __fmul_rn(p.opsin[3 * i + 2], b);
    float s = __fadd_rn(__fadd_rn(t0, t1), t2);
    s = __fadd_rn(s, p.bias[i]);
    m[i] = s < 0.0f ? 0.0f : s;
    root[i] = cbrt_fast(m[i], ok[i]);
  }
  if (!(ok[0] && ok[1] && ok[2])) {
#pragma unroll
    for (int i = 0; i < 3; ++i)
      if (!ok[i]) root[i] = cbrt_slow(m[i], root[i]);
  }
  float c[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) c[i] = __fsub_rn(root[i], cb[i]);
  float x = __fmul_rn(0.5f, __fsub_rn(c[0], c[1]));
  float y = __fmul_rn(0.5f, __fadd_rn(c[0], c[1]));
  X = __fadd_rn(__fmul_rn(x, p.sx), p.ox);
  Y = __fadd_rn(y, p.oy);
  B = __fadd_rn(__fmul_rn(__fsub_rn(c[2], y), p.sb), p.ob);
}

}  // namespace ss2
