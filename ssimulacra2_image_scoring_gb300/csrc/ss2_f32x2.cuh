// ss2_f32x2.cuh — packed fp32 pairs (the PTX ISA's .f32x2 arithmetic on
// sm_100-family GPUs).  A pair lives in one 64-bit register, low half first;
// each half is rounded exactly as the scalar instruction rounds it (checked
// on a GB300 element by element against the scalar instructions for fma,
// add, mul and sub over 4 M pairs).
//
// There is deliberately no pair multiply here: on the same GPU a
// mul.rn.f32x2 whose result feeds an add.rn.f32x2 came out contracted into
// one fused operation despite the .rn modifiers (a quarter of 4 M sums of
// two squares differed from the twice-rounded scalar value), so products
// that must be rounded on their own are formed with scalar __fmul_rn.
#pragma once

#include <cstdint>

namespace ss2 {

using f2 = unsigned long long;

__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f2_unpack(f2 v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// a + b per half, one rounding each (add.rn.f32x2)
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// a - b per half, one rounding each (sub.rn.f32x2)
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
  f2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// a * b + c per half, one rounding each (fma.rn.f32x2)
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

}  // namespace ss2
