// ss2_f32x2.cuh — packed fp32 pairs (the PTX ISA's .f32x2 arithmetic on
// sm_100-family GPUs).  A pair lives in one 64-bit register, low half first;
// each half is rounded exactly as the scalar instruction rounds it.
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

// a * b + c per half, one rounding each (fma.rn.f32x2)
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

}  // namespace ss2
