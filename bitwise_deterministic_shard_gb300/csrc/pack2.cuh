// Two binary32 lanes in one 64-bit register, on the packed FP32 instructions of sm_100 and
// later (add / mul / fma .rn.f32x2).  Each lane is rounded exactly as the scalar .rn
// instruction rounds it (to nearest even, subnormals kept), so a packed evaluation gives the
// same bits as two scalar ones while issuing half the floating-point instructions.
#pragma once
#include <cstdint>
#include "numerics.cuh"

namespace detattn {
namespace f2 {

typedef unsigned long long u64;

__device__ __forceinline__ u64 pack(float lo, float hi) {
  u64 d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void unpack(u64 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ u64 splat(float c) { return pack(c, c); }
__device__ __forceinline__ u64 add(u64 a, u64 b) {
  u64 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 sub(u64 a, u64 b) {
  u64 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 mul(u64 a, u64 b) {
  u64 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 fma(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

}  // namespace f2

// exp32_det_poly on two arguments at once (both in [-104, 0]): the same reduction and
// polynomial, step for step, in the packed lanes.  RN(tr - MAGIC) is taken as RN(tr + (-MAGIC))
// and RN(-kf C + r) as RN(kf (-C) + r): the same exact values, so the same roundings.
// t = RN(x log2 e) is two scalar multiplies: a packed multiply whose result feeds a packed add
// has come out of the compiler as one fused operation (one rounding of x log2 e + 1.5 2^23),
// which moves k by one where RN(x log2 e) lands on a half-integer; the scalar .rn multiply is
// never fused.  An exhaustive device test compares this form with the scalar one.
__device__ __forceinline__ void exp32_det_poly2(float xa, float xb, float& pa, float& pb, int& ka, int& kb) {
  using namespace f2;
  const u64 xx = pack(xa, xb);
  const u64 tr = add(pack(__fmul_rn(xa, 0x1.715476p+0f), __fmul_rn(xb, 0x1.715476p+0f)), splat(12582912.0f));
  const u64 kf = add(tr, splat(-12582912.0f));
  const u64 r = fma(kf, splat(-0x1.7f7d1cp-20f), fma(kf, splat(-0x1.62e4p-1f), xx));
  u64 p = fma(splat(0x1.a01a02p-13f), r, splat(0x1.6c16c2p-10f));
  p = fma(p, r, splat(0x1.111112p-7f));
  p = fma(p, r, splat(0x1.555556p-5f));
  p = fma(p, r, splat(0x1.555556p-3f));
  p = fma(p, r, splat(0.5f));
  p = fma(p, r, splat(1.0f));
  p = fma(p, r, splat(1.0f));
  float ta, tb;
  unpack(tr, ta, tb);
  ka = __float_as_int(ta) - 0x4B400000;
  kb = __float_as_int(tb) - 0x4B400000;
  unpack(p, pa, pb);
}

}  // namespace detattn
