// RN32(RN64(p / d)) of a binary32 p by a binary64 d on the FP32 pipe, with a certificate.
//
// The cross-entropy gradient divides every weight of a row by the row's binary64
// denominator (det-cross-entropy "Method": softmax(x_i) = w / denom, one RN64 and one RN32;
// the quotient then feeds the binary32 gradient).  The divisor is split once per row into
// d_hi = RN32(d), d_lo = RN32(d - d_hi) and r = RN32(1 / d_hi); each quotient then
// takes one multiply and five fused multiply-adds:
//   q0 = RN(p r)                      (within about 2 units of 2^-24 of Q = p / d)
//   e  = RN(p - q0 d_hi), e2 = RN(e - q0 d_lo)      (the residual p - q0 d)
//   q1 = RN(q0 + e2 r)                (the candidate, RN32 of a value within 2^-44 Q of Q)
//   dl = RN((q0 - q1) + e2 r)         (Q - q1, q0 - q1 exact)
// With u = 2^-24: d = d_hi + d_lo + eta, |eta| <= u^2 d; the residual e2 is within 6 u^2 p
// of p - q0 d; r is within (2 u + u^2) / d of 1 / d; so (q0 - q1) + e2 r is within 12.1 u^2 Q
// of Q - q1 and dl within 14.3 u^2 Q < 2^-44 Q (the rounding of dl adds about u^2 Q).  Let
// h = 2^(E - 24), half a unit in the last place of q1 in [2^E, 2^(E+1)).  If
// |dl| < h - 2^(E - 39), then |Q - q1| < h - 2^(E - 39) + 2^-44 Q < h - 2^(E - 40) (as
// Q < 2^(E+2)): q1 = RN32(Q), and every half-way point lies more than 2^(E - 40) > 2^-53 Q
// from Q, farther than RN64 moves it, so q1 = RN32(RN64(Q)) too.  q1 a power of two (a
// smaller half-unit below it) is not certified.  Arguments: p in [0.5, 2), d in
// [2^-60, 2^60], so that every intermediate is a normal binary32.  Otherwise, or when the
// certificate fails (about one quotient in 2^15), the caller divides exactly (divide.cuh).
//
// This is the classical correction of a reciprocal-based quotient by its residual (as in
// P. Markstein, "Computation of elementary functions on the IBM RISC System/6000 processor",
// IBM J. Res. Dev. 34(1), 1990), with an explicit bound in place of a proof of correct
// rounding for every input.  Also compiles as plain C++ for the host tests.
#pragma once
#include <cstdint>
#if !defined(__CUDA_ARCH__)
#include <cmath>
#include <cstring>
#endif

#if defined(__CUDACC__)
#define DA_FD __host__ __device__ __forceinline__
#else
#define DA_FD inline
#endif

namespace detattn {
namespace fdiv {

#if defined(__CUDA_ARCH__)
DA_FD float fma_rn(float a, float b, float c) { return __fmaf_rn(a, b, c); }
DA_FD float mul_rn(float a, float b) { return __fmul_rn(a, b); }
DA_FD float sub_rn(float a, float b) { return __fsub_rn(a, b); }
DA_FD uint32_t bits(float f) { return __float_as_uint(f); }
DA_FD float from_bits(uint32_t u) { return __uint_as_float(u); }
DA_FD float d2f_rn(double d) { return __double2float_rn(d); }
DA_FD float rcp_rn(float x) { return __frcp_rn(x); }   // correctly rounded, no FP64 instruction
DA_FD double dsub_rn(double a, double b) { return __dsub_rn(a, b); }
#else   // the host's IEEE operations (the host tests build with -ffp-contract=off)
inline float fma_rn(float a, float b, float c) { return std::fmaf(a, b, c); }
inline float mul_rn(float a, float b) { return a * b; }
inline float sub_rn(float a, float b) { return a - b; }
inline uint32_t bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}
inline float from_bits(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}
inline float d2f_rn(double d) { return (float)d; }
inline float rcp_rn(float x) { return 1.0f / x; }
inline double dsub_rn(double a, double b) { return a - b; }
#endif

struct FpDivisor {
  float hi, lo, r;
};

// false for d outside [2^-60, 2^60] (and NaN): those rows divide exactly
DA_FD bool make_fp_divisor(double d, FpDivisor& F) {
  if (!(d >= 0x1p-60 && d <= 0x1p60)) return false;
  F.hi = d2f_rn(d);
  F.lo = d2f_rn(dsub_rn(d, (double)F.hi));   // d - d_hi is exact (Sterbenz)
  F.r = rcp_rn(F.hi);   // within 2^-24 of 1 / d_hi, as the bound above takes it
  return true;
}

// the certificate: |dl| below h - 2^(E - 39) = h (1 - 2^-15); q1 not a power of two
DA_FD bool certain(uint32_t qb, float dl) {
  const float t = mul_rn(from_bits(qb & 0x7F800000u), 0x1.fffcp-25f);   // 2^E (2^-24 - 2^-39)
  return (bits(dl) & 0x7FFFFFFFu) < bits(t) && (qb & 0x7FFFFFu) != 0u;
}

// bits of RN32(RN64(p / d)) for p in [0.5, 2) when ok; ok = false asks for the exact division
DA_FD uint32_t div_rn32(float p, const FpDivisor& F, bool& ok) {
  const float q0 = mul_rn(p, F.r);
  const float e = fma_rn(q0, -F.hi, p);
  const float e2 = fma_rn(q0, -F.lo, e);
  const float q1 = fma_rn(e2, F.r, q0);
  const float dl = fma_rn(e2, F.r, sub_rn(q0, q1));
  const uint32_t qb = bits(q1);
  ok = certain(qb, dl);
  return qb;
}

}  // namespace fdiv
}  // namespace detattn
