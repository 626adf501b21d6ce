// Correctly rounded division on the integer pipe: RN64(n / d) of two binary64 magnitudes
// and the RN32 of the result, with no FP64 instruction.
//
// GB300 issues FP64 at a small fraction of its integer rate, so a binary64 division costs
// as much as a few hundred integer instructions.  The finalize steps divide many numerators
// by one divisor per row (det-attn "Method": o = RN32(RN64(RN64(NUM) / RN64(DEN))); the
// det-cross-entropy gradient w / denom), so the divisor's reciprocal is computed once per
// row and each quotient takes one 64 x 64 -> 128 multiply plus one exact correction step:
// division by an invariant integer with a precomputed reciprocal (N. Moller and
// T. Granlund, "Improved division by invariant integers", IEEE Trans. Computers 60(2),
// 2011: the 2-by-1 division with the reciprocal v = floor((2^128 - 1) / d) - 2^64 of a
// normalized 64-bit d).  The quotient and remainder are exact, so the roundings that follow
// are exact too.
//
// Everything here also compiles as plain C++ (host tests check it against exact rational
// division), hence the DA_HD qualifier and the portable 128-bit products.
#pragma once
#include <cstdint>

#if defined(__CUDACC__)
#define DA_HD __host__ __device__ __forceinline__
#else
#define DA_HD inline
#endif

namespace detattn {
namespace idiv {

DA_HD uint64_t mul_hi(uint64_t a, uint64_t b) {
#if defined(__CUDA_ARCH__)
  return __umul64hi(a, b);
#else
  return (uint64_t)(((unsigned __int128)a * b) >> 64);
#endif
}

DA_HD int clz64(uint64_t x) {   // x != 0
#if defined(__CUDA_ARCH__)
  return __clzll((long long)x);
#else
  return __builtin_clzll(x);
#endif
}

// v = floor((2^128 - 1) / d) - 2^64 for d >= 2^63.  (2^128 - 1) - 2^64 d = (2^64 - 1 - d) 2^64 +
// (2^64 - 1), whose high word ~d is below d, so the quotient fits 64 bits.  Once per divisor.
DA_HD uint64_t reciprocal(uint64_t d) {
  const unsigned __int128 n = ((unsigned __int128)(~d) << 64) | ~0ull;
  return (uint64_t)(n / d);
}

// q = floor((u1 2^64 + u0) / d), r the remainder, for normalized d (>= 2^63), u1 < d, v its
// reciprocal.  q1 2^64 + q0 = v u1 + (u1 2^64 + u0) estimates the quotient in its high word
// within a small constant below; the remainder test against the low word q0 and one final
// comparison with d correct it.
DA_HD void divrem(uint64_t u1, uint64_t u0, uint64_t d, uint64_t v, uint64_t& q, uint64_t& r) {
  uint64_t q0 = v * u1;
  uint64_t q1 = mul_hi(v, u1);
  const uint64_t s0 = q0 + u0;
  q1 += u1 + (s0 < q0 ? 1u : 0u);
  q0 = s0;
  q1 += 1;
  r = u0 - q1 * d;
  if (r > q0) {
    q1 -= 1;
    r += d;
  }
  if (r >= d) {
    q1 += 1;
    r -= d;
  }
  q = q1;
}

// A divisor m 2^e (m in [2^52, 2^53)) prepared for div_rn64: dn = m 2^11, v its reciprocal.
struct Divisor {
  uint64_t dn, v;
  int e;
};

DA_HD Divisor make_divisor(uint64_t m, int e) {
  Divisor D;
  D.dn = m << 11;
  D.v = reciprocal(D.dn);
  D.e = e;
  return D;
}

// RN64(n / d) for n = mn 2^en, mn in [2^52, 2^53), d the prepared divisor: the result is
// q53 2^E with q53 in [2^52, 2^53).  Q = floor(mn 2^55 / md) = floor(mn 2^66 / dn) has 55
// or 56 bits (mn / md lies in (1/2, 2)); the bits below the 53 kept, and a nonzero
// remainder as sticky, decide the rounding, ties to even.
DA_HD void div_rn64(uint64_t mn, int en, const Divisor& D, uint64_t& q53, int& E) {
  uint64_t Q, r;
  divrem(mn << 2, 0, D.dn, D.v, Q, r);
  const int s = (Q >> 55) ? 3 : 2;
  uint64_t m = Q >> s;
  const uint64_t rb = Q & ((1ull << s) - 1), half = 1ull << (s - 1);
  if (rb > half || (rb == half && (r != 0 || (m & 1)))) m += 1;
  int e = en - D.e - 55 + s;
  if (m >> 53) {
    m >>= 1;
    e += 1;
  }
  q53 = m;
  E = e;
}

// RN32 (bits) of the binary64 value (-1)^neg q53 2^E, q53 in [2^52, 2^53): normal, subnormal,
// zero and overflow to infinity, ties to even.
DA_HD uint32_t rn32_bits(uint64_t q53, int E, bool neg) {
  const uint32_t sign = neg ? 0x80000000u : 0u;
  int x = E + 52;   // the value lies in [2^x, 2^(x+1))
  if (x >= -126) {
    uint64_t m = q53 >> 29;
    const uint64_t rb = q53 & ((1ull << 29) - 1);
    if (rb > (1ull << 28) || (rb == (1ull << 28) && (m & 1))) m += 1;
    if (m >> 24) {
      m >>= 1;
      x += 1;
    }
    if (x > 127) return sign | 0x7F800000u;
    return sign | ((uint32_t)(x + 127) << 23) | (uint32_t)(m & 0x7FFFFFu);
  }
  // subnormal: units of 2^-149
  const int sh = -(E + 149);   // >= 30 here
  if (sh > 54) return sign;     // below half the smallest subnormal
  uint64_t m = q53 >> sh;
  const uint64_t rb = q53 & ((1ull << sh) - 1), half = 1ull << (sh - 1);
  if (rb > half || (rb == half && (m & 1))) m += 1;   // m = 2^23 is the smallest normal's encoding
  return sign | (uint32_t)m;
}

// The binary64 (-1)^neg m 2^e, m in [2^52, 2^53), for a normal-range result.
DA_HD double make_f64(bool neg, uint64_t m, int e) {
  const uint64_t bits = ((uint64_t)neg << 63) | ((uint64_t)(e + 1075) << 52) | (m & 0x000FFFFFFFFFFFFFull);
#if defined(__CUDA_ARCH__)
  return __longlong_as_double((long long)bits);
#else
  double d;
  __builtin_memcpy(&d, &bits, 8);
  return d;
#endif
}

// The binary32-numerator routines below (split_f32_24, div_f32_rn32, div_f32_rn32_direct)
// served the cross-entropy gradient before its quotient moved to the FP32 pipe (fdiv.cuh);
// no kernel calls them now.  They stay as the host tests' exact integer reference for that
// quotient (checked themselves against exact rationals).

// A nonzero binary32 magnitude as mw 2^ew with mw in [2^23, 2^24).
DA_HD void split_f32_24(uint32_t bits, uint32_t& mw, int& ew) {
  const int be = (int)((bits >> 23) & 0xFF);
  if (be) {
    mw = (bits & 0x7FFFFFu) | 0x800000u;
    ew = be - 150;
  } else {   // subnormal
    const uint32_t f = bits & 0x7FFFFFu;
#if defined(__CUDA_ARCH__)
    const int sh = __clz(f) - 8;
#else
    const int sh = __builtin_clz(f) - 8;
#endif
    mw = f << sh;
    ew = -149 - sh;
  }
}

// RN32 bits of RN64(w / d) for w = mw 2^ew (mw in [2^23, 2^24)) and the prepared divisor.
// The same 2-by-1 division as div_rn64 (u1 = mw 2^31, u0 = 0), with v u1 formed from two
// 32 x 32 -> 64 products since mw has 24 bits, then both roundings.
DA_HD uint32_t div_f32_rn32(uint32_t mw, int ew, const Divisor& D) {
  const uint64_t A = (uint64_t)(uint32_t)D.v * mw, B = (D.v >> 32) * (uint64_t)mw;   // each < 2^56
  const uint64_t Plo = A + (B << 32);                                                 // P = v mw, 88 bits
  const uint64_t Phi = (B >> 32) + (Plo < A ? 1u : 0u);
  const uint64_t q0 = Plo << 31;                                                      // (q1, q0) = P 2^31
  uint64_t q1 = (Phi << 31) | (Plo >> 33);
  q1 += ((uint64_t)mw << 31) + 1;                                                     // + u1 2^64, + 2^64
  uint64_t r = 0 - q1 * D.dn;
  if (r > q0) {
    q1 -= 1;
    r += D.dn;
  }
  if (r >= D.dn) {
    q1 += 1;
    r -= D.dn;
  }
  const uint64_t Q = q1;   // floor(mw 2^84 / md): 55 or 56 bits
  const int s = (Q >> 55) ? 3 : 2;
  uint64_t m = Q >> s;
  const uint64_t rb = Q & ((1ull << s) - 1), half = 1ull << (s - 1);
  if (rb > half || (rb == half && (r != 0 || (m & 1)))) m += 1;
  int e = ew - 29 - D.e - 55 + s;
  if (m >> 53) {
    m >>= 1;
    e += 1;
  }
  return rn32_bits(m, e, false);
}

// RN32 bits of RN64(w / d) straight from the reciprocal, for w = mw 2^ew (mw in [2^23, 2^24))
// and the prepared divisor, when that is certain; ok = false asks for div_f32_rn32.
// R = 2^64 + v = floor((2^128 - 1) / dn) lies in (2^128 / dn - 1 - 2^-63, 2^128 / dn), so
// T = mw 2^128 / dn lies in (mw R, mw R + 2^24) and T' = T / 2^32 in (Y, Y + 1.01) with
// Y = floor(mw R / 2^32) = mw 2^32 + mw v_hi + floor(mw v_lo / 2^32) (two 32 x 32 products;
// 56 or 57 bits).  Y's top 32 bits yh (shifted right once when Y has 57 bits, the dropped bit
// going to the top of yl) hold the 24 kept bits, yl the 32 below them; the rounding is
// certain when yl is more than 64 from the half-way point 2^31: neither T''s uncertainty
// (below 2 units of Y) nor the binary64 rounding before it (at most 8 units, which could only
// matter by landing on the half-way point) can then change it.  Subnormal, zero and
// overflowing results also take the exact path.  32-bit operations after the products.
DA_HD uint32_t div_f32_rn32_direct(uint32_t mw, int ew, const Divisor& D, bool& ok) {
  const uint64_t Y = ((uint64_t)mw << 32) + (uint64_t)mw * (uint32_t)(D.v >> 32) +
                     (uint32_t)(((uint64_t)mw * (uint32_t)D.v) >> 32);
  uint32_t yh = (uint32_t)(Y >> 32), yl = (uint32_t)Y;
  int be = ew - D.e + 97;   // biased exponent of yh 2^(ew - D.e - 53) for yh in [2^23, 2^24)
  if (yh >> 24) {
    yl = (yl >> 1) | (yh << 31);
    yh >>= 1;
    be += 1;
  }
  ok = (uint32_t)((int32_t)(yl ^ 0x80000000u) + 64) > 128u && be >= 1 && be <= 253;   // |yl - 2^31| > 64
  const uint32_t M = yh + (yl > 0x80000000u ? 1u : 0u);   // 2^24 carries into the exponent below
  return ((uint32_t)(be - 1) << 23) + M;
}

// RN32 bits of RN64(n / d) straight from the reciprocal, for n = (-1)^neg mn 2^en (mn in
// [2^52, 2^53)) and the prepared divisor, when that is certain; ok = false asks for div_rn64
// and rn32_bits.  T = mn 2^128 / dn lies in (mn R, mn R + mn) with R = 2^64 + v, so T / 2^64
// lies in (H, H + 2) for H = mn + floor(mn v / 2^64) (one 64 x 64 high product), which has 53
// or 54 bits.  The 24 kept bits M and the s = 29 or 30 bits F below them decide the binary32
// rounding unless F is within 64 of the half-way point: the binary64 rounding of the quotient
// moves it by at most one unit of H, T''s uncertainty is below two.  Subnormal and
// overflowing results also take the exact path.
DA_HD uint32_t div_rn64_rn32_direct(uint64_t mn, int en, const Divisor& D, bool neg, bool& ok) {
  const uint64_t H = mn + mul_hi(mn, D.v);
  const int s = (H >> 53) ? 30 : 29;
  const uint64_t M = H >> s, F = H & ((1ull << s) - 1), half = 1ull << (s - 1);
  const int be = s + en - D.e + 97;   // biased exponent of M 2^(s + en - D.e - 53), M in [2^23, 2^24)
  ok = F - half + 64 > 128 && be >= 1 && be <= 253;   // |F - half| > 64 (unsigned wrap below)
  const uint32_t m = (uint32_t)M + (F > half ? 1u : 0u);   // 2^24 carries into the exponent below
  return (neg ? 0x80000000u : 0u) | (((uint32_t)(be - 1) << 23) + m);
}

// RN32 bits of RN64(n / d), n = (-1)^neg mn 2^en: the direct rounding, the exact division when
// that is not certain.
DA_HD uint32_t div_rn32(uint64_t mn, int en, const Divisor& D, bool neg) {
  bool ok;
  const uint32_t r = div_rn64_rn32_direct(mn, en, D, neg, ok);
  if (ok) return r;
  uint64_t q;
  int E;
  div_rn64(mn, en, D, q, E);
  return rn32_bits(q, E, neg);
}

// A binary64's magnitude as m 2^e with m in [2^52, 2^53); false for zero, subnormal,
// infinity or NaN (the callers route those through their slow path).
DA_HD bool split_f64(uint64_t bits, uint64_t& m, int& e) {
  const int be = (int)((bits >> 52) & 0x7FF);
  if (be == 0 || be == 0x7FF) return false;
  m = (bits & 0x000FFFFFFFFFFFFFull) | (1ull << 52);
  e = be - 1075;
  return true;
}

// A nonzero binary32 magnitude (normal or subnormal) as m 2^e with m in [2^52, 2^53).
DA_HD void split_f32_53(uint32_t bits, uint64_t& m, int& e) {
  const int be = (int)((bits >> 23) & 0xFF);
  uint64_t f = bits & 0x7FFFFFu;
  int ee;
  if (be == 0) {
    ee = -149;
  } else {
    f |= 1u << 23;
    ee = be - 150;
  }
  const int sh = clz64(f) - 11;   // top bit to position 52
  m = f << sh;
  e = ee - sh;
}

// RN64 of a Kulisch digit value (radix 2^32, word k weighs 2^(32 k + base)) as a sign and
// m 2^e with m in [2^52, 2^53); false when the value is zero.  Normalizes the words in place.
template <int N>
DA_HD bool digits_split_rn64(long long (&a)[N], int base, bool& neg, uint64_t& m, int& e) {
#pragma unroll
  for (int k = 0; k < N - 1; k++) {
    const long long c = a[k] >> 32;
    a[k] -= c * 4294967296ll;
    a[k + 1] += c;
  }
  neg = a[N - 1] < 0;
  if (neg) {
#pragma unroll
    for (int k = 0; k < N; k++) a[k] = -a[k];
#pragma unroll
    for (int k = 0; k < N - 1; k++) {
      const long long c = a[k] >> 32;
      a[k] -= c * 4294967296ll;
      a[k + 1] += c;
    }
  }
  // the top nonzero word and the two below it, with the OR of everything lower as sticky;
  // static indices only (a select on "k == top" would turn into an indexed local-memory load)
  int top = -1;
  uint64_t w2 = 0, w1 = 0, w0 = 0;
  long long below = 0;
  bool sticky = false;
#pragma unroll
  for (int k = 0; k < N; k++) {
    if (a[k] != 0) {
      top = k;
      w2 = (uint64_t)a[k];   // the top word may exceed 32 bits after the carries
      w1 = k >= 1 ? (uint32_t)a[k >= 1 ? k - 1 : 0] : 0u;
      w0 = k >= 2 ? (uint32_t)a[k >= 2 ? k - 2 : 0] : 0u;
      sticky = below != 0;
    }
    if (k >= 2) below |= a[k >= 2 ? k - 2 : 0];
  }
  if (top < 0) return false;
  // window w2 2^64 + w1 2^32 + w0 with its top bit moved to bit 127; 64 bits kept, sticky below
  const int lz = clz64(w2);
  const unsigned __int128 W = (((unsigned __int128)w2 << 64) | ((unsigned __int128)w1 << 32) | w0) << lz;
  const uint64_t t64 = (uint64_t)(W >> 64);
  if ((uint64_t)W) sticky = true;
  uint64_t mm = t64 >> 11;
  const uint64_t rb = t64 & 0x7FF;
  if (rb > 0x400 || (rb == 0x400 && (sticky || (mm & 1)))) mm += 1;
  int ee = 32 * (top - 2) + base + 64 - lz + 11;
  if (mm >> 53) {
    mm >>= 1;
    ee += 1;
  }
  m = mm;
  e = ee;
  return true;
}

// RN64 of X 2^lsb for a signed 128-bit integer X as a sign and m 2^e with m in [2^52, 2^53)
// (the caller keeps X 2^lsb inside the normal binary64 range); false when X is zero.  The same
// rounding as digits_split_rn64, for a value held in one 128-bit word.
DA_HD bool i128_split_rn64(__int128 X, int lsb, bool& neg, uint64_t& m, int& e) {
  if (X == 0) return false;
  neg = X < 0;
  const unsigned __int128 M = neg ? (unsigned __int128)0 - (unsigned __int128)X : (unsigned __int128)X;
  const uint64_t hi = (uint64_t)(M >> 64), lo = (uint64_t)M;
  const int lz = hi ? clz64(hi) : 64 + clz64(lo);
  const unsigned __int128 W = M << lz;   // top bit at 127
  const uint64_t t64 = (uint64_t)(W >> 64);
  const bool sticky = (uint64_t)W != 0;
  uint64_t mm = t64 >> 11;
  const uint64_t rb = t64 & 0x7FF;
  if (rb > 0x400 || (rb == 0x400 && (sticky || (mm & 1)))) mm += 1;
  int ee = (127 - lz) - 52 + lsb;
  if (mm >> 53) {
    mm >>= 1;
    ee += 1;
  }
  m = mm;
  e = ee;
  return true;
}

}  // namespace idiv
}  // namespace detattn
