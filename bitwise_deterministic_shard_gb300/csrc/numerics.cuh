// Device numerics of the order-invariant softmax reduction (sm_103a).
//
// Every floating-point step is an explicit round-to-nearest intrinsic (__fmul_rn,
// __fmaf_rn, __fsub_rn, __ddiv_rn, ...), so nothing is contracted or reassociated by the
// compiler; every sum of products is exact integer arithmetic.  The contract these
// routines implement (page "det-attn", section "Method"; page "det-cross-entropy",
// section "Method"):
//   d_ij = RN32(sum_d q_id k_jd) (exact dot, one rounding), s_ij = RN32(scale32 * d_ij)
//   w_ij = exp32_det(RN32(s_ij - m_i))
//   digits: value = sum_k digit_k 2^(E0 + 32 k), digits 0..n-2 in [0, 2^32), top signed.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace detattn {

constexpr int NUM_NDIG = 15, DEN_NDIG = 6;
constexpr int NUM_E0 = -320, DEN_E0 = -160;
enum : int { ST_NONFINITE = 1, ST_VIOLATION = 2, ST_HEADROOM = 4, ST_BAD_TARGET = 8, ST_TIMEOUT = 16 };

// ---------------------------------------------------------------------------------------
// element access: bf16 is the upper half of a binary32, so widening is exact
// ---------------------------------------------------------------------------------------
template <int DT> struct In;
template <> struct In<0> {
  using T = float;
  __device__ __forceinline__ static uint32_t bits(const T* p, int64_t i) { return __float_as_uint(__ldg(p + i)); }
};
template <> struct In<1> {
  using T = uint16_t;
  __device__ __forceinline__ static uint32_t bits(const T* p, int64_t i) { return (uint32_t)__ldg(p + i) << 16; }
};

// binary32 bits -> |x| = mant * 2^lsb (mant < 2^24), sign
struct Split {
  uint32_t mant;
  int lsb;
  int neg;
};
__device__ __forceinline__ Split split_f32(uint32_t u) {
  Split s;
  uint32_t ex = (u >> 23) & 0xFFu, fr = u & 0x7FFFFFu;
  s.neg = (int)(u >> 31);
  s.mant = ex ? (fr | 0x800000u) : fr;
  s.lsb = (ex ? (int)ex : 1) - 150;
  return s;
}
__device__ __forceinline__ bool nonfinite_bits(uint32_t u) { return ((u >> 23) & 0xFFu) == 0xFFu; }
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xFF800000); }

// ---------------------------------------------------------------------------------------
// exp32_det: Cody-Waite argument reduction (Cody & Waite, "Software Manual for the
// Elementary Functions", 1980) and a degree-7 Taylor polynomial, every step one binary32
// rounding.  Constants: RN32(log2 e); ln 2 to 16 significant bits; RN32(ln 2 - that);
// RN32(1/n!) for n = 0..7.  Valid for x <= 0 (callers clamp); x < -104 gives +0.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float exp32_det(float x) {
  if (x != x) return x;
  if (x < -104.0f) return 0.0f;
  const float L2E = 0x1.715476p+0f, C1 = 0x1.62e4p-1f, C2 = 0x1.7f7d1cp-20f, MAGIC = 12582912.0f;  // 1.5 * 2^23
  float t = __fmul_rn(x, L2E);
  // k = rint(t), ties to even: |t| <= 151, so t + 1.5 * 2^23 rounds t to an integer exactly
  float tr = __fadd_rn(t, MAGIC);
  int k = __float_as_int(tr) - 0x4B400000;
  float kf = __fsub_rn(tr, MAGIC);    // exact
  float r1 = __fmaf_rn(-kf, C1, x);   // exact (Cody-Waite)
  float r = __fmaf_rn(-kf, C2, r1);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  // RN32(p * 2^k) in one rounding: an exact normal pre-scale, then one multiply
  if (k >= -126) return __fmul_rn(p, __uint_as_float((uint32_t)(k + 127) << 23));
  return __fmul_rn(__fmul_rn(p, __uint_as_float((uint32_t)(k + 64 + 127) << 23)), 0x1p-64f);
}

// exp32_det without branches, for x <= 0 or x = -inf (not NaN): the same operations in the
// same order as exp32_det, the special cases taken by selects, so the caller's independent
// evaluations can interleave.
__device__ __forceinline__ float exp32_det_poly(float xx, int& k);
__device__ __forceinline__ float exp32_det_nb(float x) {
  const bool under = x < -104.0f;
  const float xx = under ? 0.0f : x;
  int k;
  const float p = exp32_det_poly(xx, k);
  const bool sub = k < -126;
  const float res = __fmul_rn(p, __uint_as_float((uint32_t)(k + (sub ? 64 : 0) + 127) << 23));
  const float out = sub ? __fmul_rn(res, 0x1p-64f) : res;
  return under ? 0.0f : out;
}

// exp32_det's reduction and polynomial for -104 <= xx <= 0: returns p and k with
// exp32_det(xx) = RN32(p 2^k).  p lies in (0.7, 1.5), so for k >= -125 the product is a
// normal binary32 and exp32_det(xx) is p 2^k exactly (p's mantissa, p's exponent + k).
__device__ __forceinline__ float exp32_det_poly(float xx, int& k) {
  const float L2E = 0x1.715476p+0f, C1 = 0x1.62e4p-1f, C2 = 0x1.7f7d1cp-20f, MAGIC = 12582912.0f;
  const float t = __fmul_rn(xx, L2E);
  const float tr = __fadd_rn(t, MAGIC);
  k = __float_as_int(tr) - 0x4B400000;
  const float kf = __fsub_rn(tr, MAGIC);
  const float r1 = __fmaf_rn(-kf, C1, xx);
  const float r = __fmaf_rn(-kf, C2, r1);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return p;
}

// exact small-integer <-> binary32 conversions on the FP32/integer pipes (|v| <= 2^22)
__device__ __forceinline__ int small_f2i(float f) { return __float_as_int(__fadd_rn(f, 12582912.0f)) - 0x4B400000; }
__device__ __forceinline__ float small_i2f(int v) { return __fsub_rn(__int_as_float(0x4B400000 + v), 12582912.0f); }

// ---------------------------------------------------------------------------------------
// Round an exact value to binary32 (ties to even, gradual underflow, overflow -> inf).
// The value is (neg ? -1 : 1) * (W + t) * 2^lsb with W a 128-bit magnitude and t in
// [0, 1) nonzero iff `sticky`.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float round_f32(unsigned __int128 W, bool sticky, int lsb, int neg) {
  if (W == 0) return neg ? -0.0f : 0.0f;   // callers only pass sticky with W == 0 when the value underflows
  uint64_t hi = (uint64_t)(W >> 64), lo = (uint64_t)W;
  int tb = hi ? 127 - __clzll((long long)hi) : 63 - __clzll((long long)lo);  // top bit index
  int e = tb + lsb;                        // 2^e <= |value| < 2^(e+1)
  int q = (e > -126 ? e : -126) - 23;      // exponent of the last kept bit
  int cut = q - lsb;                       // bit index in W of the last kept bit
  uint64_t n;
  bool rb, st = sticky;
  if (cut <= 0) {
    n = (uint64_t)W << (-cut);             // exact (W < 2^24 here)
    rb = false;
  } else {
    int rpos = cut - 1;                    // index of the rounding bit
    n = cut >= 128 ? 0 : (uint64_t)(W >> cut);
    rb = rpos >= 128 ? false : (bool)((W >> rpos) & 1);
    unsigned __int128 below = rpos >= 128 ? W : (W & ((((unsigned __int128)1) << rpos) - 1));
    st = st || (below != 0);
  }
  if (rb && (st || (n & 1))) n++;
  uint32_t bitsv;
  if (n == 0) {
    bitsv = 0;
  } else if (n < 0x800000u) {              // subnormal (q == -149)
    bitsv = (uint32_t)n;
  } else {
    if (n == 0x1000000u) { n = 0x800000u; q++; }
    int be = q + 150;
    bitsv = be >= 255 ? 0x7F800000u : (((uint32_t)be << 23) | ((uint32_t)n & 0x7FFFFFu));
  }
  return __uint_as_float(bitsv | (neg ? 0x80000000u : 0u));
}

// RN32(T * 2^F) for an integer T, |T| < 2^63: integer operations only (the 64-bit
// integer -> float conversion runs on the slow FP64 path of this GPU).
__device__ __forceinline__ float cr32_scaled(long long T, int F) {
  if (T == 0) return 0.0f;
  const int neg = T < 0;
  const unsigned long long mag = neg ? 0ull - (unsigned long long)T : (unsigned long long)T;
  const int tb = 63 - __clzll((long long)mag);   // top bit index
  const int e = tb + F;                           // 2^e <= |value| < 2^(e+1)
  int q = (e > -126 ? e : -126) - 23;             // exponent of the last kept bit
  const int sh = q - F;                           // low bits of mag to drop
  unsigned long long n;
  if (sh <= 0) {
    n = mag << (-sh);                             // exact, n < 2^24
  } else if (sh >= 64) {
    n = 0;                                        // below half the smallest subnormal
  } else {
    n = mag >> sh;
    const unsigned long long rem = mag & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (n & 1ull))) n++;
  }
  uint32_t bitsv;
  if (n < 0x800000ull) {
    bitsv = (uint32_t)n;                          // subnormal or zero (q == -149)
  } else {
    if (n == 0x1000000ull) { n = 0x800000ull; q++; }
    const int be = q + 150;
    bitsv = be >= 255 ? 0x7F800000u : (((uint32_t)be << 23) | ((uint32_t)n & 0x7FFFFFu));
  }
  return __uint_as_float(bitsv | (neg ? 0x80000000u : 0u));
}

// cr32_scaled without branches for results in the normal binary32 range: the top 24 bits of
// |T| rounded to nearest-even on the round bit and the sticky bits below it.  *special is set
// (and the result is meaningless) when T 2^F is nonzero and subnormal or beyond the largest
// exponent; the caller then takes cr32_scaled.
__device__ __forceinline__ float cr32_scaled_nb(long long T, int F, bool& special) {
  const bool neg = T < 0;
  const unsigned long long mag = neg ? 0ull - (unsigned long long)T : (unsigned long long)T;
  const int lz = __clzll((long long)mag);   // 64 for T == 0
  const int e = 63 - lz + F;                // 2^e <= |value| < 2^(e+1)
  special = mag != 0ull && (e < -126 || e > 127);
  const unsigned long long nrm = mag << (lz & 63);
  const uint32_t hi = (uint32_t)(nrm >> 32), lo = (uint32_t)nrm;
  uint32_t m = hi >> 8;   // 24 bits
  const uint32_t rb = (hi >> 7) & 1u, st = ((hi & 0x7Fu) | lo) != 0u ? 1u : 0u;
  m += rb & (st | (m & 1u));
  const uint32_t carry = m >> 24;   // rounded up to 2^24
  const uint32_t bitsv = ((uint32_t)(e + 127 + (int)carry) << 23) | ((m >> carry) & 0x7FFFFFu) | (neg ? 0x80000000u : 0u);
  return mag == 0ull ? 0.0f : __uint_as_float(bitsv);
}

// cr32_scaled_nb through the hardware's correctly rounded 64-bit integer -> binary32
// conversion (cvt.rn.f32.s64, issued on the FP64 pipe, which the score kernels otherwise leave
// idle): RN32(T) times 2^F, exact when that product is a normal binary32, so equal to
// RN32(T 2^F) there (rounding to 24 bits commutes with an exact power-of-two scale; a value
// whose 24-bit rounding reaches 2^-126 also rounds to 2^-126 on the subnormal grid).
// *special is set when T is nonzero and the scaled result is not normal, or F lies outside
// [-126, 127]; the caller then takes cr32_scaled.
__device__ __forceinline__ float cr32_scaled_cvt(long long T, int F, bool& special) {
  const float f = __ll2float_rn(T);
  const int be = (int)((__float_as_uint(f) >> 23) & 0xFFu) + F;
  special = T != 0 && (be < 1 || be > 254 || F < -126 || F > 127);
  return __fmul_rn(f, __uint_as_float((uint32_t)(min(max(F, -126), 127) + 127) << 23));
}

// ---------------------------------------------------------------------------------------
// Kulisch accumulator in radix 2^32 (int64 words with lazy carries); word k weighs
// 2^(32k - 320).  Used by the exact fallback dot and by digit conversions.
// ---------------------------------------------------------------------------------------
constexpr int KW = 20;

__device__ __forceinline__ void kul_add(long long* a, unsigned long long mag, int neg, int lsb) {
  if (mag == 0) return;
  int pos = lsb + 320;
  int k = pos >> 5, sh = pos & 31;
  unsigned long long lo = mag << sh;
  unsigned long long hi = sh ? (mag >> (64 - sh)) : 0ull;
  long long c0 = (long long)(lo & 0xFFFFFFFFull), c1 = (long long)(lo >> 32), c2 = (long long)hi;
  if (neg) { a[k] -= c0; a[k + 1] -= c1; a[k + 2] -= c2; }
  else     { a[k] += c0; a[k + 1] += c1; a[k + 2] += c2; }
}

__device__ __forceinline__ void kul_carry(long long* a, int n) {
  for (int k = 0; k < n - 1; k++) {
    long long c = a[k] >> 32;
    a[k] -= c * 4294967296ll;
    a[k + 1] += c;
  }
}

// RN32 of a Kulisch value (words weigh 2^(32k + base))
static __device__ __noinline__ float kul_round_f32(long long* a, int n, int base) {
  kul_carry(a, n);
  int neg = a[n - 1] < 0;
  if (neg) {
    for (int k = 0; k < n; k++) a[k] = -a[k];
    kul_carry(a, n);
  }
  int top = -1;
  for (int k = n - 1; k >= 0; k--)
    if (a[k] != 0) { top = k; break; }
  if (top < 0) return 0.0f;
  unsigned __int128 W = 0;
  bool sticky = false;
  int lo = top - 2;
  for (int k = top; k >= lo; k--) W = (W << 32) | (unsigned long long)(k >= 0 ? (uint32_t)a[k] : 0u);
  for (int k = 0; k < lo; k++) sticky = sticky || (a[k] != 0);
  return round_f32(W, sticky, 32 * lo + base, neg);
}

// Exact fallback score: d = RN32(sum_d q_d k_d) from the raw inputs, any finite values.
template <int DT>
__device__ float exact_dot_slow(const typename In<DT>::T* q, const typename In<DT>::T* k, int D) {
  long long a[KW];
#pragma unroll
  for (int t = 0; t < KW; t++) a[t] = 0;
  for (int d = 0; d < D; d++) {
    uint32_t qb = In<DT>::bits(q, d), kb = In<DT>::bits(k, d);
    if (nonfinite_bits(qb) || nonfinite_bits(kb)) continue;
    Split sq = split_f32(qb), sk = split_f32(kb);
    kul_add(a, (unsigned long long)sq.mant * sk.mant, sq.neg ^ sk.neg, sq.lsb + sk.lsb);
  }
  return kul_round_f32(a, KW, -320);
}

// ---------------------------------------------------------------------------------------
// Exact score of one pair by one warp, for rows outside the 26-bit fixed-point window:
// each row is taken as a 52-bit fixed point X = x 2^-Flo (Flo = row max exponent - 178),
// split in two signed 26-bit limbs; lanes split D, the four limb-product sums are exact
// int64s reduced across the warp, and the 128-bit total is rounded once.  A row whose
// elements span even more than the 52-bit window takes the Kulisch fallback.  Every lane
// returns the same value.
// ---------------------------------------------------------------------------------------
template <int DT>
__device__ float exact_dot_warp(const typename In<DT>::T* q, const typename In<DT>::T* k, int D, int lane) {
  int eq = 1, ek = 1;
  for (int d = lane; d < D; d += 32) {
    const uint32_t a = In<DT>::bits(q, d), b = In<DT>::bits(k, d);
    if (!nonfinite_bits(a)) eq = max(eq, (int)((a >> 23) & 0xFFu));
    if (!nonfinite_bits(b)) ek = max(ek, (int)((b >> 23) & 0xFFu));
  }
  eq = __reduce_max_sync(0xFFFFFFFFu, eq);
  ek = __reduce_max_sync(0xFFFFFFFFu, ek);
  const int Fq = eq - 178, Fk = ek - 178;   // |X| < 2^52
  long long shh = 0, shl = 0, slh = 0, sll = 0;
  bool ok = true;
  for (int d = lane; d < D; d += 32) {
    uint32_t a = In<DT>::bits(q, d), b = In<DT>::bits(k, d);
    if (nonfinite_bits(a)) a = 0u;
    if (nonfinite_bits(b)) b = 0u;
    long long X[2];
    const uint32_t uu[2] = {a, b};
    const int FF[2] = {Fq, Fk};
#pragma unroll
    for (int z = 0; z < 2; z++) {
      const Split s = split_f32(uu[z]);
      const int sh = s.lsb - FF[z];   // <= 28
      long long v = 0;
      if (s.mant) {
        if (sh >= 0) {
          v = (long long)s.mant << sh;
        } else if (sh > -32) {
          v = (long long)(s.mant >> (-sh));
          ok = ok && ((s.mant & ((1u << (-sh)) - 1u)) == 0u);
        } else {
          ok = false;
        }
        if (s.neg) v = -v;
      }
      X[z] = v;
    }
    const long long qh = X[0] >> 26, ql = X[0] - qh * (1ll << 26);   // ql in [0, 2^26)
    const long long kh = X[1] >> 26, kl = X[1] - kh * (1ll << 26);
    shh += qh * kh;
    shl += qh * kl;
    slh += ql * kh;
    sll += ql * kl;
  }
  if (!__all_sync(0xFFFFFFFFu, ok)) return exact_dot_slow<DT>(q, k, D);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    shh += __shfl_xor_sync(0xFFFFFFFFu, shh, o);
    shl += __shfl_xor_sync(0xFFFFFFFFu, shl, o);
    slh += __shfl_xor_sync(0xFFFFFFFFu, slh, o);
    sll += __shfl_xor_sync(0xFFFFFFFFu, sll, o);
  }
  const __int128 T = (__int128)shh * ((__int128)1 << 52) + (__int128)(shl + slh) * (1ll << 26) + (__int128)sll;
  if (T == 0) return 0.0f;
  const int neg = T < 0;
  const unsigned __int128 mag = neg ? (unsigned __int128)(-T) : (unsigned __int128)T;
  return round_f32(mag, false, Fq + Fk, neg);
}

// ---------------------------------------------------------------------------------------
// Exact score of one pair by one thread, for a pair with a row outside its 26-bit window.
// Both rows are read as 52-bit fixed point X = x 2^-(F - 26), F the row's 26-bit window
// exponent (|X| < 2^52), and X is split into a signed high limb X >> 26 and a low limb in
// [0, 2^26), exactly as the warp version above; the four limb-product sums are exact int64s
// and the 128-bit total is rounded once.  A row that fits its 26-bit window has zero low
// limbs, so QLO / KLO false drops the products that would vanish.  An element below the
// 52-bit window sends the pair to the Kulisch fallback.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ bool limbs52(uint32_t u, int Flo, int& h, int& l) {
  h = 0;
  l = 0;
  if (nonfinite_bits(u)) return true;   // counted where the row was converted; it adds nothing
  const Split s = split_f32(u);
  if (s.mant == 0u) return true;
  const int sh = s.lsb - Flo;   // <= 28
  long long X;
  bool ok = true;
  if (sh >= 0) {
    X = (long long)((unsigned long long)s.mant << sh);
  } else if (sh > -32) {
    X = (long long)(s.mant >> (-sh));
    ok = (s.mant & ((1u << (-sh)) - 1u)) == 0u;
  } else {
    X = 0;
    ok = false;
  }
  if (s.neg) X = -X;
  h = (int)(X >> 26);
  l = (int)(X & 0x3FFFFFFll);
  return ok;
}

template <int DT, bool QLO, bool KLO>
__device__ __noinline__ float exact_dot_lane(const typename In<DT>::T* q, int Fq, const typename In<DT>::T* k, int Fk,
                                             int D) {
  long long shh = 0, shl = 0, slh = 0, sll = 0;
  bool ok = true;
  constexpr int U = 16;   // elements loaded before any is used: the loads overlap
  for (int d0 = 0; d0 < D; d0 += U) {
    uint32_t qb[U], kb[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
      qb[u] = d0 + u < D ? In<DT>::bits(q, d0 + u) : 0u;
      kb[u] = d0 + u < D ? In<DT>::bits(k, d0 + u) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      int qh, ql, kh, kl;
      ok &= limbs52(qb[u], Fq - 26, qh, ql);
      ok &= limbs52(kb[u], Fk - 26, kh, kl);
      shh += (long long)qh * kh;
      if (KLO) shl += (long long)qh * kl;
      if (QLO) slh += (long long)ql * kh;
      if (QLO && KLO) sll += (long long)ql * kl;
    }
  }
  if (!ok) return exact_dot_slow<DT>(q, k, D);
  const __int128 T = (__int128)shh * ((__int128)1 << 52) + (__int128)(shl + slh) * (1ll << 26) + (__int128)sll;
  if (T == 0) return 0.0f;
  const int neg = T < 0;
  const unsigned __int128 mag = neg ? (unsigned __int128)(-T) : (unsigned __int128)T;
  return round_f32(mag, false, Fq + Fk - 52, neg);
}

// ---------------------------------------------------------------------------------------
// Round a digit array (radix 2^32 int64, word k weighs 2^(32k + base), any carries) to
// binary64, ties to even.  Values here lie in [2^-320, 2^192): normal binary64 range.
// ---------------------------------------------------------------------------------------
template <int N>
__device__ __forceinline__ double digits_rn64(long long (&a)[N], int base) {
  kul_carry(a, N);
  int neg = a[N - 1] < 0;
  if (neg) {
#pragma unroll
    for (int k = 0; k < N; k++) a[k] = -a[k];
    kul_carry(a, N);
  }
  int top = -1;
#pragma unroll
  for (int k = 0; k < N; k++)
    if (a[k] != 0) top = k;
  if (top < 0) return 0.0;
  // 96-bit window from the top word, sticky for everything below
  unsigned long long w2 = (uint32_t)a[top];
  unsigned long long w1 = top >= 1 ? (uint32_t)a[top - 1] : 0u;
  unsigned long long w0 = top >= 2 ? (uint32_t)a[top - 2] : 0u;
  bool sticky = false;
#pragma unroll
  for (int k = 0; k < N; k++)
    if (k < top - 2 && a[k] != 0) sticky = true;
  int lz = __clzll((long long)w2) - 32;            // leading zeros of the 32-bit top word
  unsigned __int128 W = ((unsigned __int128)w2 << 64) | ((unsigned __int128)w1 << 32) | w0;
  W <<= lz;                                         // top bit now at bit 95
  unsigned long long top64 = (unsigned long long)(W >> 32);
  if ((uint32_t)W != 0) sticky = true;
  if (sticky) top64 |= 1ull;                        // below the rounding position (bit 10)
  double r = __ull2double_rn(top64);                // one rounding to 53 bits
  int e = 32 * (top - 2) + base + 32 - lz;          // weight of top64's bit 0
  // exact scaling by 2^e (result stays normal)
  int e1 = e / 2, e2 = e - e1;
  r = __dmul_rn(r, __longlong_as_double((long long)(e1 + 1023) << 52));
  r = __dmul_rn(r, __longlong_as_double((long long)(e2 + 1023) << 52));
  return neg ? -r : r;
}

// ---------------------------------------------------------------------------------------
// log64_det: reduction to [sqrt(1/2), sqrt(2)], the atanh series log f = 2 sum
// u^(2n+1)/(2n+1), u = (f-1)/(f+1), ten terms after the first, then + e ln 2 in two parts.
// binary64, every operation one rounding, nothing fused.  For positive finite normal d.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ double log64_det(double d) {
  long long b = __double_as_longlong(d);
  int e = (int)((b >> 52) & 0x7FF) - 1023;
  double f = __longlong_as_double((b & 0x000FFFFFFFFFFFFFll) | 0x3FF0000000000000ll);  // [1, 2)
  if (f > 0x1.6a09e667f3bcdp+0) { f = __dmul_rn(f, 0.5); e += 1; }
  double a = __dsub_rn(f, 1.0);
  double bb = __dadd_rn(f, 1.0);
  double u = __ddiv_rn(a, bb);
  double u2 = __dmul_rn(u, u);
  double p = __ddiv_rn(1.0, 21.0);
#pragma unroll
  for (int n = 9; n >= 1; n--) p = __dadd_rn(__dmul_rn(p, u2), __ddiv_rn(1.0, (double)(2 * n + 1)));
  double t1 = __dmul_rn(u2, p);
  double t2 = __dmul_rn(u, t1);
  double lf = __dmul_rn(__dadd_rn(u, t2), 2.0);
  double fe = (double)e;
  double hi = __dmul_rn(fe, 0x1.62e42fefa38p-1);
  double lo = __dmul_rn(fe, 0x1.ef35793c7673p-45);
  return __dadd_rn(hi, __dadd_rn(lo, lf));
}

// ---------------------------------------------------------------------------------------
// exact atomic digit adds (integer adds commute, so concurrent adds stay deterministic)
// ---------------------------------------------------------------------------------------
// add (neg ? -1 : 1) * mag * 2^lsb, mag < 2^49, into digits whose word k weighs
// 2^(32k + e0), word stride `stride` (elements)
__device__ __forceinline__ void atomic_digits_add(long long* dg, int64_t stride, int e0, unsigned long long mag, int neg,
                                                  int lsb) {
  if (mag == 0) return;
  int pos = lsb - e0;
  int k = pos >> 5, sh = pos & 31;
  unsigned long long lo = mag << sh;
  unsigned long long hi = sh ? (mag >> (64 - sh)) : 0ull;
  unsigned long long c[3] = {lo & 0xFFFFFFFFull, lo >> 32, hi};
#pragma unroll
  for (int t = 0; t < 3; t++)
    if (c[t]) atomicAdd((unsigned long long*)(dg + (int64_t)(k + t) * stride), neg ? (0ull - c[t]) : c[t]);
}

// acc += a * b exactly: one 32x32 -> 64-bit signed multiply-add (mad.wide.s32)
// (The #else branches let host tests compile this header with a host C++ compiler; device
// code always takes the PTX.)
__device__ __forceinline__ void mad_wide(long long& acc, int a, int b) {
#if defined(__CUDA_ARCH__)
  asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc) : "r"(a), "r"(b));
#else
  acc += (long long)a * b;
#endif
}

// 16-byte asynchronous global -> shared copy (zero-filled when src_bytes == 0)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
#if defined(__CUDA_ARCH__)
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem), "r"(src_bytes));
#else
  for (int b = 0; b < 16; b++) ((unsigned char*)smem)[b] = b < src_bytes ? ((const unsigned char*)gmem)[b] : 0;
#endif
}
__device__ __forceinline__ void cp_async_wait_all() {
#if defined(__CUDA_ARCH__)
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
#endif
}

// order-preserving int key of a binary32 (not NaN): key(a) < key(b) iff a < b, with -0 < +0
__device__ __forceinline__ int float_key(float f) {
  const int b = __float_as_int(f);
  return b >= 0 ? b : (b ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float key_float(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7FFFFFFF)); }

__device__ __forceinline__ void report(int* status, int bits) {
  if (bits && status) atomicOr(status, bits);
}

}  // namespace detattn
