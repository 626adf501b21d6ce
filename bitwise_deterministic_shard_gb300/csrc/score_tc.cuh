// Exact scores on the tensor cores (sm_103a, mma.sync bf16 -> f32).
//
// Each Q/K row is first turned into int32 fixed point X_d = x_d 2^-F_row with |X_d| < 2^26
// (the same window as the integer-pipe path; rows that do not fit take the exact
// fallback).  X is then split into four balanced base-128 digits,
//   X = s0 + s1 2^7 + s2 2^14 + s3 2^21,   s_t in [-64, 64],
// each held exactly as a bf16 value.  The exact dot is
//   sum_d Xq_d Xk_d = sum_{c=0..6} 2^(7c) A_c,   A_c = sum_{a+b=c} sum_d sq_a(d) sk_b(d),
// and every A_c is an integer with |A_c| <= 4 * 64 * 64 * D <= 2^22 (D <= 256): all partial
// sums of the bf16 MMA's float32 accumulation are integers below 2^24, so the tensor core
// adds them exactly, in any order.  The 16 slice products per k-step go to 7 diagonal
// accumulators; the int64 dot is recombined in registers and rounded once (cr32_scaled).
#pragma once
#include "numerics.cuh"

namespace detattn {

constexpr int NSLICE = 4, NDIAG = 2 * NSLICE - 1;

// balanced base-128 digits of X (|X| < 2^26) as bf16 bit patterns (exact: |s| <= 64)
__device__ __forceinline__ void slice4(int X, uint16_t (&s)[NSLICE]) {
#pragma unroll
  for (int t = 0; t < NSLICE; t++) {
    int r;
    if (t < NSLICE - 1) {
      r = X & 127;
      if (r >= 64) r -= 128;
      X = (X - r) >> 7;
    } else {
      r = X;   // |r| <= 33 for |X| < 2^26
    }
    s[t] = (uint16_t)(__float_as_uint(small_i2f(r)) >> 16);
  }
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
#if defined(__CUDA_ARCH__)   // (host tests compile this header too; they never call it)
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
#endif
}

// Fragment loads from slice tiles laid out [NSLICE][rows][LDS] (bf16, d contiguous).
// A (16 x 16, row major): rows r0 + g (+8), k = k0 + 2t (+8).  B (16 x 8, col major):
// key n0 + g, k = k0 + 2t (+8).  LDS (elements) must be = 8 (mod 64) so these 32-bit
// loads are free of bank conflicts.
__device__ __forceinline__ void load_a(uint32_t (&a)[4], const uint16_t* S, int LDS, int r0, int k0, int g, int t) {
  const uint16_t* p = S + (r0 + g) * LDS + k0 + 2 * t;
  a[0] = *reinterpret_cast<const uint32_t*>(p);
  a[1] = *reinterpret_cast<const uint32_t*>(p + 8 * LDS);
  a[2] = *reinterpret_cast<const uint32_t*>(p + 8);
  a[3] = *reinterpret_cast<const uint32_t*>(p + 8 * LDS + 8);
}
__device__ __forceinline__ void load_b(uint32_t (&b)[2], const uint16_t* S, int LDS, int n0, int k0, int g, int t) {
  const uint16_t* p = S + (n0 + g) * LDS + k0 + 2 * t;
  b[0] = *reinterpret_cast<const uint32_t*>(p);
  b[1] = *reinterpret_cast<const uint32_t*>(p + 8);
}

// Accumulate the 7 diagonals of one 16 x 8 output tile over k = [0, DP).
// Qs, Ks: slice tiles [NSLICE][rows][LDS]; plane stride = rows * LDS.
template <int DP>
__device__ __forceinline__ void score_tile_mma(float (&acc)[NDIAG][4], const uint16_t* Qs, int qplane, const uint16_t* Ks,
                                               int kplane, int LDS, int r0, int n0, int g, int t) {
#pragma unroll
  for (int c = 0; c < NDIAG; c++)
#pragma unroll
    for (int e = 0; e < 4; e++) acc[c][e] = 0.0f;
#pragma unroll 2
  for (int k0 = 0; k0 < DP; k0 += 16) {
    uint32_t a[NSLICE][4], bb[NSLICE][2];
#pragma unroll
    for (int s = 0; s < NSLICE; s++) {
      load_a(a[s], Qs + s * qplane, LDS, r0, k0, g, t);
      load_b(bb[s], Ks + s * kplane, LDS, n0, k0, g, t);
    }
#pragma unroll
    for (int sa = 0; sa < NSLICE; sa++)
#pragma unroll
      for (int sb = 0; sb < NSLICE; sb++) mma_bf16(acc[sa + sb], a[sa], bb[sb]);
  }
}

// exact int64 dot sum_c 2^(7c) A_c from the 7 diagonal sums of output element e (f32
// integers, |A_c| <= 2^22): v + 1.5 2^23 puts A_c in the low bits of the float's pattern.
// Summed as a shallow tree: pairs A_c + 128 A_(c+1) fit 32 bits, then three exact 64-bit
// multiply-adds
template <int N>
__device__ __forceinline__ long long combine_diag(const float (&acc)[NDIAG][N], int e) {
  int A[NDIAG];
#pragma unroll
  for (int c = 0; c < NDIAG; c++) A[c] = __float_as_int(__fadd_rn(acc[c][e], 12582912.0f)) - 0x4B400000;
  const int s01 = A[0] + A[1] * 128, s23 = A[2] + A[3] * 128, s56 = A[5] + A[6] * 128;   // each below 2^30
  long long lo = (long long)s01, hi = (long long)((unsigned long long)(long long)s56 << 35);
  mad_wide(lo, s23, 1 << 14);   // s01 + 2^14 s23
  mad_wide(hi, A[4], 1 << 28);  // 2^28 A_4 + 2^35 s56
  return lo + hi;
}

// Rows outside the 26-bit window.  Such a row's digit slices hold its truncated part
// X_hi = trunc(x 2^-F); the rest is the low limb X_lo = (x 2^-F - X_hi) 2^26, an integer in
// (-2^26, 2^26) whenever the element has no bit below 2^(F - 26).  In practice few elements
// of a row have a low limb, so up to NLO of them are listed as (d, X_lo); a row with more,
// or with bits below 2^(F - 26), is "deep" and its pairs take the general exact dot.
constexpr int NLO = 4;
constexpr unsigned char LO_DEEP = 0xFF;
constexpr int KLO_DEEP = 15;   // the low-limb field of a deep key row's meta word

// key meta word: window exponent, fit flag, low-limb count (or KLO_DEEP)
__device__ __forceinline__ int kmeta_F(int mv) { return (mv & 0xFFFF) - 1024; }
__device__ __forceinline__ int kmeta_fit(int mv) { return (mv >> 16) & 1; }
__device__ __forceinline__ int kmeta_lon(int mv) { return (mv >> 17) & 15; }

// Convert one row (one warp) to fixed point and hand its four digit slices to
// store(slice, d, bf16 bits) for d in [0, DP) (zeros past D).  F_out / fit_out receive the
// row's window exponent and whether every element fits the 26-bit window.  With lo_out,
// the row's low limbs go to lo_out[0 .. NLO) and *lon_out receives their count (0 for a row
// that fits) or LO_DEEP.
template <int DT, int DP, class Store>
__device__ __forceinline__ void row_slices(const typename In<DT>::T* src, int D, Store store, int* F_out,
                                           unsigned char* fit_out, int& nf, int lane, int2* lo_out = nullptr,
                                           unsigned char* lon_out = nullptr) {
  constexpr int PER = DP / 32;
  uint32_t bv[PER];
  int emax = 1;
#pragma unroll
  for (int t = 0; t < PER; t++) {
    int d = lane + 32 * t;
    uint32_t u = (src != nullptr && d < D) ? In<DT>::bits(src, d) : 0u;
    if (nonfinite_bits(u)) { nf |= ST_NONFINITE; u = 0u; }
    bv[t] = u;
    emax = max(emax, (int)((u >> 23) & 0xFFu));
  }
  emax = __reduce_max_sync(0xFFFFFFFFu, emax);
  const int F = emax - 152;
  bool ok = true, deep = false;
  int nlo = 0;
#pragma unroll
  for (int t = 0; t < PER; t++) {
    Split s = split_f32(bv[t]);
    int sh = s.lsb - F;   // <= 2
    int X = 0, Xl = 0;
    if (s.mant != 0) {
      if (sh >= 0) {
        X = (int)(s.mant << sh);
      } else {
        X = sh > -32 ? (int)(s.mant >> (-sh)) : 0;
        const uint32_t rem = sh > -32 ? (s.mant & ((1u << (-sh)) - 1u)) : s.mant;
        if (rem != 0u) {
          ok = false;
          const int sl = sh + 26;   // the remainder's lsb in units of 2^(F - 26)
          if (sl >= 0)
            Xl = (int)(rem << sl);   // < 2^26
          else if (sl > -32 && (rem & ((1u << (-sl)) - 1u)) == 0u)
            Xl = (int)(rem >> (-sl));
          else
            deep = true;
        }
      }
      if (s.neg) {
        X = -X;
        Xl = -Xl;
      }
    }
    uint16_t sl4[NSLICE];
    slice4(X, sl4);
#pragma unroll
    for (int q = 0; q < NSLICE; q++) store(q, lane + 32 * t, sl4[q]);
    if (lo_out != nullptr) {
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, Xl != 0);
      const int idx = nlo + __popc(bal & ((1u << lane) - 1u));
      if (Xl != 0 && idx < NLO) lo_out[idx] = make_int2(lane + 32 * t, Xl);
      nlo += __popc(bal);
    }
  }
  ok = __all_sync(0xFFFFFFFFu, ok);
  deep = __any_sync(0xFFFFFFFFu, deep) || nlo > NLO;
  if (lane == 0) {
    *F_out = F;
    *fit_out = ok ? 1 : 0;
    if (lon_out != nullptr) *lon_out = ok ? 0 : (deep ? LO_DEEP : (unsigned char)nlo);
  }
}

// truncated 26-bit fixed point of one element, trunc(x 2^-F) (the value its digit slices hold)
__device__ __forceinline__ int hi26(uint32_t u, int F) {
  if (nonfinite_bits(u)) return 0;
  const Split s = split_f32(u);
  const int sh = s.lsb - F;
  const int X = sh >= 0 ? (int)(s.mant << sh) : (sh > -32 ? (int)(s.mant >> (-sh)) : 0);
  return s.neg ? -X : X;
}

// Exact score of a pair with a row outside its window (neither row deep), from the dot of
// the truncated parts T_hh = sum_d Xq_hi Xk_hi (the tensor core's) and the rows' low limbs:
//   x_q . x_k = 2^(Fq + Fk - 52) (T_hh 2^52 + (sum ql Xk_hi + sum Xq_hi kl) 2^26 + sum ql kl),
// the cross sums over the listed elements only.  Rounded once to binary32.
template <int DT>
__device__ __noinline__ float dot_lo(long long Thh, const typename In<DT>::T* qrow, int Fq, const int2* qlo, int nq,
                                        const typename In<DT>::T* krow, int Fk, const int2* klo, int nk) {
  long long cross = 0, ll = 0;
  for (int i = 0; i < nq; i++) {
    const int2 e = qlo[i];
    cross += (long long)e.y * hi26(In<DT>::bits(krow, e.x), Fk);
  }
  for (int i = 0; i < nk; i++) {
    const int2 e = klo[i];
    cross += (long long)hi26(In<DT>::bits(qrow, e.x), Fq) * e.y;
    for (int i2 = 0; i2 < nq; i2++)
      if (qlo[i2].x == e.x) ll += (long long)qlo[i2].y * e.y;
  }
  const __int128 T = (__int128)Thh * ((__int128)1 << 52) + (__int128)cross * (1ll << 26) + (__int128)ll;
  if (T == 0) return 0.0f;
  const int neg = T < 0;
  const unsigned __int128 mag = neg ? (unsigned __int128)(-T) : (unsigned __int128)T;
  return round_f32(mag, false, Fq + Fk - 52, neg);
}

// the same, stored as slice planes dst[q * plane + d]
template <int DT, int DP>
__device__ __forceinline__ void convert_row_slices(const typename In<DT>::T* src, int D, uint16_t* dst, int plane,
                                                   int* F_out, unsigned char* fit_out, int& nf, int lane) {
  row_slices<DT, DP>(src, D, [&](int q, int d, uint16_t v) { dst[q * plane + d] = v; }, F_out, fit_out, nf, lane);
}

}  // namespace detattn
