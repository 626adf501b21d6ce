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
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
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
// integers, |A_c| <= 2^22): v + 1.5 2^23 puts A_c in the low bits of the float's pattern,
// and the patterns' common offset is folded into one constant (arithmetic mod 2^64)
template <int N>
__device__ __forceinline__ long long combine_diag(const float (&acc)[NDIAG][N], int e) {
  int raw[NDIAG];
#pragma unroll
  for (int c = 0; c < NDIAG; c++) raw[c] = __float_as_int(__fadd_rn(acc[c][e], 12582912.0f));
  const int hi = (raw[5] - 0x4B400000) + (raw[6] - 0x4B400000) * 128;   // |hi| < 2^30
  long long T = (long long)((unsigned long long)(long long)hi << 35);
#pragma unroll
  for (int c = 0; c < 5; c++) mad_wide(T, raw[c], 1 << (7 * c));
  return (long long)((unsigned long long)T - 0x4B400000ull * 0x10204081ull);
}

// Convert one row (one warp) to fixed point and hand its four digit slices to
// store(slice, d, bf16 bits) for d in [0, DP) (zeros past D).  F_out / fit_out receive the
// row's window exponent and whether every element fits the 26-bit window.
template <int DT, int DP, class Store>
__device__ __forceinline__ void row_slices(const typename In<DT>::T* src, int D, Store store, int* F_out,
                                           unsigned char* fit_out, int& nf, int lane) {
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
  bool ok = true;
#pragma unroll
  for (int t = 0; t < PER; t++) {
    Split s = split_f32(bv[t]);
    int sh = s.lsb - F;   // <= 2
    int X = 0;
    if (s.mant != 0) {
      if (sh >= 0) {
        X = (int)(s.mant << sh);
      } else if (sh > -32) {
        X = (int)(s.mant >> (-sh));
        ok = ok && ((s.mant & ((1u << (-sh)) - 1u)) == 0u);
      } else {
        ok = false;
      }
      if (s.neg) X = -X;
    }
    uint16_t sl[NSLICE];
    slice4(X, sl);
#pragma unroll
    for (int q = 0; q < NSLICE; q++) store(q, lane + 32 * t, sl[q]);
  }
  ok = __all_sync(0xFFFFFFFFu, ok);
  if (lane == 0) {
    *F_out = F;
    *fit_out = ok ? 1 : 0;
  }
}

// the same, stored as slice planes dst[q * plane + d]
template <int DT, int DP>
__device__ __forceinline__ void convert_row_slices(const typename In<DT>::T* src, int D, uint16_t* dst, int plane,
                                                   int* F_out, unsigned char* fit_out, int& nf, int lane) {
  row_slices<DT, DP>(src, D, [&](int q, int d, uint16_t v) { dst[q * plane + d] = v; }, F_out, fit_out, nf, lane);
}

}  // namespace detattn
