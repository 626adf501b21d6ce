// Exact accumulation of binary32 weights 0 <= w <= 1 into the six radix-2^32 DEN digits
// (word k weighs 2^(32 k - 160)), for the cross-entropy denominator (page "det-cross-entropy",
// section "Method": den_i = sum_v exp(x_iv - m_i) summed exactly in a long accumulator).
//
// A weight w >= 2^-31 is M 2^(e - 150) with a 24-bit M and biased exponent e >= 96, so
// w 2^54 = M 2^(e - 96) is an integer below 2^55: it is added to one private 64-bit word U
// (one shift and one 64-bit add), which is moved into the digits before it can overflow.
// Smaller weights (w < 2^-31, rare: a logit more than 21 below the row maximum) are placed
// into their two digit words directly.  Both routes are exact, so the digits are the exact
// sum in any order.  Also compiles as plain C++ for the host tests.
#pragma once
#include <cstdint>

#ifndef DA_HD
#if defined(__CUDACC__)
#define DA_HD __host__ __device__ __forceinline__
#else
#define DA_HD inline
#endif
#endif

namespace detattn {

struct DenAcc {
  uint64_t U;        // sum of w 2^54 over the weights w >= 2^-31 since the last flush
  long long d[6];    // digits, word k weighs 2^(32 k - 160)
};

DA_HD void den_init(DenAcc& A) {
  A.U = 0;
#pragma unroll
  for (int k = 0; k < 6; k++) A.d[k] = 0;
}

// U 2^-54 into the digits: 2^-54 is 2^10 units of word 3 (2^-64)
DA_HD void den_flush(DenAcc& A) {
  const uint64_t lo = A.U << 10, hi = A.U >> 54;
  A.d[3] += (long long)(lo & 0xFFFFFFFFull);
  A.d[4] += (long long)(lo >> 32);
  A.d[5] += (long long)hi;
  A.U = 0;
}

// keep U below 2^62 before a group of at most 128 adds (each is below 2^55)
DA_HD void den_guard(DenAcc& A) {
  if (A.U >> 62) den_flush(A);
}

// add the weight with bits wb (0 <= w <= 1, finite); at most 128 adds between den_guard calls
DA_HD void den_add(DenAcc& A, uint32_t wb) {
  const int ex = (int)(wb >> 23);
  if (ex >= 96) {
    A.U += (uint64_t)((wb & 0x7FFFFFu) | 0x800000u) << (ex - 96);
    return;
  }
  if (wb == 0u) return;
  const uint32_t M = ex ? ((wb & 0x7FFFFFu) | 0x800000u) : wb;
  const int pos = (ex ? ex : 1) + 10;   // bit position of M's unit above 2^-160
  const int k = pos >> 5;               // 0 .. 3 here
  const unsigned long long ch = (unsigned long long)M << (pos & 31);
  const long long c0 = (long long)(ch & 0xFFFFFFFFull), c1 = (long long)(ch >> 32);
  if (k == 0) {
    A.d[0] += c0;
    A.d[1] += c1;
  } else if (k == 1) {
    A.d[1] += c0;
    A.d[2] += c1;
  } else if (k == 2) {
    A.d[2] += c0;
    A.d[3] += c1;
  } else {
    A.d[3] += c0;
    A.d[4] += c1;
  }
}

}  // namespace detattn
