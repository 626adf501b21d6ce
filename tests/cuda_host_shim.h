// Host stand-ins for the CUDA device intrinsics that the numerics headers use, so that those
// headers compile with a host C++ compiler for the host tests.  Each round-to-nearest
// binary32 / binary64 intrinsic is the host's IEEE operation in the default rounding mode
// (the drivers build with -ffp-contract=off, so nothing is fused unless fmaf is written);
// bit casts are memcpy.  Atomics and warp collectives are single-thread stand-ins: the host
// tests call no routine that needs more than one lane.
#pragma once
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#ifndef __noinline__
#define __noinline__ __attribute__((noinline))
#endif
inline int max(int a, int b) { return a > b ? a : b; }
inline int min(int a, int b) { return a < b ? a : b; }

template <class To, class From>
inline To da_bitcast(From f) {
  To t;
  std::memcpy(&t, &f, sizeof t);
  return t;
}
inline float __fmaf_rn(float a, float b, float c) { return std::fmaf(a, b, c); }
inline float __fmul_rn(float a, float b) { return a * b; }
inline float __fadd_rn(float a, float b) { return a + b; }
inline float __fsub_rn(float a, float b) { return a - b; }
inline double __dmul_rn(double a, double b) { return a * b; }
inline double __dadd_rn(double a, double b) { return a + b; }
inline double __dsub_rn(double a, double b) { return a - b; }
inline double __ddiv_rn(double a, double b) { return a / b; }
inline double __ull2double_rn(unsigned long long x) { return (double)x; }
inline float __ll2float_rn(long long x) { return (float)x; }   // IEEE conversion, round to nearest even
inline float __double2float_rn(double x) { return (float)x; }
inline float __uint_as_float(uint32_t u) { return da_bitcast<float>(u); }
inline uint32_t __float_as_uint(float f) { return da_bitcast<uint32_t>(f); }
inline int __float_as_int(float f) { return da_bitcast<int>(f); }
inline float __int_as_float(int i) { return da_bitcast<float>(i); }
inline double __longlong_as_double(long long i) { return da_bitcast<double>(i); }
inline long long __double_as_longlong(double d) { return da_bitcast<long long>(d); }
inline int __clzll(long long x) { return x ? __builtin_clzll((unsigned long long)x) : 64; }
inline int __clz(int x) { return x ? __builtin_clz((unsigned)x) : 32; }
template <class T>
inline T __ldg(const T* p) { return *p; }
inline unsigned long long atomicAdd(unsigned long long* p, unsigned long long v) {
  const unsigned long long o = *p;
  *p += v;
  return o;
}
inline int atomicOr(int* p, int v) {
  const int o = *p;
  *p |= v;
  return o;
}
template <class T>
inline T __shfl_xor_sync(unsigned, T v, int, int = 32) { return v; }
template <class T>
inline T __shfl_sync(unsigned, T v, int, int = 32) { return v; }
inline int __all_sync(unsigned, int p) { return p; }
inline int __reduce_max_sync(unsigned, int v) { return v; }
inline unsigned __reduce_add_sync(unsigned, unsigned v) { return v; }
inline void __syncwarp(unsigned = 0xFFFFFFFFu) {}
inline unsigned __ballot_sync(unsigned, int p) { return p ? 1u : 0u; }
inline int __any_sync(unsigned, int p) { return p; }
inline int __popc(unsigned x) { return __builtin_popcount(x); }
