// Measurement and self-test entry points that sit beside the method (include/detattn.h,
// "probes"): they compute nothing of the attention or cross-entropy path.
//
// da_probe_int_mac: the issue rate of exact 32 x 32 -> 64-bit integer multiply-adds
// (mad.wide.s32) over the whole GPU, the unit of exact arithmetic the integer pipe offers.
// The benchmark divides the path's exact multiply-adds per second by this rate to state
// the fraction of the integer pipe's peak that the path reaches.
//
// da_probe_bounded_wait: one warp waits on an mbarrier phase that nothing completes, through
// the same bounded wait (tc5.cuh) every pipelined kernel of the library uses.  The wait gives
// up after its time limit, the kernel returns normally and reports DA_STATUS_TIMEOUT in the
// status word, so the caller's context stays usable: the timeout path is exercised without
// a fault or a hang.
//
// da_probe_packed: the packed two-lane forms (pack2.cuh) of the exponential and of the
// backward's quotient against the scalar ones, on every binary32 bit pattern of a range; the
// cross-entropy kernels take the packed forms for two adjacent logits, so they must give the
// same bits for every argument.
#include "../../include/detattn.h"
#include "numerics.cuh"
#include "pack2.cuh"
#include "fdiv.cuh"
#include "tc5.cuh"

namespace detattn {

constexpr int PROBE_ACC = 8;   // independent accumulators per thread (hides the multiply latency)
constexpr int PROBE_UNROLL = 4;

// Thread pairs (u, u + 1) of the range [lo, lo + count) (bit patterns, wrapping mod 2^32).
// which 0: x is the binary32 with those bits, clamped as the kernels clamp (NaN -> -inf, then
// to [-104, 0]); counts the patterns whose packed exp32_det_poly2 (p or k) differs from the
// scalar exp32_det_poly in any bit.  which 1: p in [0.5, 2) takes the pattern's low 24 bits,
// the divisor d in [1, 2^21) a hash of it; counts the patterns whose packed quotient and
// residual estimate (the backward's pair form) differ from the scalar ones in any bit.
__global__ void __launch_bounds__(256) probe_packed_kernel(int which, uint32_t lo, long long count,
                                                           unsigned long long* mismatches) {
  unsigned long long bad = 0;
  const long long npairs = (count + 1) / 2;
  for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < npairs;
       q += (long long)gridDim.x * blockDim.x) {
    const uint32_t u0 = lo + (uint32_t)(2 * q);
    const uint32_t u1 = 2 * q + 1 < count ? u0 + 1u : u0;
    bool m0, m1;
    if (which == 0) {
      auto arg = [](uint32_t u) {
        const float x = __uint_as_float(u);
        return fmaxf(x != x ? neg_inf() : (x > 0.0f ? 0.0f : x), -104.0f);
      };
      const float x0 = arg(u0), x1 = arg(u1);
      float p0, p1;
      int k0, k1, s0, s1;
      exp32_det_poly2(x0, x1, p0, p1, k0, k1);
      const float sp0 = exp32_det_poly(x0, s0), sp1 = exp32_det_poly(x1, s1);
      m0 = __float_as_uint(p0) != __float_as_uint(sp0) || k0 != s0;
      m1 = __float_as_uint(p1) != __float_as_uint(sp1) || k1 != s1;
    } else {
      const uint32_t h = (u0 >> 1) * 0x9E3779B1u;
      const double d = 1.0 + (double)(h >> 1) * 0x1p-11;   // one divisor per pair, as in a row
      fdiv::FpDivisor F;
      fdiv::make_fp_divisor(d, F);
      auto pv = [](uint32_t u) { return __uint_as_float(((126u + ((u >> 23) & 1u)) << 23) | (u & 0x7FFFFFu)); };
      const float p0 = pv(u0), p1 = pv(u1);
      using namespace f2;   // the pair form, as the backward evaluates it
      const u64 q0 = pack(__fmul_rn(p0, F.r), __fmul_rn(p1, F.r));
      const u64 e2 = fma(q0, splat(-F.lo), fma(q0, splat(-F.hi), pack(p0, p1)));
      const u64 q1 = fma(e2, splat(F.r), q0);
      float qa, qb, da, db;
      unpack(q1, qa, qb);
      unpack(fma(e2, splat(F.r), sub(q0, q1)), da, db);
      auto scalar = [&](float p, float& q, float& dl) {   // the single form
        const float s0 = __fmul_rn(p, F.r);
        const float s2 = __fmaf_rn(s0, -F.lo, __fmaf_rn(s0, -F.hi, p));
        q = __fmaf_rn(s2, F.r, s0);
        dl = __fmaf_rn(s2, F.r, __fsub_rn(s0, q));
      };
      float sq0, sd0, sq1, sd1;
      scalar(p0, sq0, sd0);
      scalar(p1, sq1, sd1);
      m0 = __float_as_uint(qa) != __float_as_uint(sq0) || __float_as_uint(da) != __float_as_uint(sd0);
      m1 = __float_as_uint(qb) != __float_as_uint(sq1) || __float_as_uint(db) != __float_as_uint(sd1);
    }
    bad += (unsigned long long)m0 + (unsigned long long)(m1 && u1 != u0);
  }
  for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xFFFFFFFFu, bad, o);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(mismatches, bad);
}

__global__ void __launch_bounds__(512) probe_int_mac_kernel(long long iters, long long* sink) {
  long long acc[PROBE_ACC];
  int a[PROBE_ACC];
#pragma unroll
  for (int k = 0; k < PROBE_ACC; k++) {
    acc[k] = threadIdx.x + k;
    a[k] = (int)(0x9E3779B1u * (threadIdx.x * PROBE_ACC + k + 1));
  }
  const int b = (int)(blockIdx.x * 2654435761u) | 1;
  for (long long it = 0; it < iters; it++) {
#pragma unroll
    for (int u = 0; u < PROBE_UNROLL; u++)
#pragma unroll
      for (int k = 0; k < PROBE_ACC; k++) asm volatile("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc[k]) : "r"(a[k]), "r"(b));
  }
  long long s = 0;
#pragma unroll
  for (int k = 0; k < PROBE_ACC; k++) s ^= acc[k];
  if (s == 0x7FFFFFFFFFFFFFFFll) sink[0] = s;   // keeps the chain alive; practically never stored
}

__global__ void probe_bounded_wait_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    tc5::mbar_init(&bar, 1);   // one arrival would complete phase 0; none comes
    abort_flag = 0;
    tc5::mbar_fence_init();
  }
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) ok = tc5::mbar_wait(&bar, 0, &abort_flag, 1000);
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  if (!ok && threadIdx.x == 0) report(status, ST_TIMEOUT);
}

}  // namespace detattn

#define DA_EXPORT __attribute__((visibility("default")))

extern "C" {

DA_EXPORT int da_probe_packed(int which, uint32_t lo_bits, int64_t count, int64_t* mismatches, da_stream_t stream) {
  if (which < 0 || which > 1 || count < 0 || count > (1ll << 32) || !mismatches) return DA_EINVAL;
  if (reinterpret_cast<uintptr_t>(mismatches) % 8) return DA_EALIGN;
  if (count == 0) return DA_OK;
  detattn::probe_packed_kernel<<<1216, 256, 0, (cudaStream_t)stream>>>(which, lo_bits, (long long)count,
                                                                       (unsigned long long*)mismatches);
  return cudaGetLastError() == cudaSuccess ? DA_OK : DA_ECUDA;
}

DA_EXPORT int da_probe_int_mac(int64_t iters, int nblocks, int64_t* sink, da_stream_t stream) {
  if (iters < 0 || nblocks < 1 || nblocks > (1 << 20)) return DA_EINVAL;
  if (!sink) return DA_EINVAL;
  if (reinterpret_cast<uintptr_t>(sink) % 8) return DA_EALIGN;
  detattn::probe_int_mac_kernel<<<nblocks, 512, 0, (cudaStream_t)stream>>>(iters, (long long*)sink);
  return cudaGetLastError() == cudaSuccess ? DA_OK : DA_ECUDA;
}

DA_EXPORT int64_t da_probe_int_mac_per_thread_iter(void) {
  return (int64_t)detattn::PROBE_ACC * detattn::PROBE_UNROLL;
}

DA_EXPORT int da_probe_bounded_wait(int32_t* dev_status, da_stream_t stream) {
  if (!dev_status) return DA_EINVAL;
  if (reinterpret_cast<uintptr_t>(dev_status) % 4) return DA_EALIGN;
  detattn::probe_bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((int*)dev_status);
  return cudaGetLastError() == cudaSuccess ? DA_OK : DA_ECUDA;
}

}  // extern "C"
