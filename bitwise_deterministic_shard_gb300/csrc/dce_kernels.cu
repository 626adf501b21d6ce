// det-cross-entropy kernels for sm_103a: vocab-range rowmax, exact denominator digits,
// finalize to (loss, denom).
//
// Page "det-cross-entropy", section "Method": m_i = max_v x_iv (order-invariant), then
// den_i = sum_v exp(x_iv - m_i) in a Kulisch long accumulator of signed int64 digits;
// shards compose by an elementwise max and an int64 digit add; the loss is
// logsumexp - x_target.  The contract here: weights exp32_det(RN32(x - m)), digits in
// radix 2^32 with E0 = -160, loss = RN32(RN64(log64_det(RN64(den)) + RN64(m - x_t))).
//
// One CTA streams one row of logits with 16-byte loads (HBM-bound: 4 B per f32 logit,
// 2 B per bf16 logit) and keeps six int64 digits per thread; the CTA sum of digits is
// exact, so the reduction order does not matter.
#include "numerics.cuh"
#include "attn_kernels.h"

namespace detattn {

// visit every element of row[v_lo, v_hi) owned by this thread: scalar head up to a 16-byte
// boundary, 16-byte vectors, scalar tail
template <int DT, typename F>
__device__ __forceinline__ void for_row(const typename In<DT>::T* row, int64_t v_lo, int64_t v_hi, F&& f) {
  using T = typename In<DT>::T;
  constexpr int VEC = 16 / sizeof(T);
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row + v_lo);
  int64_t head = (int64_t)(((16 - (addr & 15)) & 15) / sizeof(T));
  if (((addr & 15) % sizeof(T)) != 0) head = v_hi - v_lo;   // unaligned element pointer: scalar only
  const int64_t hend = min(v_hi, v_lo + head);
  for (int64_t v = v_lo + threadIdx.x; v < hend; v += blockDim.x) f(In<DT>::bits(row, v));
  const int64_t nvec = (v_hi - hend) / VEC;
  const uint4* vp = reinterpret_cast<const uint4*>(row + hend);
  for (int64_t k = threadIdx.x; k < nvec; k += blockDim.x) {
    uint4 q = __ldg(vp + k);
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
    if constexpr (DT == 0) {
#pragma unroll
      for (int t = 0; t < 4; t++) f(w[t]);
    } else {
#pragma unroll
      for (int t = 0; t < 4; t++) {
        f(w[t] << 16);
        f(w[t] & 0xFFFF0000u);
      }
    }
  }
  for (int64_t v = hend + nvec * VEC + threadIdx.x; v < v_hi; v += blockDim.x) f(In<DT>::bits(row, v));
}

template <int DT>
__global__ void __launch_bounds__(256) dce_rowmax_kernel(const DceArgs a) {
  using T = typename In<DT>::T;
  const int64_t i = blockIdx.x;
  const T* row = (const T*)a.x + i * a.rs;
  float mx = __int_as_float(0xFF800000);
  int nf = 0;
  for_row<DT>(row, a.v_lo, a.v_hi, [&](uint32_t u) {
    if (nonfinite_bits(u)) { nf = ST_NONFINITE; return; }
    float x = __uint_as_float(u);
    mx = x > mx ? x : mx;
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  __shared__ float wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = wm[0];
    for (int w = 1; w < 8; w++) m = wm[w] > m ? wm[w] : m;
    if (m == 0.0f) m = __int_as_float(0);   // -0 -> +0
    a.m_out[i] = m;
  }
  report(a.status, nf);
}

template <int DT>
__global__ void __launch_bounds__(256) dce_denom_kernel(const DceArgs a) {
  using T = typename In<DT>::T;
  const int64_t i = blockIdx.x;
  const T* row = (const T*)a.x + i * a.rs;
  const float m = a.m_in[i];
  long long d0 = 0, d1 = 0, d2 = 0, d3 = 0, d4 = 0, d5 = 0;   // word k weighs 2^(32k - 160)
  int st = 0;
  for_row<DT>(row, a.v_lo, a.v_hi, [&](uint32_t u) {
    if (nonfinite_bits(u)) { st |= ST_NONFINITE; return; }
    float x = __fsub_rn(__uint_as_float(u), m);
    if (x != x) { st |= ST_NONFINITE; return; }
    if (x > 0.0f) { st |= ST_VIOLATION; x = 0.0f; }
    const uint32_t wb = __float_as_uint(exp32_det(x));
    if (wb == 0u) return;
    const int ex = (int)(wb >> 23);
    const uint32_t M = ex ? ((wb & 0x7FFFFFu) | 0x800000u) : wb;
    const int pos = (ex ? ex : 1) + 10;        // bit position of M's unit above 2^-160
    const int k = pos >> 5;
    const unsigned long long ch = (unsigned long long)M << (pos & 31);
    const long long c0 = (long long)(ch & 0xFFFFFFFFull), c1 = (long long)(ch >> 32);
    if (k >= 3) {                               // w >= 2^-74: the common case
      const bool k4 = (k == 4);
      d3 += k4 ? 0 : c0;
      d4 += k4 ? c0 : c1;
      d5 += k4 ? c1 : 0;
    } else {
      if (k == 0) { d0 += c0; d1 += c1; }
      else if (k == 1) { d1 += c0; d2 += c1; }
      else { d2 += c0; d3 += c1; }
    }
  });
  long long dg[6] = {d0, d1, d2, d3, d4, d5};
#pragma unroll
  for (int k = 0; k < 6; k++)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dg[k] += __shfl_xor_sync(0xFFFFFFFFu, dg[k], o);
  __shared__ long long wsum[8][6];
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int k = 0; k < 6; k++) wsum[threadIdx.x >> 5][k] = dg[k];
  __syncthreads();
  if (threadIdx.x == 0) {
    long long t[6];
    long long* out = a.den + i * DEN_NDIG;
#pragma unroll
    for (int k = 0; k < 6; k++) {
      t[k] = a.add_into ? out[k] : 0;
      for (int w = 0; w < 8; w++) t[k] += wsum[w][k];
    }
    kul_carry(t, 6);
    if (t[5] > (1ll << 62) || t[5] < -(1ll << 62)) st |= ST_HEADROOM;
#pragma unroll
    for (int k = 0; k < 6; k++) out[k] = t[k];
  }
  report(a.status, st);
}

template <int DT>
__global__ void dce_finalize_kernel(const DceArgs a) {
  using T = typename In<DT>::T;
  int st = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < a.N; i += (int64_t)gridDim.x * blockDim.x) {
    long long e[DEN_NDIG];
#pragma unroll
    for (int k = 0; k < DEN_NDIG; k++) e[k] = a.den[i * DEN_NDIG + k];
    const double d64 = digits_rn64<DEN_NDIG>(e, DEN_E0);
    a.denom[i] = d64;
    const int64_t t = a.targets[i];
    if (t < 0 || t >= a.V) {
      st |= ST_BAD_TARGET;
      a.loss[i] = __int_as_float(0x7FC00000);
      continue;
    }
    const double xt = (double)__uint_as_float(In<DT>::bits((const T*)a.x + i * a.rs, t));
    const double diff = __dsub_rn((double)a.m_in[i], xt);
    a.loss[i] = __double2float_rn(__dadd_rn(log64_det(d64), diff));
  }
  report(a.status, st);
}

cudaError_t launch_dce_rowmax(const DceArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  if (a.dtype == 0) dce_rowmax_kernel<0><<<(unsigned)a.N, 256, 0, st>>>(a);
  else dce_rowmax_kernel<1><<<(unsigned)a.N, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dce_denom(const DceArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  if (a.dtype == 0) dce_denom_kernel<0><<<(unsigned)a.N, 256, 0, st>>>(a);
  else dce_denom_kernel<1><<<(unsigned)a.N, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dce_finalize(const DceArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((a.N + 255) / 256);
  if (a.dtype == 0) dce_finalize_kernel<0><<<blocks, 256, 0, st>>>(a);
  else dce_finalize_kernel<1><<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace detattn
