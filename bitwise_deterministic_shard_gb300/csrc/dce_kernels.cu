// det-cross-entropy kernels for sm_103a: vocab-range rowmax, exact denominator digits,
// finalize to (loss, denom), the backward dLogits and the exact loss reductions.
//
// Page "det-cross-entropy", section "Method": m_i = max_v x_iv (order-invariant), then
// den_i = sum_v exp(x_iv - m_i) in a Kulisch long accumulator of signed int64 digits;
// shards compose by an elementwise max and an int64 digit add; the loss is
// logsumexp - x_target.  The contract here: weights exp32_det(RN32(x - m)), digits in
// radix 2^32 with E0 = -160, loss = RN32(RN64(log64_det(RN64(den)) + RN64(m - x_t))).
//
// The denominator streams each row of logits with 16-byte loads (HBM-bound: 4 B per f32
// logit, 2 B per bf16 logit), one CTA or one cluster of CTAs per row, six int64 digits per
// thread; the sums of digits are exact, so the reduction order does not matter.  The
// exponentials of adjacent logits are evaluated in pairs on the packed FP32 instructions.
#include <cuda_bf16.h>
#include <cooperative_groups.h>
#include "numerics.cuh"
#include "fdiv.cuh"
#include "den_acc.cuh"
#include "pack2.cuh"
#include "attn_kernels.h"

namespace detattn {

namespace cg = cooperative_groups;

// visit every element of row[v_lo, v_hi) owned by this thread: scalar head up to a 16-byte
// boundary, 16-byte vectors, scalar tail.  f(bits) takes one element, f2(bits, bits) the
// adjacent pairs of a vector; group() runs before each vector or scalar element.
template <int DT, typename F, typename F2, typename G>
__device__ __forceinline__ void for_row2(const typename In<DT>::T* row, int64_t v_lo, int64_t v_hi, F&& f, F2&& f2,
                                         G&& group) {
  using T = typename In<DT>::T;
  constexpr int VEC = 16 / sizeof(T);
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row + v_lo);
  int64_t head = (int64_t)(((16 - (addr & 15)) & 15) / sizeof(T));
  if (((addr & 15) % sizeof(T)) != 0) head = v_hi - v_lo;   // unaligned element pointer: scalar only
  const int64_t hend = min(v_hi, v_lo + head);
  for (int64_t v = v_lo + threadIdx.x; v < hend; v += blockDim.x) {
    group();
    f(In<DT>::bits(row, v));
  }
  const int64_t nvec = (v_hi - hend) / VEC;
  const uint4* vp = reinterpret_cast<const uint4*>(row + hend);
  auto vec = [&](const uint4& q) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    group();
    if constexpr (DT == 0) {
      f2(w[0], w[1]);
      f2(w[2], w[3]);
    } else {
#pragma unroll
      for (int t = 0; t < 4; t++) f2(w[t] << 16, w[t] & 0xFFFF0000u);
    }
  };
  // NB vectors per thread in flight before their arithmetic (the loop body is long, so one
  // load at a time would leave the memory system short of requests)
  constexpr int NB = 3;
  const int64_t step = blockDim.x;
  int64_t k = threadIdx.x;
  for (; k + (NB - 1) * step < nvec; k += NB * step) {
    uint4 q[NB];
#pragma unroll
    for (int b = 0; b < NB; b++) q[b] = __ldg(vp + k + b * step);
#pragma unroll
    for (int b = 0; b < NB; b++) vec(q[b]);
  }
  for (; k < nvec; k += step) vec(__ldg(vp + k));
  for (int64_t v = hend + nvec * VEC + threadIdx.x; v < v_hi; v += blockDim.x) {
    group();
    f(In<DT>::bits(row, v));
  }
}

template <int DT, typename F, typename G>
__device__ __forceinline__ void for_row(const typename In<DT>::T* row, int64_t v_lo, int64_t v_hi, F&& f, G&& group) {
  for_row2<DT>(row, v_lo, v_hi, f, [&](uint32_t u0, uint32_t u1) { f(u0); f(u1); }, group);
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
  }, [] {});
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

// A row is split over `parts` CTAs (1, 2, 4 or 8), one thread-block cluster per row; six
// CTAs resident per SM.  Each CTA sums its share of the columns; the others' sums reach the
// cluster's first CTA through distributed shared memory, and it adds them (integers: exact in
// any order), carries and writes the row's digits.  Splitting the rows fills the GPU when the
// rows are fewer than its CTA slots.
constexpr int DEN_THREADS = 256, DEN_MAX_PARTS = 8;

template <int DT>
__global__ void __launch_bounds__(DEN_THREADS, 6) dce_denom_kernel(const DceArgs a, int parts) {
  using T = typename In<DT>::T;
  const int64_t i = blockIdx.x / parts;
  const int c = (int)(blockIdx.x % parts);   // the CTA's rank in its cluster
  const T* row = (const T*)a.x + i * a.rs;
  const float m = a.m_in[i];
  // this CTA's columns: equal shares of the range, each a multiple of 64 columns
  const int64_t share = ((a.v_hi - a.v_lo + parts - 1) / parts + 63) / 64 * 64;
  const int64_t c_lo = min(a.v_hi, a.v_lo + c * share), c_hi = min(a.v_hi, c_lo + share);
  DenAcc A;   // exact: a private word for w >= 2^-31, digit words for the rest (den_acc.cuh)
  den_init(A);
  int st = 0;
  // common case, one unsigned test on the bits of x = RN32(logit - m): x in [-21.4, -0].  Then
  // the weight w = exp32_det(x) is at least 2^-31 (exp(-21.4) > 2^-31) and exp32_det's p 2^k
  // (exact for k >= -125), so its mantissa goes straight into the private word, shifted by
  // sh = (biased exponent of w) - 96 >= 0 (den_add's first case, without forming w).  NaN,
  // infinite, above-maximum and +0 logits and smaller weights take the general handling; the
  // packed evaluation runs on x unclamped, and its values are used only inside the range.
  auto fast = [&](float x, float p, int k) -> bool {
    if (__float_as_uint(x) - 0x80000000u <= 0x41AB3333u) {   // -21.4f = 0xC1AB3333
      const uint32_t pbits = __float_as_uint(p);
      A.U += (uint64_t)((pbits & 0x7FFFFFu) | 0x800000u) << ((int)(pbits >> 23) + k - 96);
      return true;
    }
    return false;
  };
  auto general = [&](uint32_t u, float x) {
    if (nonfinite_bits(u)) { st |= ST_NONFINITE; return; }
    if (x != x) { st |= ST_NONFINITE; return; }
    if (x > 0.0f) { st |= ST_VIOLATION; x = 0.0f; }
    den_add(A, __float_as_uint(exp32_det_nb(x)));   // x <= 0, not NaN
  };
  for_row2<DT>(row, c_lo, c_hi,
               [&](uint32_t u) {
                 const float x = __fsub_rn(__uint_as_float(u), m);
                 int k;
                 const float p = exp32_det_poly(fmaxf(x, -104.0f), k);
                 if (!fast(x, p, k)) general(u, x);
               },
               [&](uint32_t u0, uint32_t u1) {   // two logits on the packed FP32 lanes
                 float x0, x1, p0, p1;
                 int k0, k1;
                 f2::unpack(f2::sub(f2::pack(__uint_as_float(u0), __uint_as_float(u1)), f2::splat(m)), x0, x1);
                 exp32_det_poly2(x0, x1, p0, p1, k0, k1);
                 if (!fast(x0, p0, k0)) general(u0, x0);
                 if (!fast(x1, p1, k1)) general(u1, x1);
               },
               [&] { den_guard(A); });
  den_flush(A);
  long long dg[6] = {A.d[0], A.d[1], A.d[2], A.d[3], A.d[4], A.d[5]};
#pragma unroll
  for (int k = 0; k < 6; k++)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dg[k] += __shfl_xor_sync(0xFFFFFFFFu, dg[k], o);
  __shared__ long long wsum[DEN_THREADS / 32][6];
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int k = 0; k < 6; k++) wsum[threadIdx.x >> 5][k] = dg[k];
  __shared__ long long psum[DEN_MAX_PARTS][6];   // the cluster's first CTA: the others' sums
  __syncthreads();
  long long t[6];
  if (threadIdx.x == 0)
#pragma unroll
    for (int k = 0; k < 6; k++) {
      t[k] = 0;
      for (int w = 0; w < DEN_THREADS / 32; w++) t[k] += wsum[w][k];
    }
  if (parts > 1) {
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();   // every CTA of the cluster runs: the first one's psum may be written
    if (threadIdx.x == 0 && c > 0) {
      long long* dst = cl.map_shared_rank(&psum[c][0], 0);
#pragma unroll
      for (int k = 0; k < 6; k++) dst[k] = t[k];
    }
    cl.sync();   // the sums have landed
    if (c > 0) {
      report(a.status, st);
      return;
    }
    if (threadIdx.x == 0)
      for (int q = 1; q < parts; q++)
#pragma unroll
        for (int k = 0; k < 6; k++) t[k] += psum[q][k];
  }
  if (threadIdx.x == 0) {
    long long* out = a.den + i * DEN_NDIG;
#pragma unroll
    for (int k = 0; k < 6; k++) t[k] += a.add_into ? out[k] : 0;
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
    if (t < 0 || t >= a.v_total) {
      st |= ST_BAD_TARGET;
      a.loss[i] = __int_as_float(0x7FC00000);
      continue;
    }
    const int64_t c = t - a.v_base;   // the target's column in this matrix
    if (c < 0 || c >= a.V) {          // another vocabulary shard holds it: this shard adds +0
      a.loss[i] = 0.0f;
      continue;
    }
    const double xt = (double)__uint_as_float(In<DT>::bits((const T*)a.x + i * a.rs, c));
    const double diff = __dsub_rn((double)a.m_in[i], xt);
    a.loss[i] = __double2float_rn(__dadd_rn(log64_det(d64), diff));
  }
  report(a.status, st);
}

// Backward (page "det-cross-entropy", "API": cross_entropy with a deterministic dLogits;
// "Method": the gradient softmax(x_i) - onehot(t_i)), one IEEE rounding per step:
//   p = RN32(RN64(exp32_det(RN32(x - m)) / denom)),  g = RN32(p - [v == t]),
//   dLogits = RN32(go * g),  go = grad[i] ("none"), grad[0] ("sum"), RN32(RN64(grad[0] / N))
// ("mean").  A logit above the rowmax is clamped like the forward's (violation flag); NaN
// propagates.  Streaming: 2 B or 4 B read and 2 B or 4 B written per logit; one CTA covers
// BW_CHUNK columns of one row.  The quotient is rounded to binary32 on the FP32 pipe from the
// row's split divisor with a residual certificate (fdiv.cuh), and divided in binary64 only
// when that rounding is not certain (a quotient within about 2^-15 binary32 ulp of a
// half-way point, or a subnormal one) or the operands are special.  The divisor setup is a
// few conversions for one thread of the CTA, with no division.
// 16 logits a thread and eight CTAs an SM (32 registers): occupancy decides this kernel, whose
// loads of a thread are all issued before its arithmetic (measured on the 4096 x V128256 f32
// rows: 0.73 ms against 0.92 ms with 32 logits a thread at 64 registers)
constexpr int BW_THREADS = 256, BW_PER = 16, BW_CHUNK = BW_THREADS * BW_PER, BW_BATCH = 8, BW_MINB = 8;

// VEC: the row and the output row start on 16-byte boundaries and hold a whole number of
// 16-byte vectors, so each thread moves its logits as 16-byte loads and stores (f32: 8 x 4,
// bf16: 4 x 8), the loads all issued before the arithmetic.
template <int DT, bool VEC>
__global__ void __launch_bounds__(BW_THREADS, BW_MINB) dce_backward_kernel(const DceArgs a, const float* __restrict__ grad,
                                                                  int reduction, void* __restrict__ dlogits) {
  using T = typename In<DT>::T;
  __shared__ fdiv::FpDivisor sfd;
  __shared__ int sfast;
  __shared__ float sgo;
  const int64_t nch = (a.V + BW_CHUNK - 1) / BW_CHUNK;
  const int64_t i = blockIdx.x / nch, c0 = (blockIdx.x % nch) * BW_CHUNK;
  const T* __restrict__ row = (const T*)a.x + i * a.rs + c0;
  T* __restrict__ orow = (T*)dlogits + i * a.V + c0;
  const int nv = (int)(a.V - c0 < BW_CHUNK ? a.V - c0 : BW_CHUNK);
  const float m = a.m_in[i];
  const double d64 = a.denom[i];
  if (threadIdx.x == 0) {   // the row's divisor, once per CTA (a few conversions, no division)
    sfast = fdiv::make_fp_divisor(d64, sfd);   // d in [2^-60, 2^60]: the FP32-pipe quotient
    float g0 = reduction == 0 ? grad[i] : grad[0];
    if (reduction == 2) g0 = __double2float_rn(__ddiv_rn((double)g0, (double)a.N));   // once per CTA
    sgo = g0;
  }
  __syncthreads();
  const fdiv::FpDivisor F = sfd;
  const bool fast = sfast;
  const float go = sgo;
  const int64_t tg64 = a.targets[i] - a.v_base - c0;   // the target's column within this chunk (any value)
  const int tg = tg64 >= 0 && tg64 < nv ? (int)tg64 : -1;
  int st = 0;
  // fin: dLogits of the logit in column v of the chunk, from x = RN32(logit - m),
  // exp32_det_poly(max(x, -104)) = (pp, k) and the FP32-pipe quotient of pp by the row's
  // denominator (candidate bits qb, residual estimate dl; fdiv.cuh).  Fast path: the weight is
  // exp32_det's pp 2^k (exact for k >= -125), so RN32(RN64(w / d)) is the certified quotient of
  // pp times 2^k when that is a normal binary32.  Otherwise (NaN, deep or zero weights, special
  // denominators, an uncertain rounding: rare) the binary64 division, correctly rounded, so
  // RN32 of its result is the contract's quotient by definition.
  auto fin = [&](float x, int k, uint32_t qb, float dl, int v) -> float {
    // the common case: x in [-86.5, -0] (one unsigned test on its bits: not NaN, not infinite,
    // not above the maximum), so k >= -125 and the weight p 2^k is exact and normal; the
    // exponential and the quotient were evaluated on x unclamped and are used only then
    const int be = (int)(qb >> 23) + k;   // the quotient's biased exponent after the 2^k
    float p;
    if (fast && __float_as_uint(x) - 0x80000000u <= 0x42AD0000u && be >= 1 && fdiv::certain(qb, dl)) {   // -86.5f
      p = __uint_as_float(qb + ((uint32_t)k << 23));
    } else {
      if (x > 0.0f) {   // above the maximum: clamped as in the forward
        st |= ST_VIOLATION;
        x = 0.0f;
      }
      const float w = x != x ? x : exp32_det_nb(x);
      p = __double2float_rn(__ddiv_rn((double)w, d64));
    }
    const float g = v == tg ? __fsub_rn(p, 1.0f) : p;
    return __fmul_rn(go, g);
  };
  auto one = [&](uint32_t u, int v) -> float {
    const float x = __fsub_rn(__uint_as_float(u), m);
    int k;
    const float pp = exp32_det_poly(fmaxf(x, -104.0f), k);
    const float q0 = __fmul_rn(pp, F.r);
    const float e2 = __fmaf_rn(q0, -F.lo, __fmaf_rn(q0, -F.hi, pp));
    const float q1 = __fmaf_rn(e2, F.r, q0);
    return fin(x, k, __float_as_uint(q1), __fmaf_rn(e2, F.r, __fsub_rn(q0, q1)), v);
  };
  // two adjacent logits (columns v, v + 1): the exponentials and the quotients on the packed
  // FP32 lanes (the same operations as `one`, lane by lane; q0 from scalar multiplies, as a
  // packed multiply feeding the packed subtraction could be fused into it)
  auto two = [&](uint32_t u0, uint32_t u1, int v, float& o0, float& o1) {
    using namespace f2;
    float x0, x1, p0, p1;
    int k0, k1;
    unpack(sub(pack(__uint_as_float(u0), __uint_as_float(u1)), splat(m)), x0, x1);
    exp32_det_poly2(x0, x1, p0, p1, k0, k1);
    const u64 q0 = pack(__fmul_rn(p0, F.r), __fmul_rn(p1, F.r));
    const u64 e2 = fma(q0, splat(-F.lo), fma(q0, splat(-F.hi), pack(p0, p1)));
    const u64 q1 = fma(e2, splat(F.r), q0);
    float qa, qb, da, db;
    unpack(q1, qa, qb);
    unpack(fma(e2, splat(F.r), sub(q0, q1)), da, db);
    o0 = fin(x0, k0, __float_as_uint(qa), da, v);
    o1 = fin(x1, k1, __float_as_uint(qb), db, v + 1);
  };
  if constexpr (VEC) {
    constexpr int EV = 16 / (int)sizeof(T), NV = BW_PER / EV;
    const uint4* __restrict__ src = reinterpret_cast<const uint4*>(row);
    uint4* __restrict__ dst = reinterpret_cast<uint4*>(orow);
    uint4 q[NV];
#pragma unroll
    for (int k = 0; k < NV; k++) {   // every load in flight before the arithmetic
      const int gv = k * BW_THREADS + threadIdx.x;
      q[k] = gv * EV < nv ? __ldcs(src + gv) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < NV; k++) {
      const int gv = k * BW_THREADS + threadIdx.x;
      if (gv * EV >= nv) continue;   // nv is a multiple of EV here
      const uint32_t wd[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
      uint32_t o[4];
      if constexpr (DT == 0) {
#pragma unroll
        for (int t = 0; t < 4; t += 2) {
          float r0, r1;
          two(wd[t], wd[t + 1], gv * 4 + t, r0, r1);
          o[t] = __float_as_uint(r0);
          o[t + 1] = __float_as_uint(r1);
        }
      } else {
#pragma unroll
        for (int t = 0; t < 4; t++) {
          float r0, r1;
          two(wd[t] << 16, wd[t] & 0xFFFF0000u, gv * 8 + 2 * t, r0, r1);
          const __nv_bfloat162 h = __floats2bfloat162_rn(r0, r1);
          o[t] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      __stcs(dst + gv, make_uint4(o[0], o[1], o[2], o[3]));
    }
  } else {
    for (int k0 = 0; k0 < BW_PER; k0 += BW_BATCH) {
      uint32_t u[BW_BATCH];
#pragma unroll
      for (int j = 0; j < BW_BATCH; j++) {   // the batch's loads first, all in flight together
        const int v = (k0 + j) * BW_THREADS + threadIdx.x;
        u[j] = v < nv ? In<DT>::bits(row, v) : 0u;
      }
#pragma unroll
      for (int j = 0; j < BW_BATCH; j++) {
        const int v = (k0 + j) * BW_THREADS + threadIdx.x;
        if (v >= nv) continue;
        const float o = one(u[j], v);
        if constexpr (DT == 0)
          ((float*)orow)[v] = o;
        else
          ((__nv_bfloat16*)orow)[v] = __float2bfloat16_rn(o);
      }
    }
  }
  report(a.status, st);
}

// Loss reductions: S = the exact sum of the f32 losses (Kulisch words of 2^(32k - 320)),
// "sum" = RN32(RN64(S)), "mean" = RN32(RN64(RN64(S) / N)); a NaN loss gives NaN, infinite
// losses their IEEE sum.  One CTA: per-thread words, combined by exact shared-memory adds.
__global__ void __launch_bounds__(256) dce_reduce_kernel(const float* loss, int64_t N, int reduction, float* out) {
  __shared__ long long tot[KW];
  __shared__ int flags;   // 1 NaN, 2 +inf, 4 -inf
  for (int k = threadIdx.x; k < KW; k += blockDim.x) tot[k] = 0;
  if (threadIdx.x == 0) flags = 0;
  __syncthreads();
  long long acc[KW];
#pragma unroll
  for (int k = 0; k < KW; k++) acc[k] = 0;
  int fl = 0;
  for (int64_t i = threadIdx.x; i < N; i += blockDim.x) {
    const uint32_t u = __float_as_uint(loss[i]);
    if (nonfinite_bits(u)) {
      fl |= (u & 0x7FFFFFu) ? 1 : ((u >> 31) ? 4 : 2);
      continue;
    }
    const Split s = split_f32(u);
    kul_add(acc, s.mant, s.neg, s.lsb);
    if ((i / blockDim.x) % 1024 == 1023) kul_carry(acc, KW);   // keep the words far from overflow
  }
  kul_carry(acc, KW);
#pragma unroll
  for (int k = 0; k < KW; k++)
    if (acc[k]) atomicAdd((unsigned long long*)&tot[k], (unsigned long long)acc[k]);
  if (fl) atomicOr(&flags, fl);
  __syncthreads();
  if (threadIdx.x == 0) {
    float r;
    if (flags & 1 || (flags & 6) == 6) {
      r = __int_as_float(0x7FC00000);
    } else if (flags) {
      r = __int_as_float(flags & 2 ? 0x7F800000 : 0xFF800000);
    } else {
      long long w[KW];
#pragma unroll
      for (int k = 0; k < KW; k++) w[k] = tot[k];
      double s64 = digits_rn64<KW>(w, -320);
      if (reduction == 2) s64 = __ddiv_rn(s64, (double)N);
      r = s64 == s64 ? __double2float_rn(s64) : __int_as_float(0x7FC00000);   // 0 / 0: the canonical NaN
    }
    *out = r;
  }
}

cudaError_t launch_dce_backward(const DceArgs& a, const float* grad, int reduction, void* dlogits, cudaStream_t st) {
  if (a.N <= 0 || a.V <= 0) return cudaSuccess;
  const int64_t blocks = a.N * ((a.V + BW_CHUNK - 1) / BW_CHUNK);
  if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  const int esz = a.dtype == 0 ? 4 : 2;
  const bool vec = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 && (reinterpret_cast<uintptr_t>(dlogits) & 15) == 0 &&
                   (a.rs * esz) % 16 == 0 && (a.V * esz) % 16 == 0;
  if (a.dtype == 0) {
    if (vec) dce_backward_kernel<0, true><<<(unsigned)blocks, BW_THREADS, 0, st>>>(a, grad, reduction, dlogits);
    else dce_backward_kernel<0, false><<<(unsigned)blocks, BW_THREADS, 0, st>>>(a, grad, reduction, dlogits);
  } else {
    if (vec) dce_backward_kernel<1, true><<<(unsigned)blocks, BW_THREADS, 0, st>>>(a, grad, reduction, dlogits);
    else dce_backward_kernel<1, false><<<(unsigned)blocks, BW_THREADS, 0, st>>>(a, grad, reduction, dlogits);
  }
  return cudaGetLastError();
}

cudaError_t launch_dce_reduce(const float* loss, int64_t N, int reduction, float* out, cudaStream_t st) {
  dce_reduce_kernel<<<1, 256, 0, st>>>(loss, N, reduction, out);
  return cudaGetLastError();
}

cudaError_t launch_dce_rowmax(const DceArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  if (a.dtype == 0) dce_rowmax_kernel<0><<<(unsigned)a.N, 256, 0, st>>>(a);
  else dce_rowmax_kernel<1><<<(unsigned)a.N, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// CTAs per row: the fewest of 1, 2, 4, 8 that fill the GPU's CTA slots (six per SM) once, each
// CTA keeping at least 4,096 columns.  Measured on the V128256 f32 rows: 256 rows run 1.4x
// faster on clusters of 8; from about one row per slot on, splitting gains nothing (the
// streaming CTAs of a partial last wave take the whole bandwidth).
static int denom_parts(int64_t N, int64_t cols) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 1;
  }
  int p = 1;
  while (p < DEN_MAX_PARTS && N * p < 6ll * sms && cols / (2 * p) >= 4096) p *= 2;
  return p;
}

cudaError_t launch_dce_denom(const DceArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  const int parts = denom_parts(a.N, a.v_hi - a.v_lo);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.N * parts));
  cfg.blockDim = dim3(DEN_THREADS);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)parts;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = parts > 1 ? 1 : 0;
  return a.dtype == 0 ? cudaLaunchKernelEx(&cfg, dce_denom_kernel<0>, a, parts)
                      : cudaLaunchKernelEx(&cfg, dce_denom_kernel<1>, a, parts);
}

cudaError_t launch_dce_finalize(const DceArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((a.N + 255) / 256);
  if (a.dtype == 0) dce_finalize_kernel<0><<<blocks, 256, 0, st>>>(a);
  else dce_finalize_kernel<1><<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace detattn
