// Key/value preparation for sm_103a: every K row of a call's key range becomes the four
// bf16 digit slices of its 26-bit fixed point (score_tc.cuh) plus its window exponent and
// fit flag; every V row becomes int32 fixed point against its column's largest exponent
// over the range (|Vint| < 2^23) plus a bit mask of the elements that do not fit.  Done
// once per call (O(S D) work), so the attention kernels copy ready tiles with cp.async
// instead of converting each tile once per block of query rows.
#include <cuda_fp16.h>
#include "numerics.cuh"
#include "score_tc.cuh"
#include "tc5.cuh"
#include "attn_kernels.h"

namespace detattn {

// column maxima of the V biased exponents over rows [lo, hi), atomically into vcol (zeroed);
// VCOL_ROWS rows per CTA, so that a short range still spreads over many CTAs
constexpr int VCOL_ROWS = 64;
template <int DT>
__global__ void __launch_bounds__(256) prep_vcol_kernel(const AttnArgs a, KvPrep p) {
  using T = typename In<DT>::T;
  const int hk = blockIdx.y, b = blockIdx.z;
  const T* vbase = (const T*)a.v + b * a.vs[0] + hk * a.vs[1];
  int* vcol = p.vcol + ((int64_t)b * a.Hkv + hk) * p.DP;
  const int j0 = a.kv_lo + blockIdx.x * VCOL_ROWS, j1 = min(a.kv_hi, j0 + VCOL_ROWS);
  for (int d = threadIdx.x % 64; d < a.D; d += 64) {
    int em = 0;
#pragma unroll 4
    for (int j = j0 + threadIdx.x / 64; j < j1; j += 4) {
      const uint32_t u = In<DT>::bits(vbase + (int64_t)j * a.vs[2], d);
      const int ex = (int)((u >> 23) & 0xFFu);
      if (ex != 0xFF) em = max(em, ex);
    }
    if (em) atomicMax(&vcol[d], em);
  }
}

// one warp per key row: K slices (both layouts) + meta, and (if p.do_v) V fixed point +
// spill bits.  Rows in [kv_hi, end of the last key tile) only zero their operand tile rows.
template <int DT, int DP>
__global__ void __launch_bounds__(256) prep_kv_kernel(const AttnArgs a, KvPrep p) {
  using T = typename In<DT>::T;
  constexpr int NW = DP / 32, NDS = DP / 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int jr = blockIdx.x * 8 + warp, j = a.kv_lo + jr;
  const int n = a.kv_hi - a.kv_lo;
  if (jr >= ((n + KTILE - 1) / KTILE) * KTILE) return;
  unsigned char* tile = p.ktc + ((int64_t)(b * a.Hkv + hk) * p.ntk + jr / KTILE) * NDS * KT_BLOCK;
  const int rt = jr % KTILE;
  auto store_tc = [&](int q, int d, uint16_t v) {
    *reinterpret_cast<uint16_t*>(tile + (d >> 4) * KT_BLOCK + q * (KTILE * 32) + tc5::canon_off(rt, d & 15)) = v;
  };
  unsigned char* vblk = (p.do_v && p.vtc != nullptr)
                            ? p.vtc + ((int64_t)(b * a.Hkv + hk) * p.ntk * (KTILE / VKEYS) + jr / VKEYS) * VP_BLOCK
                            : nullptr;
  auto store_v = [&](int t, int d, int r) {   // digit t of Vint(key, d) into its operand plane (f16, exact)
    *reinterpret_cast<uint16_t*>(vblk + t * (VP_BLOCK / 3) + tc5::canon_off(d, jr % VKEYS)) =
        __half_as_ushort(__int2half_rn(r));
  };
  if (j >= a.kv_hi) {
    for (int d = lane; d < DP; d += 32) {
#pragma unroll
      for (int q = 0; q < NSLICE; q++) store_tc(q, d, 0);
      if (vblk)
#pragma unroll
        for (int t = 0; t < 3; t++) store_v(t, d, 0);
    }
    return;
  }
  const int64_t row = ((int64_t)b * a.Hkv + hk) * a.Skv + j;
  int nf = 0;
  {
    const T* krow = (const T*)a.k + b * a.ks[0] + hk * a.ks[1] + (int64_t)j * a.ks[2];
    __shared__ int Fk_s[8];
    __shared__ unsigned char fit_s[8], lon_s[8];
    uint16_t* ks = p.ksl + row * NSLICE * DP;   // row-major slices: only the D = 256 kernel reads them
    row_slices<DT, DP>(krow, a.D,
                       [&](int q, int d, uint16_t v) {
                         if constexpr (DP == 256) ks[q * DP + d] = v;
                         store_tc(q, d, v);
                       },
                       &Fk_s[warp], &fit_s[warp], nf, lane, p.klo + row * NLO, &lon_s[warp]);
    __syncwarp();
    if (lane == 0) {
      const int lon = lon_s[warp] == LO_DEEP ? KLO_DEEP : (int)lon_s[warp];
      p.kmeta[row] = (Fk_s[warp] + 1024) | ((int)fit_s[warp] << 16) | (lon << 17);
    }
  }
  if (p.do_v) {
    const T* vrow = (const T*)a.v + b * a.vs[0] + hk * a.vs[1] + (int64_t)j * a.vs[2];
    const int* vcol = p.vcol + ((int64_t)b * a.Hkv + hk) * DP;
#pragma unroll
    for (int tv = 0; tv < NW; tv++) {
      const int d = lane + 32 * tv;
      const uint32_t u = d < a.D ? In<DT>::bits(vrow, d) : 0u;
      bool fit = true;
      int X = 0;
      if (nonfinite_bits(u)) {
        nf |= ST_NONFINITE;
      } else {
        const Split s = split_f32(u);
        if (s.mant) {
          const int sh = (min(max(vcol[d], 1), 254) - 149) - s.lsb;   // >= 1
          if (sh < 32) {
            X = (int)(s.mant >> sh);
            fit = (s.mant & ((1u << sh) - 1u)) == 0u;
          } else {
            fit = false;
          }
          if (!fit) X = 0;
          if (s.neg) X = -X;
        }
      }
      p.vint[row * DP + d] = X;
      if (vblk) {   // balanced base-256 digits: X = r0 + 256 r1 + 65536 r2, |r_t| <= 128
        int r0 = X & 255;
        if (r0 >= 128) r0 -= 256;
        const int X1 = (X - r0) >> 8;
        int r1 = X1 & 255;
        if (r1 >= 128) r1 -= 256;
        const int r2 = (X1 - r1) >> 8;
        store_v(0, d, r0);
        store_v(1, d, r1);
        store_v(2, d, r2);
      }
      const uint32_t bad = __ballot_sync(0xFFFFFFFFu, !fit);
      if (lane == 0) p.vbad[row * NW + tv] = bad;
    }
  }
  report(a.status, nf);
}

static size_t vtc_bytes(int B, int Hkv, int Skv, int dp) {
  if (dp != 128) return 0;
  const size_t ntk = (size_t)(Skv + KTILE - 1) / KTILE;
  return (size_t)B * Hkv * ntk * (KTILE / VKEYS) * VP_BLOCK;
}

static size_t spill_bytes(int dp) { return dp == 128 ? (size_t)SPILL_SLOTS * spill_slot_words(dp) * 8 : 0; }

static size_t ktc_bytes(int B, int Hkv, int Skv, int dp) {
  const size_t ntk = (size_t)(Skv + KTILE - 1) / KTILE;
  return (size_t)B * Hkv * ntk * (dp / 16) * KT_BLOCK;
}

size_t kv_prep_bytes(int B, int Hkv, int Skv, int D) {
  const int dp = D <= 128 ? 128 : 256;   // the kernels' padded width (attn_kernels.cu)
  const size_t rows = (size_t)B * Hkv * Skv;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return up(dp == 256 ? rows * NSLICE * dp * 2 : 0) + up(rows * 4) + up(rows * NLO * 8) + up((size_t)B * Hkv * dp * 4) +
         up(rows * dp * 4) + up(rows * (dp / 32) * 4) + up(ktc_bytes(B, Hkv, Skv, dp)) + up(vtc_bytes(B, Hkv, Skv, dp)) +
         up(spill_bytes(dp));
}

KvPrep kv_prep_layout(void* ws, int B, int Hkv, int Skv, int D, int do_v) {
  const int dp = D <= 128 ? 128 : 256;   // the kernels' padded width (attn_kernels.cu)
  const size_t rows = (size_t)B * Hkv * Skv;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  char* c = (char*)ws;
  KvPrep p;
  p.DP = dp;
  p.do_v = do_v;
  p.ksl = (uint16_t*)c;   // row-major key slices, for the D = 256 kernel only
  c += up(dp == 256 ? rows * NSLICE * dp * 2 : 0);
  p.kmeta = (int*)c;
  c += up(rows * 4);
  p.klo = (int2*)c;
  c += up(rows * NLO * 8);
  p.vcol = (int*)c;
  c += up((size_t)B * Hkv * dp * 4);
  p.vint = (int*)c;
  c += up(rows * dp * 4);
  p.vbad = (uint32_t*)c;
  c += up(rows * (dp / 32) * 4);
  p.ktc = (unsigned char*)c;
  p.ntk = (Skv + KTILE - 1) / KTILE;
  c += up(ktc_bytes(B, Hkv, Skv, dp));
  p.vtc = dp == 128 ? (unsigned char*)c : nullptr;
  c += up(vtc_bytes(B, Hkv, Skv, dp));
  p.spill = dp == 128 ? (long long*)c : nullptr;
  return p;
}

template <int DT, int DP>
static cudaError_t launch_prep_t(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  const int n = a.kv_hi - a.kv_lo;
  if (p.do_v) {   // the column exponents are read even when the range is empty
    cudaError_t e = cudaMemsetAsync(p.vcol, 0, sizeof(int) * (size_t)a.B * a.Hkv * DP, st);
    if (e != cudaSuccess) return e;
    if (n > 0) prep_vcol_kernel<DT><<<dim3((n + VCOL_ROWS - 1) / VCOL_ROWS, a.Hkv, a.B), 256, 0, st>>>(a, p);
  }
  const int padded = ((n + KTILE - 1) / KTILE) * KTILE;
  if (n > 0) prep_kv_kernel<DT, DP><<<dim3(padded / 8, a.Hkv, a.B), 256, 0, st>>>(a, p);
  return cudaGetLastError();
}

cudaError_t launch_kv_prep(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  if (a.dtype == 0) {
    if (p.DP == 64) return launch_prep_t<0, 64>(a, p, st);
    if (p.DP == 128) return launch_prep_t<0, 128>(a, p, st);
    return launch_prep_t<0, 256>(a, p, st);
  }
  if (p.DP == 64) return launch_prep_t<1, 64>(a, p, st);
  if (p.DP == 128) return launch_prep_t<1, 128>(a, p, st);
  return launch_prep_t<1, 256>(a, p, st);
}

}  // namespace detattn
