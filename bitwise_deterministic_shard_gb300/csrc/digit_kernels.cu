// Digit kernels for sm_103a: compose (max / add), canonical normalization, finalize.
//
// Page "det-attn", sections "Method" and "API": KV shards compose by an elementwise max of
// the rowmax and an int64 add of digit arrays; finalize composes digits into the f32
// output.  The contract's finalize: o = RN32(RN64(RN64(NUM) / RN64(DEN))).  All three are
// HBM-bound streaming kernels: grids cover the arrays with 16-byte accesses where aligned.
#include "numerics.cuh"
#include "divide.cuh"
#include "attn_kernels.h"

namespace detattn {

static int grid_for(int64_t n, int per_thread) {
  int64_t blocks = (n + 256LL * per_thread - 1) / (256LL * per_thread);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t cap = (int64_t)sms * 8;
  return (int)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

__global__ void compose_max_kernel(float* __restrict__ dst, const float* __restrict__ src, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    float a = dst[i], b = src[i];
    float m = (b > a || a != a) ? b : a;   // max; a NaN never wins
    if (m == 0.0f) m = __int_as_float(0);  // -0 -> +0
    dst[i] = m;
  }
}

__global__ void compose_add_kernel(long long* __restrict__ dst, const long long* __restrict__ src, int64_t n) {
  const int64_t n2 = n / 2;
  longlong2* d2 = reinterpret_cast<longlong2*>(dst);
  const longlong2* s2 = reinterpret_cast<const longlong2*>(src);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n2; i += (int64_t)gridDim.x * blockDim.x) {
    longlong2 a = d2[i], b = __ldg(s2 + i);
    a.x += b.x;
    a.y += b.y;
    d2[i] = a;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && (n & 1)) dst[n - 1] += src[n - 1];
}

// canonical form of accumulators laid out [nrows][ndig][inner]
template <int ND>
__global__ void normalize_kernel(long long* __restrict__ dg, int64_t nrows, int64_t inner, int* status) {
  const int64_t n = nrows * inner;
  int bad = 0;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / inner, c = t % inner;
    long long* p = dg + r * ND * inner + c;
    long long a[ND];
#pragma unroll
    for (int k = 0; k < ND; k++) a[k] = p[k * inner];
    // carries in radix 2^32; the top digit keeps the sign
#pragma unroll
    for (int k = 0; k < ND - 1; k++) {
      long long cy = a[k] >> 32;
      a[k] -= cy * 4294967296ll;
      a[k + 1] += cy;
    }
    if (a[ND - 1] > (1ll << 62) || a[ND - 1] < -(1ll << 62)) bad = ST_HEADROOM;
#pragma unroll
    for (int k = 0; k < ND; k++) p[k * inner] = a[k];
  }
  report(status, bad);
}

// One warp per group of FIN_ROWS rows.  Lanes 0 .. FIN_ROWS - 1 first round one row's DEN to
// binary64 and prepare its reciprocal (idiv::Divisor); the warp then walks the group's rows,
// each lane over the columns d = lane, lane + 32, ..., with coalesced loads of the NUM digit
// planes.  RN64(NUM) / RN64(DEN) and the final RN32 run on the integer pipe; a row whose DEN
// is zero or negative (outside the contract: no key, or corrupted digits) takes the binary64
// division so that 0/0 and x/0 give IEEE's NaN and infinities.
constexpr int FIN_ROWS = 8;

__device__ __noinline__ float finalize_slow(const long long* __restrict__ num, const long long* __restrict__ den,
                                            int D) {
  long long a[NUM_NDIG];
#pragma unroll
  for (int k = 0; k < NUM_NDIG; k++) a[k] = num[(int64_t)k * D];
  long long e[DEN_NDIG];
#pragma unroll
  for (int k = 0; k < DEN_NDIG; k++) e[k] = den[k];
  bool sn, sd;
  uint64_t mn, md;
  int en, ed;
  const double n64 = idiv::digits_split_rn64<NUM_NDIG>(a, NUM_E0, sn, mn, en) ? idiv::make_f64(sn, mn, en) : 0.0;
  const double d64 = idiv::digits_split_rn64<DEN_NDIG>(e, DEN_E0, sd, md, ed) ? idiv::make_f64(sd, md, ed) : 0.0;
  return __double2float_rn(__ddiv_rn(n64, d64));
}

__global__ void __launch_bounds__(256) finalize_kernel(const long long* __restrict__ num,
                                                       const long long* __restrict__ den, int64_t rows, int D,
                                                       float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t ngroups = (rows + FIN_ROWS - 1) / FIN_ROWS;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < ngroups; g += nwarps) {
    const int64_t r0 = g * FIN_ROWS;
    uint64_t dn = 0, dv = 0;
    int de = 0, slow = 1;
    if (lane < FIN_ROWS && r0 + lane < rows) {
      long long e[DEN_NDIG];
#pragma unroll
      for (int k = 0; k < DEN_NDIG; k++) e[k] = __ldg(den + (r0 + lane) * DEN_NDIG + k);
      bool neg;
      uint64_t m;
      int ee;
      if (idiv::digits_split_rn64<DEN_NDIG>(e, DEN_E0, neg, m, ee) && !neg) {
        const idiv::Divisor Dv = idiv::make_divisor(m, ee);
        dn = Dv.dn;
        dv = Dv.v;
        de = Dv.e;
        slow = 0;
      }
    }
    const int nr = (int)(rows - r0 < FIN_ROWS ? rows - r0 : FIN_ROWS);
    for (int j = 0; j < nr; j++) {
      idiv::Divisor Dv;
      Dv.dn = __shfl_sync(0xFFFFFFFFu, dn, j);
      Dv.v = __shfl_sync(0xFFFFFFFFu, dv, j);
      Dv.e = __shfl_sync(0xFFFFFFFFu, de, j);
      const int sl = __shfl_sync(0xFFFFFFFFu, slow, j);
      const int64_t r = r0 + j;
      const long long* nr0 = num + r * NUM_NDIG * D;
      for (int c = lane; c < D; c += 32) {
        float o;
        if (sl) {
          o = finalize_slow(nr0 + c, den + r * DEN_NDIG, D);
        } else {
          long long a[NUM_NDIG];
#pragma unroll
          for (int k = 0; k < NUM_NDIG; k++) a[k] = __ldg(nr0 + (int64_t)k * D + c);
          bool neg;
          uint64_t m;
          int en;
          o = 0.0f;   // RN64(NUM) = +0: +0 / DEN = +0
          if (idiv::digits_split_rn64<NUM_NDIG>(a, NUM_E0, neg, m, en))
            o = __uint_as_float(idiv::div_rn32(m, en, Dv, neg));
        }
        out[r * D + c] = o;
      }
    }
  }
}

cudaError_t launch_compose_max(float* dst, const float* src, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  compose_max_kernel<<<grid_for(n, 4), 256, 0, st>>>(dst, src, n);
  return cudaGetLastError();
}

cudaError_t launch_compose_add(long long* dst, const long long* src, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  compose_add_kernel<<<grid_for((n + 1) / 2, 4), 256, 0, st>>>(dst, src, n);
  return cudaGetLastError();
}

cudaError_t launch_normalize(long long* dg, int64_t nrows, int ndig, int64_t inner, int* status, cudaStream_t st) {
  const int64_t n = nrows * inner;
  if (n <= 0) return cudaSuccess;
  if (ndig == NUM_NDIG)
    normalize_kernel<NUM_NDIG><<<grid_for(n, 2), 256, 0, st>>>(dg, nrows, inner, status);
  else
    normalize_kernel<DEN_NDIG><<<grid_for(n, 2), 256, 0, st>>>(dg, nrows, inner, status);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const long long* num, const long long* den, int64_t rows, int D, float* out, int* status,
                            cudaStream_t st) {
  (void)status;
  const int64_t n = rows * D;
  if (n <= 0) return cudaSuccess;
  const int64_t warps = (rows + FIN_ROWS - 1) / FIN_ROWS;
  finalize_kernel<<<grid_for(warps * 32, 1), 256, 0, st>>>(num, den, rows, D, out);
  return cudaGetLastError();
}

}  // namespace detattn
