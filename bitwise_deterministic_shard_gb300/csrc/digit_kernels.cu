// Digit kernels for sm_103a: compose (max / add), canonical normalization, finalize.
//
// Page "det-attn", sections "Method" and "API": KV shards compose by an elementwise max of
// the rowmax and an int64 add of digit arrays; finalize composes digits into the f32
// output.  The contract's finalize: o = RN32(RN64(RN64(NUM) / RN64(DEN))).  All three are
// HBM-bound streaming kernels: grids cover the arrays with 16-byte accesses where aligned.
#include "numerics.cuh"
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

// one thread per output element; DEN is shared by the D threads of a row
__global__ void finalize_kernel(const long long* __restrict__ num, const long long* __restrict__ den, int64_t rows,
                                int D, float* __restrict__ out) {
  const int64_t n = rows * D;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / D;
    const int d = (int)(t % D);
    long long a[NUM_NDIG];
    const long long* p = num + r * NUM_NDIG * D + d;
#pragma unroll
    for (int k = 0; k < NUM_NDIG; k++) a[k] = __ldg(p + (int64_t)k * D);
    long long e[DEN_NDIG];
#pragma unroll
    for (int k = 0; k < DEN_NDIG; k++) e[k] = __ldg(den + r * DEN_NDIG + k);
    const double n64 = digits_rn64<NUM_NDIG>(a, NUM_E0);
    const double d64 = digits_rn64<DEN_NDIG>(e, DEN_E0);
    out[t] = __double2float_rn(__ddiv_rn(n64, d64));
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
  finalize_kernel<<<grid_for(n, 2), 256, 0, st>>>(num, den, rows, D, out);
  return cudaGetLastError();
}

}  // namespace detattn
