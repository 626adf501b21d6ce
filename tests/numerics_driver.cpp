// Host driver for the device numerics of the CUDA path (csrc/numerics.cuh, compiled for the
// host through cuda_host_shim.h): reads raw inputs from stdin, writes raw outputs to stdout.
//   mode 0: binary32 x        -> exp32_det(x), exp32_det_nb(x), p 2^k from exp32_det_poly (bits)
//   mode 1: (int64 T, int32 F) -> cr32_scaled(T, F), cr32_scaled_nb(T, F) (bits), its special flag,
//           cr32_scaled_cvt(T, F) (bits), its special flag
//   mode 2: 15 int64 digits    -> digits_rn64<15>(digits, -320)            (binary64)
//   mode 3: 6 int64 digits     -> digits_rn64<6>(digits, -160)             (binary64)
//   mode 4: binary64 d         -> log64_det(d)                             (binary64)
//   mode 5: int32 X            -> slice4(X): four bf16 bit patterns
//   mode 6: 7 binary32 A_c     -> combine_diag: int64 sum_c 2^(7c) A_c
//   mode 7: (uint32 u, int32 F) -> hi26(u, F)
//   mode 8: records for dot_lo (see below)                                  (binary32 bits)
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>
#include "numerics.cuh"
#include "score_tc.cuh"
using namespace detattn;

template <class T>
static std::vector<T> read_all() {
  std::vector<T> v;
  T x;
  while (fread(&x, sizeof x, 1, stdin) == 1) v.push_back(x);
  return v;
}

int main(int argc, char** argv) {
  const int mode = atoi(argv[1]);
  if (mode == 0) {
    for (float x : read_all<float>()) {
      // third: p 2^k assembled from exp32_det_poly's p and k (the bits of p with k added to its
      // exponent) where k >= -125, else all ones
      uint32_t pk = 0xFFFFFFFFu;
      if (x == x && x >= -104.0f) {
        int k;
        const uint32_t pb = __float_as_uint(exp32_det_poly(x, k));
        if (k >= -125) pk = pb + ((uint32_t)k << 23);
      }
      const uint32_t r[3] = {__float_as_uint(exp32_det(x)), x != x ? 0u : __float_as_uint(exp32_det_nb(x)), pk};
      fwrite(r, 4, 3, stdout);
    }
  } else if (mode == 1) {
    const std::vector<long long> in = read_all<long long>();   // pairs (T, F)
    for (size_t i = 0; i + 1 < in.size(); i += 2) {
      bool sp = false, sc = false;
      const int F = (int)in[i + 1];
      const uint32_t nb = __float_as_uint(cr32_scaled_nb(in[i], F, sp));
      const uint32_t cv = __float_as_uint(cr32_scaled_cvt(in[i], F, sc));
      const uint32_t r[5] = {__float_as_uint(cr32_scaled(in[i], F)), nb, sp ? 1u : 0u, cv, sc ? 1u : 0u};
      fwrite(r, 4, 5, stdout);
    }
  } else if (mode == 2 || mode == 3) {
    const std::vector<long long> in = read_all<long long>();
    const int n = mode == 2 ? 15 : 6;
    for (size_t i = 0; i + n <= in.size(); i += n) {
      double r;
      if (mode == 2) {
        long long a[15];
        for (int k = 0; k < 15; k++) a[k] = in[i + k];
        r = digits_rn64<15>(a, -320);
      } else {
        long long a[6];
        for (int k = 0; k < 6; k++) a[k] = in[i + k];
        r = digits_rn64<6>(a, -160);
      }
      fwrite(&r, 8, 1, stdout);
    }
  } else if (mode == 4) {
    for (double d : read_all<double>()) {
      const double r = log64_det(d);
      fwrite(&r, 8, 1, stdout);
    }
  } else if (mode == 5) {
    for (int X : read_all<int>()) {
      uint16_t s[NSLICE];
      slice4(X, s);
      fwrite(s, 2, NSLICE, stdout);
    }
  } else if (mode == 6) {
    const std::vector<float> in = read_all<float>();
    for (size_t i = 0; i + NDIAG <= in.size(); i += NDIAG) {
      float acc[NDIAG][1];
      for (int c = 0; c < NDIAG; c++) acc[c][0] = in[i + c];
      const long long T = combine_diag<1>(acc, 0);
      fwrite(&T, 8, 1, stdout);
    }
  } else if (mode == 7) {
    const std::vector<int> in = read_all<int>();
    for (size_t i = 0; i + 1 < in.size(); i += 2) {
      const int r = hi26((uint32_t)in[i], in[i + 1]);
      fwrite(&r, 4, 1, stdout);
    }
  } else if (mode == 8) {
    // record: int32 D, Fq, Fk, nq, nk; int64 Thh; D binary32 q; D binary32 k; nq (d, lo); nk (d, lo)
    const std::vector<int> in = read_all<int>();
    size_t i = 0;
    while (i + 7 <= in.size()) {
      const int D = in[i], Fq = in[i + 1], Fk = in[i + 2], nq = in[i + 3], nk = in[i + 4];
      long long Thh;
      memcpy(&Thh, &in[i + 5], 8);
      i += 7;
      const float* q = reinterpret_cast<const float*>(&in[i]);
      const float* k = reinterpret_cast<const float*>(&in[i + D]);
      i += 2 * D;
      const int2* ql = reinterpret_cast<const int2*>(&in[i]);
      i += 2 * nq;
      const int2* kl = reinterpret_cast<const int2*>(&in[i]);
      i += 2 * nk;
      const uint32_t r = __float_as_uint(dot_lo<0>(Thh, q, Fq, ql, nq, k, Fk, kl, nk));
      fwrite(&r, 4, 1, stdout);
    }
  }
  return 0;
}
