// Host driver for the device numerics of the CUDA path (csrc/numerics.cuh, compiled for the
// host through cuda_host_shim.h): reads raw inputs from stdin, writes raw outputs to stdout.
//   mode 0: binary32 x        -> exp32_det(x), exp32_det_nb(x)            (binary32 bits)
//   mode 1: (int64 T, int32 F) -> cr32_scaled(T, F), cr32_scaled_nb(T, F) (bits), special flag
//   mode 2: 15 int64 digits    -> digits_rn64<15>(digits, -320)            (binary64)
//   mode 3: 6 int64 digits     -> digits_rn64<6>(digits, -160)             (binary64)
//   mode 4: binary64 d         -> log64_det(d)                             (binary64)
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "numerics.cuh"
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
      const uint32_t r[2] = {__float_as_uint(exp32_det(x)), x != x ? 0u : __float_as_uint(exp32_det_nb(x))};
      fwrite(r, 4, 2, stdout);
    }
  } else if (mode == 1) {
    const std::vector<long long> in = read_all<long long>();   // pairs (T, F)
    for (size_t i = 0; i + 1 < in.size(); i += 2) {
      bool sp = false;
      const int F = (int)in[i + 1];
      const uint32_t r[3] = {__float_as_uint(cr32_scaled(in[i], F)), __float_as_uint(cr32_scaled_nb(in[i], F, sp)),
                             sp ? 1u : 0u};
      fwrite(r, 4, 3, stdout);
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
  }
  return 0;
}
