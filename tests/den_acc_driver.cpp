// Host driver for the exact DEN accumulation of the cross-entropy denominator kernel
// (den_acc.cuh): reads weights as binary32 bit patterns (one per line, a blank line ends a
// sequence), accumulates each sequence, prints its six digits.
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include "den_acc.cuh"
using namespace detattn;

int main() {
  DenAcc A;
  den_init(A);
  char line[64];
  bool any = false;
  long n = 0;
  auto emit = [&]() {
    den_flush(A);
    for (int k = 0; k < 6; k++) printf("%lld%c", A.d[k], k == 5 ? '\n' : ' ');
    den_init(A);
    any = false;
  };
  while (fgets(line, sizeof line, stdin)) {
    if (line[0] == '\n') {
      emit();
      continue;
    }
    if (++n % 8 == 0) den_guard(A);   // the kernel guards once per 16-byte vector (<= 8 weights)
    den_add(A, (uint32_t)strtoul(line, nullptr, 10));
    any = true;
  }
  if (any) emit();
  return 0;
}
