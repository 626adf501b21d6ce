// Host driver for the integer-pipe division helpers of the CUDA kernels (divide.cuh): prints
// seeded random and edge-case inputs with the helpers' results, which test_divide_host.py
// checks against exact rational arithmetic.
#include <cstdio>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cstdlib>
#include "divide.cuh"
#include "fdiv.cuh"
using namespace detattn::idiv;
static uint64_t s = 88172645463325252ull;
static uint64_t rnd() { s ^= s << 13; s ^= s >> 7; s ^= s << 17; return s; }
int main(int argc, char** argv) {
  int mode = atoi(argv[1]); long n = atol(argv[2]);
  if (mode == 0) {   // div_rn64 + rn32
    for (long i = 0; i < n; i++) {
      uint64_t mn = (rnd() >> 11) | (1ull << 52), md = (rnd() >> 11) | (1ull << 52);
      int pick = rnd() % 8;
      if (pick == 0) md = 1ull << 52;
      if (pick == 1) mn = md;
      if (pick == 2) mn = (1ull << 53) - 1 - (rnd() % 4);
      if (pick == 3) md = (1ull << 53) - 1 - (rnd() % 4);
      if (pick == 4) { md = (1ull << 52) | (rnd() % 8); mn = md * 3 / 2; if (mn >> 53) mn >>= 1; mn |= 1ull<<52; }
      int en = (int)(rnd() % 600) - 300, ed = (int)(rnd() % 300) - 150;
      Divisor D = make_divisor(md, ed);
      uint64_t q; int E; div_rn64(mn, en, D, q, E);
      uint32_t f = rn32_bits(q, E, rnd() & 1);
      printf("%llu %d %llu %d %llu %d %u\n", (unsigned long long)mn, en, (unsigned long long)md, ed, (unsigned long long)q, E, f);
    }
  } else if (mode == 1) {   // rn32 on random q53 and wide exponents
    for (long i = 0; i < n; i++) {
      uint64_t q = (rnd() >> 11) | (1ull << 52);
      if (rnd() % 4 == 0) q = (q & ~((1ull << 29) - 1)) | (1ull << 28) | ((rnd()%2) ? 0 : 1);
      int E = (int)(rnd() % 500) - 260;
      bool neg = rnd() & 1;
      printf("%llu %d %d %u\n", (unsigned long long)q, E, (int)neg, rn32_bits(q, E, neg));
    }
  } else if (mode == 2) {   // digits
    for (long i = 0; i < n; i++) {
      long long a[15];
      int kind = rnd() % 4;
      for (int k = 0; k < 15; k++) {
        long long v = (long long)(rnd() >> 30) - (1ll << 33);
        if (kind == 1 && k < 13) v = (rnd() % 3 == 0) ? (long long)(rnd() >> 32) : 0;
        if (kind == 2) v = (k == (int)(rnd() % 15)) ? (long long)(rnd() >> 32) : 0;
        if (kind == 3 && k > 10) v = 0;
        a[k] = v;
      }
      if (kind == 1) { a[13] = 0; a[14] = (rnd() % 2) ? 1 : -1; }
      if (kind == 2) a[14] = 0;
      for (int k = 0; k < 15; k++) printf("%lld ", a[k]);
      bool neg; uint64_t m; int e;
      bool nz = digits_split_rn64<15>(a, -320, neg, m, e);
      printf("| %d %d %llu %d\n", (int)nz, (int)neg, (unsigned long long)m, e);
    }
  } else if (mode == 4) {   // the binary32-numerator division against the generic one
    for (long i = 0; i < n; i++) {
      uint32_t b = (uint32_t)rnd() & 0x7FFFFFFFu;
      if ((b >> 23) == 0xFF || b == 0) b = 0x3F800000u;
      if (i % 5 == 0) b &= 0x807FFFFFu;   // subnormal
      if (b == 0) b = 1;
      uint64_t md = (rnd() >> 11) | (1ull << 52);
      if (i % 7 == 0) md = 1ull << 52;
      int ed = (int)(rnd() % 120) - 60;
      Divisor D = make_divisor(md, ed);
      uint32_t mw; int ew; split_f32_24(b, mw, ew);
      uint64_t m53, q; int e53, E;
      split_f32_53(b, m53, e53);
      div_rn64(m53, e53, D, q, E);
      printf("%u %llu %d %u %u\n", b, (unsigned long long)md, ed, div_f32_rn32(mw, ew, D), rn32_bits(q, E, false));
    }
  } else if (mode == 5) {   // RN64 of three lazy radix-2^32 digits as one 128-bit integer
    for (long i = 0; i < n; i++) {
      long long d[3];
      int kind = rnd() % 4;
      for (int k = 0; k < 3; k++) d[k] = (long long)(rnd() >> 2) - (1ll << 61);   // |d| < 2^62
      if (kind == 1) d[2] = 0;
      if (kind == 2) { d[1] = 0; d[2] = 0; d[0] = (long long)(rnd() >> 40) - (1ll << 23); }
      if (kind == 3) { d[0] = (long long)(rnd() % 3) << 40; d[1] = -(long long)(rnd() % 2); d[2] = (long long)(rnd() % 2); }
      if (i == 0) { d[0] = 0; d[1] = 0; d[2] = 0; }
      int lsb = (int)(rnd() % 200) - 180;
      __int128 X = (__int128)d[0] + (__int128)d[1] * ((__int128)1 << 32) + (__int128)d[2] * ((__int128)1 << 64);
      bool neg = false; uint64_t m = 0; int e = 0;
      bool nz = i128_split_rn64(X, lsb, neg, m, e);
      printf("%lld %lld %lld %d | %d %d %llu %d\n", d[0], d[1], d[2], lsb, (int)nz, (int)neg, (unsigned long long)m, e);
    }
  } else if (mode == 6) {   // the direct binary32 quotient against the exact one
    for (long i = 0; i < n; i++) {
      uint32_t b;
      uint64_t md = (rnd() >> 11) | (1ull << 52);
      int ed = (int)(rnd() % 40) - 8;
      const int kind = (int)(i % 4);
      if (kind == 0) {   // weights exp-like in (0, 1]: exponent spread over [-40, 0]
        b = ((uint32_t)(127 - (int)(rnd() % 41)) << 23) | ((uint32_t)rnd() & 0x7FFFFFu);
      } else if (kind == 1) {   // any positive normal or subnormal binary32 (wide exponents)
        b = (uint32_t)rnd() & 0x7FFFFFFFu;
        if ((b >> 23) == 0xFF || b == 0) b = 0x3F800000u;
        ed = (int)(rnd() % 400) - 200;
      } else if (kind == 2) {   // quotients within about 2^-53 of a binary32 half-way point
        b = ((uint32_t)(120 + (int)(rnd() % 8)) << 23) | ((uint32_t)rnd() & 0x7FFFFFu);
        const uint32_t mw = (b & 0x7FFFFFu) | 0x800000u;
        const uint64_t odd = ((rnd() >> 40) & 0x7FFFFFull) * 2 + 1 + (1ull << 24);   // 2M + 1, 25 bits
        unsigned __int128 num = (unsigned __int128)(2ull * mw) << 52;
        uint64_t q = (uint64_t)(num / odd);
        if (!(q >> 52)) q = (uint64_t)((num << 1) / odd);
        md = q + (uint64_t)(rnd() % 3) - 1;
        if (!(md >> 52) || (md >> 53)) md = q;
      } else {   // power-of-two and all-ones divisors
        b = ((uint32_t)(100 + (int)(rnd() % 28)) << 23) | ((uint32_t)rnd() & 0x7FFFFFu);
        md = (rnd() & 1) ? (1ull << 52) : ((1ull << 53) - 1);
      }
      Divisor D = make_divisor(md, ed);
      uint32_t mw; int ew; split_f32_24(b, mw, ew);
      bool ok = false;
      const uint32_t fast = div_f32_rn32_direct(mw, ew, D, ok);
      printf("%u %llu %d %d %u %u\n", b, (unsigned long long)md, ed, (int)ok, fast, div_f32_rn32(mw, ew, D));
    }
  } else if (mode == 7) {   // the direct binary32 rounding of a binary64 quotient against the exact one
    for (long i = 0; i < n; i++) {
      uint64_t mn = (rnd() >> 11) | (1ull << 52), md = (rnd() >> 11) | (1ull << 52);
      int en = (int)(rnd() % 120) - 60, ed = (int)(rnd() % 120) - 60;
      const int kind = (int)(i % 4);
      if (kind == 1) {   // wide exponents: subnormal and overflowing quotients
        en = (int)(rnd() % 600) - 300;
        ed = (int)(rnd() % 300) - 150;
      } else if (kind == 2) {   // quotients within about 2^-53 of a binary32 half-way point
        const uint64_t odd = ((rnd() >> 40) & 0x7FFFFFull) * 2 + 1 + (1ull << 24);   // 2M + 1, 25 bits
        unsigned __int128 num = (unsigned __int128)mn << 25;
        uint64_t q = (uint64_t)(num / odd);
        while (q >> 53) q >>= 1;
        while (!(q >> 52)) q <<= 1;
        md = q + (uint64_t)(rnd() % 5) - 2;
        if (!(md >> 52) || (md >> 53)) md = q;
      } else if (kind == 3) {   // exact quotients: power-of-two divisors, equal mantissas
        if (rnd() & 1) md = 1ull << 52; else md = mn;
      }
      Divisor D = make_divisor(md, ed);
      uint64_t q; int E; div_rn64(mn, en, D, q, E);
      const bool neg = rnd() & 1;
      bool ok = false;
      const uint32_t fast = div_rn64_rn32_direct(mn, en, D, neg, ok);
      printf("%llu %d %llu %d %d %d %u %u\n", (unsigned long long)mn, en, (unsigned long long)md, ed, (int)neg, (int)ok,
             fast, rn32_bits(q, E, neg));
    }
  } else if (mode == 8) {   // the FP32-pipe quotient with its certificate against the exact one
    auto f64 = [](uint64_t b) { double d; memcpy(&d, &b, 8); return d; };
    auto b64 = [](double d) { uint64_t b; memcpy(&b, &d, 8); return b; };
    auto f32 = [](uint32_t b) { float f; memcpy(&f, &b, 4); return f; };
    for (long i = 0; i < n; i++) {
      const int kind = (int)(i % 4);
      uint32_t pb = (uint32_t)(126 + (int)(rnd() & 1)) << 23 | ((uint32_t)rnd() & 0x7FFFFFu);   // p in [0.5, 2)
      double d;
      if (kind == 0) {          // denominators of ordinary size, [1, 2^20)
        d = f64(((uint64_t)(1023 + rnd() % 20) << 52) | (rnd() >> 12));
      } else if (kind == 1) {   // the whole accepted range [2^-60, 2^60] and a little outside it
        d = f64(((uint64_t)(1023 - 62 + rnd() % 125) << 52) | (rnd() >> 12));
      } else if (kind == 2) {   // quotients within about 2^-53 of a binary32 half-way point
        const int E = -(int)(rnd() % 20);
        const uint64_t mid = (((rnd() >> 40) & 0x7FFFFFull) | 0x800000ull) * 2 + 1;   // 25 bits, odd
        const double M = std::ldexp((double)mid, E - 24);
        d = f64(b64(f32(pb) / M) + (rnd() % 5) - 2);
      } else {                  // d a binary32 (d_lo = 0), a power of two, or p itself
        const int c = (int)(rnd() % 3);
        d = c == 0 ? (double)f32(((uint32_t)(127 + rnd() % 17) << 23) | ((uint32_t)rnd() & 0x7FFFFFu))
                   : c == 1 ? std::ldexp(1.0, (int)(rnd() % 41) - 20) : (double)f32(pb);
      }
      detattn::fdiv::FpDivisor F;
      bool ok = false;
      uint32_t fast = 0;
      if (detattn::fdiv::make_fp_divisor(d, F)) fast = detattn::fdiv::div_rn32(f32(pb), F, ok);
      uint64_t md; int ed; split_f64(b64(d), md, ed);
      Divisor D = make_divisor(md, ed);
      uint32_t mw; int ew; split_f32_24(pb, mw, ew);
      printf("%u %llu %d %u %u\n", pb, (unsigned long long)b64(d), (int)ok, fast, div_f32_rn32(mw, ew, D));
    }
  } else if (mode == 3) {   // f32 split
    for (long i = 0; i < n; i++) {
      uint32_t b = (uint32_t)rnd() & 0x7FFFFFFFu;
      if ((b >> 23) == 0xFF) b &= 0x7F7FFFFFu;
      if (i < 30) b = (uint32_t)(1u << i);
      if (b == 0) b = 1;
      uint64_t m; int e; split_f32_53(b, m, e);
      printf("%u %llu %d\n", b, (unsigned long long)m, e);
    }
  }
}
