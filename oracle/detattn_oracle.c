/*
 * Exact CPU reference for the order-invariant softmax reduction.
 *
 * TEST INFRASTRUCTURE ONLY: this is the oracle.  The test-suite, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product library never links or calls it, and
 * it shares no code with the CUDA path.
 *
 * What it computes (page "det-attn", sections "Method" and "API"; page
 * "det-cross-entropy", sections "Usage", "API" and "Method"):
 *   s_ij    = RN32(scale32 * RN32(sum_d q_id k_jd))        exact dot, rounded once
 *   m_i     = max_{j valid} s_ij  (-0 -> +0, empty -> -inf)  combine by max
 *   w_ij    = exp32_det(RN32(s_ij - m_i))                    fixed binary32 routine
 *   NUM_id  = sum_j w_ij v_jd,  DEN_i = sum_j w_ij           exact (Kulisch), combine by add
 *   o_id    = RN32(RN64(RN64(NUM_id) / RN64(DEN_i)))
 *   DCE:  m_i = max_v x_iv; den_i = sum_v exp32_det(RN32(x_iv - m_i)) exact;
 *         loss_i = RN32(RN64(log64_det(RN64(den_i)) + RN64(m_i - x_{i,t_i}))).
 *
 * Arithmetic: every binary32 / binary64 operation below is a single IEEE operation in
 * round-to-nearest-even (the file must be compiled with -ffp-contract=off so that no
 * multiply-add is fused unless fmaf() is written); exact sums are held in a Kulisch
 * accumulator, an array of signed 64-bit words in radix 2^32 whose word 0 weighs 2^-320,
 * and rounded once by the routine kacc_round written from the IEEE definition.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* Kulisch accumulator                                                                   */
/* ------------------------------------------------------------------------------------ */
#define KW 20          /* words: weights 2^-320 .. 2^320 */
#define KBASE (-320)   /* exponent of word 0, bit 0 */

typedef struct { int64_t w[KW]; } kacc;

static void kacc_zero(kacc* a) { memset(a, 0, sizeof(*a)); }

/* add (neg ? -1 : +1) * mag * 2^lsb, mag < 2^49, lsb >= KBASE */
static void kacc_add(kacc* a, uint64_t mag, int neg, int lsb) {
  if (mag == 0) return;
  int pos = lsb - KBASE;
  int k = pos >> 5, sh = pos & 31;
  unsigned __int128 v = (unsigned __int128)mag << sh;
  int64_t c0 = (int64_t)(uint32_t)v, c1 = (int64_t)(uint32_t)(v >> 32), c2 = (int64_t)(uint32_t)(v >> 64);
  if (neg) { a->w[k] -= c0; a->w[k + 1] -= c1; a->w[k + 2] -= c2; }
  else     { a->w[k] += c0; a->w[k + 1] += c1; a->w[k + 2] += c2; }
}

/* carries: words 0..KW-2 into [0, 2^32), top word signed */
static void kacc_carry(kacc* a) {
  for (int k = 0; k < KW - 1; k++) {
    int64_t c = a->w[k] >> 32;              /* arithmetic shift (floor) */
    a->w[k] -= c * (int64_t)4294967296LL;
    a->w[k + 1] += c;
  }
}

/* canonical digits of a carried accumulator: digits 0..ndig-2 are words word0.., the top
 * digit folds every higher word in (top-down, so sign-extension words stay small).
 * Returns 1 if the value does not fit the digit range. */
static int kacc_store(const kacc* a0, int word0, int ndig, int64_t* out, int64_t stride) {
  kacc a = *a0;
  kacc_carry(&a);
  int bad = 0;
  for (int k = 0; k < word0; k++) if (a.w[k]) bad = 1;
  int64_t t = a.w[KW - 1];
  for (int k = KW - 2; k >= word0 + ndig - 1; k--) {
    if (t > ((int64_t)1 << 30) || t < -((int64_t)1 << 30)) bad = 1;
    t = t * (int64_t)4294967296LL + a.w[k];
  }
  for (int k = 0; k < ndig - 1; k++) out[k * stride] = a.w[word0 + k];
  out[(ndig - 1) * stride] = t;
  return bad;
}

static void flag(int* f) { __atomic_store_n(f, 1, __ATOMIC_RELAXED); }

/* sign and magnitude (32-bit words) of a carried accumulator */
static int kacc_mag(const kacc* a0, uint32_t m[KW]) {
  kacc a = *a0;
  kacc_carry(&a);
  int neg = a.w[KW - 1] < 0;
  if (neg) {
    for (int k = 0; k < KW; k++) a.w[k] = -a.w[k];
    kacc_carry(&a);
  }
  for (int k = 0; k < KW; k++) m[k] = (uint32_t)a.w[k];
  return neg;
}

static int mag_bit(const uint32_t m[KW], int i) { return (i >= 0 && i < 32 * KW) ? (m[i >> 5] >> (i & 31)) & 1 : 0; }

static int mag_any_below(const uint32_t m[KW], int i) { /* any bit at positions < i */
  if (i <= 0) return 0;
  int k = i >> 5, r = i & 31;
  for (int j = 0; j < k && j < KW; j++) if (m[j]) return 1;
  if (k < KW && r && (m[k] & ((1u << r) - 1u))) return 1;
  return 0;
}

/* Round the exact accumulated value to the binary format with `prec` significand bits
 * and minimum normal exponent `emin`, ties to even, gradual underflow; overflow above
 * 2^(emax+1) gives +-inf.  Exact zero gives +0. Result returned as a double (every
 * binary32 value is a double). */
static double kacc_round(const kacc* a, int prec, int emin, int emax) {
  uint32_t m[KW];
  int neg = kacc_mag(a, m);
  int top = -1;
  for (int k = KW - 1; k >= 0 && top < 0; k--)
    if (m[k]) for (int b = 31; b >= 0; b--) if ((m[k] >> b) & 1) { top = 32 * k + b; break; }
  if (top < 0) return 0.0;
  int e = top + KBASE;                        /* 2^e <= |value| < 2^(e+1) */
  int q = (e > emin ? e : emin) - (prec - 1); /* exponent of the last kept bit */
  int cut = q - KBASE;                        /* bit index of the last kept bit */
  uint64_t n = 0;
  for (int i = top; i >= cut && i >= 0; i--) n = (n << 1) | (uint64_t)mag_bit(m, i);
  if (cut < 0) n <<= -cut;                    /* value exact with room to spare */
  int rbit = mag_bit(m, cut - 1);
  int sticky = mag_any_below(m, cut - 1);
  if (rbit && (sticky || (n & 1))) n++;
  /* n <= 2^prec; result n * 2^q */
  int nbits = 0;
  for (uint64_t t = n; t; t >>= 1) nbits++;
  double r;
  if (n == 0) r = 0.0;
  else if (nbits + q > emax + 1) r = INFINITY;
  else r = ldexp((double)n, q);
  return neg ? -r : r;
}

static float kacc_rn32(const kacc* a) { return (float)kacc_round(a, 24, -126, 127); }
static double kacc_rn64(const kacc* a) { return kacc_round(a, 53, -1022, 1023); }

/* ------------------------------------------------------------------------------------ */
/* binary32 decode: x = (neg ? -1 : 1) * mant * 2^lsb exactly, mant < 2^24                */
/* ------------------------------------------------------------------------------------ */
static void f32_split(float x, uint64_t* mant, int* neg, int* lsb) {
  uint32_t u;
  memcpy(&u, &x, 4);
  *neg = (int)(u >> 31);
  uint32_t ex = (u >> 23) & 0xFF, fr = u & 0x7FFFFF;
  if (ex == 0) { *mant = fr; *lsb = -149; }
  else { *mant = fr | 0x800000u; *lsb = (int)ex - 150; }
}

static float load_elem(const void* base, int dtype, int64_t idx) {
  if (dtype == 0) return ((const float*)base)[idx];
  uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ------------------------------------------------------------------------------------ */
/* exp32_det: Cody-Waite reduction (Cody & Waite 1980) + degree-7 Taylor polynomial,       */
/* every operation binary32 RN; the constants are RN32 of their exact definitions.        */
/* ------------------------------------------------------------------------------------ */
static const float EXP_L2E = 0x1.715476p+0f;  /* RN32(log2 e) */
static const float EXP_C1 = 0x1.62e4p-1f;     /* ln 2 to 16 significant bits */
static const float EXP_C2 = 0x1.7f7d1cp-20f;  /* RN32(ln 2 - C1) */
static const float EXP_T[8] = {1.0f, 1.0f, 0x1p-1f, 0x1.555556p-3f, 0x1.555556p-5f,
                               0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f}; /* RN32(1/n!) */

float or_exp32_det(float x) {
  if (x != x) return x;
  if (x < -104.0f) return 0.0f;
  float t = x * EXP_L2E;
  float kf = nearbyintf(t);          /* ties to even (default rounding mode) */
  int k = (int)kf;
  float r1 = fmaf(-kf, EXP_C1, x);
  float r = fmaf(-kf, EXP_C2, r1);
  float p = EXP_T[7];
  for (int n = 6; n >= 0; n--) p = fmaf(p, r, EXP_T[n]);
  /* RN32(p * 2^k): the double product is exact, the conversion rounds once */
  return (float)((double)p * ldexp(1.0, k));
}

/* ------------------------------------------------------------------------------------ */
/* log64_det: reduction to [sqrt(1/2), sqrt(2)], atanh series in u = (f-1)/(f+1) with ten */
/* terms after the first, then e*ln2 as a two-part constant; binary64 RN, nothing fused.  */
/* ------------------------------------------------------------------------------------ */
static const double LOG_SQRT2 = 0x1.6a09e667f3bcdp+0;  /* RN64(sqrt 2) */
static const double LOG_LN2_HI = 0x1.62e42fefa38p-1;   /* ln 2 truncated to 42 bits */
static const double LOG_LN2_LO = 0x1.ef35793c7673p-45; /* RN64(ln 2 - LN2_HI) */

double or_log64_det(double d) {
  int e;
  double f = frexp(d, &e);   /* d = f 2^e, f in [0.5, 1) */
  f = f * 2.0;
  e = e - 1;
  if (f > LOG_SQRT2) { f = f * 0.5; e = e + 1; }
  double a = f - 1.0;
  double b = f + 1.0;
  double u = a / b;
  double u2 = u * u;
  double p = 1.0 / 21.0;
  for (int n = 9; n >= 1; n--) {
    double t = p * u2;
    p = t + 1.0 / (double)(2 * n + 1);
  }
  double t1 = u2 * p;
  double t2 = u * t1;
  double lf = (u + t2) * 2.0;
  double fe = (double)e;
  double hi = fe * LOG_LN2_HI;
  double lo = fe * LOG_LN2_LO;
  return hi + (lo + lf);
}

/* ------------------------------------------------------------------------------------ */
/* det-attn                                                                              */
/* ------------------------------------------------------------------------------------ */
typedef struct {
  const void *q, *k, *v;
  int dtype;
  int64_t B, Hq, Hkv, Sq, Skv, D;
  int64_t qs[4], ks[4], vs[4];
  int causal;
  float scale32;
  int64_t kv_lo, kv_hi;
  const int64_t* rows;
  int64_t nrows;
  const float* m_in;
  float* m_out;
  int64_t* num_out;
  int64_t* den_out;
  int violation;
  int nonfinite;
  int64_t next;
  pthread_mutex_t lock;
} attn_job;

static int64_t grab(attn_job* J) {
  pthread_mutex_lock(&J->lock);
  int64_t r = J->next++;
  pthread_mutex_unlock(&J->lock);
  return r;
}

/* exact score of one pair (page "det-attn", "Method") */
static float attn_score(const attn_job* J, int64_t b, int64_t h, int64_t j, kacc* acc,
                        const uint64_t* qm, const int* qn, const int* ql) {
  int64_t hk = h / (J->Hq / J->Hkv);
  kacc_zero(acc);
  for (int64_t d = 0; d < J->D; d++) {
    float kv = load_elem(J->k, J->dtype, b * J->ks[0] + hk * J->ks[1] + j * J->ks[2] + d);
    uint64_t km; int kn, kl;
    f32_split(kv, &km, &kn, &kl);
    kacc_add(acc, qm[d] * km, qn[d] ^ kn, ql[d] + kl);
  }
  float dsc = kacc_rn32(acc);
  return J->scale32 * dsc;   /* one binary32 multiply */
}

static void row_q(const attn_job* J, int64_t b, int64_t h, int64_t i, uint64_t* qm, int* qn, int* ql, int* nf) {
  for (int64_t d = 0; d < J->D; d++) {
    float x = load_elem(J->q, J->dtype, b * J->qs[0] + h * J->qs[1] + i * J->qs[2] + d);
    if (!isfinite(x)) *nf = 1;
    f32_split(x, &qm[d], &qn[d], &ql[d]);
  }
}

static void* rowmax_worker(void* arg) {
  attn_job* J = (attn_job*)arg;
  uint64_t* qm = malloc(sizeof(uint64_t) * J->D);
  int* qn = malloc(sizeof(int) * J->D);
  int* ql = malloc(sizeof(int) * J->D);
  kacc acc;
  for (int64_t r; (r = grab(J)) < J->nrows;) {
    int64_t flat = J->rows[r];
    int64_t i = flat % J->Sq, h = (flat / J->Sq) % J->Hq, b = flat / (J->Sq * J->Hq);
    int nf = 0;
    row_q(J, b, h, i, qm, qn, ql, &nf);
    float m = -INFINITY;
    for (int64_t j = J->kv_lo; j < J->kv_hi; j++) {
      if (J->causal && j > i) break;
      float s = attn_score(J, b, h, j, &acc, qm, qn, ql);
      if (!isfinite(s)) nf = 1;
      if (s > m) m = s;
    }
    if (m == 0.0f) m = 0.0f;  /* -0 -> +0 */
    J->m_out[r] = m;
    if (nf) flag(&J->nonfinite);
  }
  free(qm); free(qn); free(ql);
  return NULL;
}

static void* accumulate_worker(void* arg) {
  attn_job* J = (attn_job*)arg;
  int64_t D = J->D;
  uint64_t* qm = malloc(sizeof(uint64_t) * D);
  int* qn = malloc(sizeof(int) * D);
  int* ql = malloc(sizeof(int) * D);
  kacc* num = malloc(sizeof(kacc) * D);
  kacc den, acc;
  for (int64_t r; (r = grab(J)) < J->nrows;) {
    int64_t flat = J->rows[r];
    int64_t i = flat % J->Sq, h = (flat / J->Sq) % J->Hq, b = flat / (J->Sq * J->Hq);
    int64_t hk = h / (J->Hq / J->Hkv);
    int nf = 0;
    row_q(J, b, h, i, qm, qn, ql, &nf);
    for (int64_t d = 0; d < D; d++) kacc_zero(&num[d]);
    kacc_zero(&den);
    float m = J->m_in[r];
    for (int64_t j = J->kv_lo; j < J->kv_hi; j++) {
      if (J->causal && j > i) break;
      float s = attn_score(J, b, h, j, &acc, qm, qn, ql);
      float x = s - m;
      if (x > 0.0f) { flag(&J->violation); x = 0.0f; }
      if (x != x) { nf = 1; x = 0.0f; }
      float w = or_exp32_det(x);
      uint64_t wm; int wn, wl;
      f32_split(w, &wm, &wn, &wl);
      if (wm == 0) continue;
      kacc_add(&den, wm, 0, wl);
      for (int64_t d = 0; d < D; d++) {
        float vv = load_elem(J->v, J->dtype, b * J->vs[0] + hk * J->vs[1] + j * J->vs[2] + d);
        if (!isfinite(vv)) nf = 1;
        uint64_t vm; int vn, vl;
        f32_split(vv, &vm, &vn, &vl);
        kacc_add(&num[d], wm * vm, vn, wl + vl);
      }
    }
    /* canonical digits: NUM words 0..14 (E0 = -320), DEN words 5..10 (E0 = -160) */
    for (int64_t d = 0; d < D; d++)
      if (kacc_store(&num[d], 0, 15, J->num_out + r * 15 * D + d, D)) nf = 1;
    if (kacc_store(&den, 5, 6, J->den_out + r * 6, 1)) nf = 1;
    if (nf) flag(&J->nonfinite);
  }
  free(qm); free(qn); free(ql); free(num);
  return NULL;
}

static int run_threads(void* (*fn)(void*), void* job, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int t = 0; t < nthreads; t++) pthread_create(&th[t], NULL, fn, job);
  for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
  return 0;
}

static void job_init(attn_job* J, const void* q, const void* k, const void* v, int dtype, int64_t B, int64_t Hq,
                     int64_t Hkv, int64_t Sq, int64_t Skv, int64_t D, const int64_t* qs, const int64_t* ks,
                     const int64_t* vs, int causal, float scale32, int64_t kv_lo, int64_t kv_hi,
                     const int64_t* rows, int64_t nrows) {
  memset(J, 0, sizeof(*J));
  J->q = q; J->k = k; J->v = v; J->dtype = dtype;
  J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->Sq = Sq; J->Skv = Skv; J->D = D;
  for (int t = 0; t < 4; t++) { J->qs[t] = qs[t]; J->ks[t] = ks[t]; J->vs[t] = vs ? vs[t] : 0; }
  J->causal = causal; J->scale32 = scale32; J->kv_lo = kv_lo; J->kv_hi = kv_hi;
  J->rows = rows; J->nrows = nrows;
  pthread_mutex_init(&J->lock, NULL);
}

/* rowmax of the listed query rows (flat index (b*Hq + h)*Sq + i) over keys [kv_lo, kv_hi).
 * Returns bit 0 = a non-finite score or input was met. */
int or_attn_rowmax(const void* q, const void* k, int dtype, int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq,
                   int64_t Skv, int64_t D, const int64_t* qs, const int64_t* ks, int causal, float scale32,
                   int64_t kv_lo, int64_t kv_hi, const int64_t* rows, int64_t nrows, float* m_out, int nthreads) {
  attn_job J;
  job_init(&J, q, k, NULL, dtype, B, Hq, Hkv, Sq, Skv, D, qs, ks, NULL, causal, scale32, kv_lo, kv_hi, rows, nrows);
  J.m_out = m_out;
  run_threads(rowmax_worker, &J, nthreads);
  pthread_mutex_destroy(&J.lock);
  return J.nonfinite ? 1 : 0;
}

/* canonical NUM digits [nrows,15,D] and DEN digits [nrows,6] of the listed rows over
 * [kv_lo, kv_hi) with the given (global) rowmax per listed row.  Returns bit 0 =
 * non-finite met, bit 1 = a score above the supplied rowmax (clamped to weight 1). */
int or_attn_accumulate(const void* q, const void* k, const void* v, int dtype, int64_t B, int64_t Hq, int64_t Hkv,
                       int64_t Sq, int64_t Skv, int64_t D, const int64_t* qs, const int64_t* ks, const int64_t* vs,
                       int causal, float scale32, const float* m_rows, int64_t kv_lo, int64_t kv_hi,
                       const int64_t* rows, int64_t nrows, int64_t* num_out, int64_t* den_out, int nthreads) {
  attn_job J;
  job_init(&J, q, k, v, dtype, B, Hq, Hkv, Sq, Skv, D, qs, ks, vs, causal, scale32, kv_lo, kv_hi, rows, nrows);
  J.m_in = m_rows; J.num_out = num_out; J.den_out = den_out;
  run_threads(accumulate_worker, &J, nthreads);
  pthread_mutex_destroy(&J.lock);
  return (J.nonfinite ? 1 : 0) | (J.violation ? 2 : 0);
}

static void load_digits(kacc* a, const int64_t* dg, int64_t stride, int ndig, int word0) {
  kacc_zero(a);
  for (int k = 0; k < ndig; k++) a->w[word0 + k] = dg[k * stride];
}

/* o = RN32(RN64(RN64(NUM) / RN64(DEN))) for nrows rows of digits (any, not only canonical) */
int or_finalize(const int64_t* num, const int64_t* den, int64_t nrows, int64_t D, float* out) {
  kacc a;
  for (int64_t r = 0; r < nrows; r++) {
    load_digits(&a, den + r * 6, 1, 6, 5);
    double d64 = kacc_rn64(&a);
    for (int64_t d = 0; d < D; d++) {
      load_digits(&a, num + r * 15 * D + d, D, 15, 0);
      double n64 = kacc_rn64(&a);
      out[r * D + d] = (float)(n64 / d64);
    }
  }
  return 0;
}

/* canonical form of digit arrays: [n, ndig, inner] with word 0 weighing 2^e0 (e0 = -320
 * or -160).  Returns 1 if a value does not fit. */
int or_normalize(int64_t* dg, int64_t n, int ndig, int64_t inner, int e0) {
  int word0 = (e0 - KBASE) / 32, bad = 0;
  for (int64_t r = 0; r < n; r++)
    for (int64_t c = 0; c < inner; c++) {
      int64_t* p = dg + r * ndig * inner + c;
      kacc a;
      load_digits(&a, p, inner, ndig, word0);
      if (kacc_store(&a, word0, ndig, p, inner)) bad = 1;
    }
  return bad;
}

/* ------------------------------------------------------------------------------------ */
/* det-cross-entropy                                                                     */
/* ------------------------------------------------------------------------------------ */
typedef struct {
  const void* x;
  int dtype;
  int64_t N, V, rs, v_lo, v_hi;
  const int64_t* rows;
  int64_t nrows;
  const float* m_in;
  float* m_out;
  int64_t* den_out;
  int violation, nonfinite;
  int64_t next;
  pthread_mutex_t lock;
} dce_job;

static int64_t dgrab(dce_job* J) {
  pthread_mutex_lock(&J->lock);
  int64_t r = J->next++;
  pthread_mutex_unlock(&J->lock);
  return r;
}

static void* dce_rowmax_worker(void* arg) {
  dce_job* J = (dce_job*)arg;
  for (int64_t r; (r = dgrab(J)) < J->nrows;) {
    int64_t i = J->rows[r];
    float m = -INFINITY;
    for (int64_t v = J->v_lo; v < J->v_hi; v++) {
      float x = load_elem(J->x, J->dtype, i * J->rs + v);
      if (!isfinite(x)) flag(&J->nonfinite);
      if (x > m) m = x;
    }
    if (m == 0.0f) m = 0.0f;
    J->m_out[r] = m;
  }
  return NULL;
}

static void* dce_denom_worker(void* arg) {
  dce_job* J = (dce_job*)arg;
  kacc a;
  for (int64_t r; (r = dgrab(J)) < J->nrows;) {
    int64_t i = J->rows[r];
    float m = J->m_in[r];
    kacc_zero(&a);
    for (int64_t v = J->v_lo; v < J->v_hi; v++) {
      float x = load_elem(J->x, J->dtype, i * J->rs + v) - m;
      if (x > 0.0f) { flag(&J->violation); x = 0.0f; }
      if (x != x) { flag(&J->nonfinite); x = 0.0f; }
      uint64_t wm; int wn, wl;
      f32_split(or_exp32_det(x), &wm, &wn, &wl);
      kacc_add(&a, wm, 0, wl);
    }
    if (kacc_store(&a, 5, 6, J->den_out + r * 6, 1)) flag(&J->nonfinite);
  }
  return NULL;
}

int or_dce_rowmax(const void* x, int dtype, int64_t N, int64_t V, int64_t rs, int64_t v_lo, int64_t v_hi,
                  const int64_t* rows, int64_t nrows, float* m_out, int nthreads) {
  dce_job J;
  memset(&J, 0, sizeof(J));
  J.x = x; J.dtype = dtype; J.N = N; J.V = V; J.rs = rs; J.v_lo = v_lo; J.v_hi = v_hi;
  J.rows = rows; J.nrows = nrows; J.m_out = m_out;
  pthread_mutex_init(&J.lock, NULL);
  run_threads(dce_rowmax_worker, &J, nthreads);
  pthread_mutex_destroy(&J.lock);
  return J.nonfinite ? 1 : 0;
}

int or_dce_denom(const void* x, int dtype, int64_t N, int64_t V, int64_t rs, const float* m_rows, int64_t v_lo,
                 int64_t v_hi, const int64_t* rows, int64_t nrows, int64_t* den_out, int nthreads) {
  dce_job J;
  memset(&J, 0, sizeof(J));
  J.x = x; J.dtype = dtype; J.N = N; J.V = V; J.rs = rs; J.v_lo = v_lo; J.v_hi = v_hi;
  J.rows = rows; J.nrows = nrows; J.m_in = m_rows; J.den_out = den_out;
  pthread_mutex_init(&J.lock, NULL);
  run_threads(dce_denom_worker, &J, nthreads);
  pthread_mutex_destroy(&J.lock);
  return (J.nonfinite ? 1 : 0) | (J.violation ? 2 : 0);
}

/* loss_i = RN32(RN64(log64_det(d64) + RN64(m_i - x_{i,t_i}))), denom_i = d64 = RN64(den_i).
 * Returns bit 3 when a target is outside [0, V) (that loss is NaN). */
int or_dce_finalize(const int64_t* den, const void* x, int dtype, int64_t V, int64_t rs, const int64_t* targets,
                    const float* m_rows, const int64_t* rows, int64_t nrows, float* loss, double* denom) {
  int bad = 0;
  kacc a;
  for (int64_t r = 0; r < nrows; r++) {
    load_digits(&a, den + r * 6, 1, 6, 5);
    double d64 = kacc_rn64(&a);
    denom[r] = d64;
    int64_t t = targets[r];
    if (t < 0 || t >= V) { bad = 1; loss[r] = NAN; continue; }
    double xt = (double)load_elem(x, dtype, rows[r] * rs + t);
    double diff = (double)m_rows[r] - xt;
    double l = or_log64_det(d64) + diff;
    loss[r] = (float)l;
  }
  return bad ? 8 : 0;
}

/* vectorised forms, for the routine sweeps of the tests */
void or_exp32_det_many(const float* x, float* y, int64_t n) {
  for (int64_t i = 0; i < n; i++) y[i] = or_exp32_det(x[i]);
}
void or_log64_det_many(const double* x, double* y, int64_t n) {
  for (int64_t i = 0; i < n; i++) y[i] = or_log64_det(x[i]);
}
