// K2 with both products on the tensor cores (sm_103a): exact accumulate of NUM / DEN
// digits for D <= 128 (head dimensions below 128 padded with zero columns).
//
// Page "det-attn", section "Method": NUM_id = sum_j exp(s_ij - rowmax_i) V_jd and
// DEN_i = sum_j exp(s_ij - rowmax_i) are exact integer sums in fixed bins.
//
// CTA = 16 query rows of one (b, h), key tiles of 128 keys, one CTA per SM.
//
// Scores.  S^T = K Q^T from integer-valued bf16 digit slices (score_tc.cuh): per
// 16-dimension step, 4 tcgen05 MMAs of M = 128 keys x N = 64 x K = 16, one per key slice sa,
// with the four query slices stacked along N (n = 16 sb + row).  The MMA of key slice sa
// writes its accumulator at TMEM column offset 16 sa, so column 16 sb + row lands on
// 16 (sa + sb) + row: the tensor core itself forms the seven diagonal sums
// A_c = sum_{sa+sb=c} sum_d K_sa Q_sb (integers below 2^22, exact in f32).  A pair with a
// row outside its 26-bit window adds the row's low limbs to that truncated dot (dot_lo,
// score_tc.cuh); a pair with a deep row takes the per-thread exact dot.
//
// PV.  Every weight w >= 2^-56 is held as W = w 2^79, an integer below 2^80, split into
// ten base-256 digits W_s (bytes, exact in f16); V is fixed point per column, |Vint| < 2^23,
// split into three balanced base-256 digits V_t (|V_t| <= 128, prepared once per call).
// The ten weight digit planes of a 16-key block lie next to each other along N (n = 16 s +
// row, MN-major), so one MMA of M = 128 value columns x N = 160 x K = 16 multiplies V digit
// t by all ten; written at column offset 16 t it adds V_t W_s into the diagonal sum
// P_c (c = s + t) at column 16 c + row: three MMAs per 16 keys.  A product is at most
// 255 * 128 and a diagonal holds at most 3 per key, so over one 128-key tile every partial
// sum is an integer below 128 * 3 * 32640 < 2^24: exact.  After each tile the compute warps
// fold sum_c P_c 2^(8c) into three radix-2^32 int64 digits per (row, column) and zero the
// accumulators.  The weight digit planes and the PV accumulators are double-buffered, so
// the PV MMAs of one tile run while the next tile's weights are computed and the tile before
// is folded in.
//
// DEN.  The same planes read as an MN-major A operand (M = 8 digits x 16 rows) times a block
// of ones give sum_k W_s for digits 0-7 in TMEM lane 16 s + row; these sums grow by at most
// 255 per key, so they stay exact for ACC_TP_MAX_TILES tiles and are read once per pass.
// Digits 8-9 (below 2^16 per key) are summed with one warp reduction per row.
//
// Products outside the window are added with exact int64 atomics by the warp that owns the
// pair, so the compute warps share no per-tile state and never wait for each other within a
// pass.  They go to this SM's spill slot (attn_kernels.h), not to the output: the epilogue
// adds the slot digits the pass touched (a bitmap in shared memory) and clears them, so every
// output digit is written exactly once.  Weights 2^-112 <= w < 2^-56 are integers W' = w 2^135 < 2^79:
// per row, the warp sums W' Vint over its keys exactly (three 32-bit words of W') and adds
// the sums, so a row costs twelve atomics per lane and tile however many such weights it
// has.  V elements below their column window (Vint = 0 there) are kept in a per-warp list of
// (key, the four weights) and their products added after the tiles; smaller weights take
// whole-product atomics.
//
// Epilogue.  Per pass the compute warps add the spill slot's touched digits and carry the
// sums into canonical digits, then either store NUM / DEN digits (accumulate), or, when the
// call covers the whole key range (AttnArgs::out, no add_into), finalize in place: each row's
// DEN is rounded to binary64 and prepared as an integer divisor (divide.cuh), and every
// (row, column) gets o = RN32(RN64(RN64(NUM) / RN64(DEN))) on the integer pipe; only the f32
// output reaches device memory (page "det-attn", section "Method": finalize rounds and
// divides).
//
// Roles: warp 16 copies key operand steps (lane 0, 4-stage ring) and V digit blocks (lane 1,
// NVB-stage ring), warps 17 and 19 (lane 0) issue the score MMAs of alternate 16-dimension
// steps, warp 18 (lane 0) the PV and DEN MMAs.  Warps 0-15 read the score diagonals, compute weights, write the weight digit
// planes and drain the PV accumulators; each zeroes the TMEM it read before releasing it,
// so every MMA accumulates.  Every mbarrier wait is bounded; one that gives up sets
// DA_STATUS_TIMEOUT, and a failed wait in the compute warps only skips work.
#include "numerics.cuh"
#include "score_tc.cuh"
#include "divide.cuh"
#include "tc5.cuh"
#include "attn_kernels.h"

namespace detattn {

// SC: the score-cache variant holds no query operand and no key ring; that room holds the
// epilogue's element list (a deeper V ring there measured slower).
template <bool SC>
struct AccTpLayoutT {
  static constexpr int DP = 128, BM = 16, NDS = DP / 16, NSK = 4, NVB = 4, NCW = 16;
  // warps: NCW compute (four warpgroups) and the control warpgroup: copies (lane 0 key steps,
  // lane 1 V blocks), score MMAs of even steps, PV and DEN MMAs, score MMAs of odd steps
  static constexpr int LOADW = NCW, ISSW = NCW + 1, PISSW = NCW + 2, ISSW2 = NCW + 3, THREADS = 32 * (NCW + 4);
  static constexpr int NWP = 10, NVP = 3, NPD = NWP + NVP - 1, NKB = KTILE / VKEYS;
  static constexpr int NQ = NSLICE * BM;                              // score MMA N: the stacked query slices
  static constexpr int NW16 = NWP * BM;                               // PV MMA N: the stacked weight digits
  static constexpr int NDEN = 8;                                      // weight digits summed on the tensor cores
  // TMEM columns: two PV buffers (diagonal P_c at 16 c), the score diagonals at 16 c, DEN
  static constexpr int PV_COL = 0, PV_BUF = NPD * BM, SC_COL = 2 * PV_BUF, DEN_COL = SC_COL + NDIAG * BM, TCOLS = 512;
  static constexpr size_t q_step = (size_t)NQ * 32;                    // one B block: 64 rows (16 sb + r) x 16 bf16
  static constexpr size_t q_bytes = SC ? 0 : (size_t)NDS * q_step;
  static constexpr size_t k_off = q_bytes;                             // NSK key operand steps
  static constexpr size_t v_off = k_off + (SC ? 0 : (size_t)NSK * KT_BLOCK);   // NVB V digit blocks
  static constexpr size_t w_blk = (size_t)BM * VKEYS * 2;              // one weight digit plane: 16 rows x 16 keys
  static constexpr size_t w_buf = (size_t)NKB * NWP * w_blk;           // one tile's weight digit planes [kb][s]
  static constexpr size_t w_off = v_off + (size_t)NVB * VP_BLOCK;      // two buffers
  static constexpr size_t one_off = w_off + 2 * w_buf;                 // 16 x 16 f16 ones: DEN's B operand
  // SC: the epilogue's list of elements that need canonical digits (every element of a pass at
  // most), in the room the query operand and key ring leave unused
  static constexpr size_t e_off = one_off + 16 * 16 * 2;
  static constexpr size_t bytes = e_off + (SC ? (size_t)BM * DP * 32 : 0);
  static_assert(DEN_COL + 16 <= TCOLS, "TMEM columns");
  static_assert(NDEN * BM == 128, "the DEN MMA's A operand is eight digit planes");
  static_assert(NW16 <= 256 && NW16 % 16 == 0, "one PV MMA covers every weight digit");
  static_assert(bytes <= 213 * 1024, "shared memory budget (plus about 8 KB static)");
};
using AccTpLayout = AccTpLayoutT<false>;

// an element of the score-cache variant's epilogue that needs canonical digits: row, column and
// its three register digits
struct EpiElem {
  int rl, d;
  long long a0, a1, a2;
};
static_assert(sizeof(EpiElem) <= 32, "element list entry");

// one 16-key block: V digit t (A) times the ten stacked weight digits (B) into P_{s+t} of
// the PV buffer at TMEM address pv; weight digits 0-7 (A, MN-major) times ones (B) into DEN
__device__ __forceinline__ void pv_block_mmas(uint32_t pv, uint32_t den, const unsigned char* vblk,
                                              const unsigned char* wblk, uint64_t ones, uint32_t idesc_pv,
                                              uint32_t idesc_den) {
  using L = AccTpLayout;
  const uint64_t va = tc5::desc(tc5::smem_addr(vblk));
  const uint64_t wa = tc5::desc(tc5::smem_addr(wblk));
#pragma unroll
  for (int t = 0; t < L::NVP; t++)   // descriptor start addresses advance in 16-byte units
    tc5::mma_bf16(pv + t * L::BM, va + (uint64_t)(t * (VP_BLOCK / 3) / 16), wa, idesc_pv, 1u);
  tc5::mma_bf16(den, wa, ones, idesc_den, 1u);
}

// two f16 values b0, b1 in [0, 255] from the pattern (0x64 b1 0x64 b0): (1024 + b) - 1024; with
// bal, (1024 + b) - 1152 = b - 128 (a balanced digit)
__device__ __forceinline__ uint32_t f16_pair_from_biased(uint32_t h, bool bal = false) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(bal ? 0x64806480u : 0x64006400u));
  return r;
}

// dg[k] (radix 2^32, int64 with lazy carries) += the digits of sign * M * 2^off, for every k
// with a static index (the digit arrays stay in registers): digit k takes bits
// [32 k - off, 32 k - off + 32) of M.
template <int N>
__device__ __forceinline__ void add_u128_at(long long (&dg)[N], unsigned __int128 M, bool neg, int off) {
#pragma unroll
  for (int k = 0; k < N; k++) {
    const int sh = 32 * k - off;
    unsigned long long c = 0;
    if (sh >= 0 && sh < 128)
      c = (unsigned long long)(M >> sh) & 0xFFFFFFFFull;
    else if (sh < 0 && sh > -32)
      c = (unsigned long long)(M << (-sh)) & 0xFFFFFFFFull;
    dg[k] += neg ? -(long long)c : (long long)c;
  }
}

// the signed radix-2^32 digits d0 + d1 2^32 + d2 2^64 (each |d| < 2^62) as sign and magnitude
__device__ __forceinline__ void digits3_to_u128(long long d0, long long d1, long long d2, unsigned __int128& M, bool& neg) {
  const __int128 X = (__int128)d0 + ((__int128)d1 << 32) + ((__int128)d2 << 64);
  neg = X < 0;
  M = neg ? (unsigned __int128)(-X) : (unsigned __int128)X;
}

// carry-normalize radix-2^32 digits with static indices: 0 .. N - 2 in [0, 2^32), the top signed
template <int N>
__device__ __forceinline__ void carry_digits(long long (&dg)[N]) {
#pragma unroll
  for (int k = 0; k < N - 1; k++) {
    const long long c = dg[k] >> 32;
    dg[k] -= c * 4294967296ll;
    dg[k + 1] += c;
  }
}

// Fold one tile's PV accumulators (12 diagonals x this thread's 4 rows, TMEM address pvb) into
// the integer digits acc[r][g] (g: diagonals 4 g .. 4 g + 3), zero them and release the buffer.
// A function rather than a lambda so that it is always inlined and acc stays in registers.
// ONE_WAIT: all twelve diagonal loads in flight before one wait (more registers live).
template <bool ONE_WAIT>
__device__ __forceinline__ void drain_pv(long long (&acc)[4][3], uint32_t pvb, uint64_t* done, uint64_t* freeb,
                                         uint32_t parity, volatile int* abort, int lane) {
  using L = AccTpLayout;
  bool ok = true;
  if (lane == 0) ok = tc5::mbar_wait(done, parity, abort, 64);
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  tc5::fence_after();
  if (ok) {
    // sum_c P_c 2^(8c) over a group of four diagonals: |P_c| < 2^24 integers, converted exactly,
    // combined by exact 32 x 32 -> 64 multiply-adds
    auto fold = [&](const float (&pv)[4][4], int g3) {
#pragma unroll
      for (int r = 0; r < 4; r++) {
        long long s = (long long)__float2int_rn(pv[0][r]);
#pragma unroll
        for (int c = 1; c < 4; c++) mad_wide(s, __float2int_rn(pv[c][r]), 1 << (8 * c));
        acc[r][g3] += s;
      }
    };
    if constexpr (ONE_WAIT) {
      float pv[3][4][4];
#pragma unroll
      for (int g3 = 0; g3 < 3; g3++)
#pragma unroll
        for (int c = 0; c < 4; c++) tc5::ld_x4(pvb + (4 * g3 + c) * L::BM, pv[g3][c]);
      tc5::ld_wait();
#pragma unroll
      for (int g3 = 0; g3 < 3; g3++) fold(pv[g3], g3);
    } else {
#pragma unroll
      for (int g3 = 0; g3 < 3; g3++) {
        float pv[4][4];
#pragma unroll
        for (int c = 0; c < 4; c++) tc5::ld_x4(pvb + (4 * g3 + c) * L::BM, pv[c]);
        tc5::ld_wait();
        fold(pv, g3);
      }
    }
#pragma unroll
    for (int c = 0; c < L::NPD; c++) tc5::st_zero_x4(pvb + c * L::BM);
    tc5::st_wait();
  }
  tc5::fence_before();
  __syncwarp();
  if (lane == 0) tc5::mbar_arrive(freeb);
}

// The weight of one pair the straight-line evaluation cannot take (a row outside its 26-bit
// window, or a score outside the normal binary32 range), with the status bits it raises.
// Out of line and with scalar arguments only, so that its code does not raise the register
// pressure of the compute warps' tile loop: only the rare calls pay for saving registers.
struct SlowWeight {
  float w;
  int flags;
};
template <int DT>
__device__ __noinline__ SlowWeight slow_pair_weight(long long Tq, const typename In<DT>::T* qr, int Fq, int qfit,
                                                    const int2* qlo, int qlon, const typename In<DT>::T* kr, int Fk,
                                                    int kf, const int2* klo, int klon, int D, float scale32, float m) {
  float dot;
  if (qfit && kf) {   // a score outside the normal range: the general rounding
    dot = cr32_scaled(Tq, Fq + Fk);
  } else if (qlon != LO_DEEP && klon != KLO_DEEP) {   // truncated dot + low limbs
    dot = dot_lo<DT>(Tq, qr, Fq, qlo, qlon, kr, Fk, klo, klon);
  } else if (!qfit && kf) {   // a deep row: the general exact dot
    dot = exact_dot_lane<DT, true, false>(qr, Fq, kr, Fk, D);
  } else if (qfit) {
    dot = exact_dot_lane<DT, false, true>(qr, Fq, kr, Fk, D);
  } else {
    dot = exact_dot_lane<DT, true, true>(qr, Fq, kr, Fk, D);
  }
  SlowWeight r;
  r.flags = 0;
  float x = __fsub_rn(__fmul_rn(scale32, dot), m);
  if (x != x) { r.flags |= ST_NONFINITE; x = neg_inf(); }
  if (x > 0.0f) { r.flags |= ST_VIOLATION; x = 0.0f; }
  r.w = exp32_det(x);
  return r;
}

// SC: the scores come from the score cache (AttnArgs::scores, written by the rowmax kernel of
// the same call) instead of the score MMAs: no key operand stream, no score issue, no
// recombination or rounding; every other step is the same.
template <int DT, bool SC>
__global__ void __launch_bounds__(AccTpLayout::THREADS, 1) accumulate_tp_kernel(const AttnArgs a, const KvPrep p) {
  using T = typename In<DT>::T;
  using L = AccTpLayoutT<SC>;
  constexpr int DP = L::DP, BM = L::BM, NDS = L::NDS, NSK = L::NSK, NVB = L::NVB, NCW = L::NCW;
  constexpr int NKB = L::NKB, NWP = L::NWP, NW = DP / 32;
  constexpr int NCT = 32 * NCW;
  constexpr int NQ = L::NQ;
  constexpr uint32_t IDESC_S = tc5::idesc_bf16(KTILE, NQ);        // scores: 128 keys x (4 slices x 16 rows)
  constexpr uint32_t IDESC_P = tc5::idesc_f16(DP, L::NW16, true);   // PV: 128 columns x (10 digits x 16 rows)
  constexpr uint32_t IDESC_D = tc5::idesc_f16(L::NDEN * BM, 16, false, true);   // DEN: (8 digits x 16 rows) x 16
  extern __shared__ __align__(1024) unsigned char smem_p[];
  unsigned char* Qs = smem_p;
  unsigned char* Kst = smem_p + L::k_off;
  unsigned char* Vst = smem_p + L::v_off;
  unsigned char* Wp = smem_p + L::w_off;
  __shared__ __align__(8) uint64_t kfull[NSK], kempty[NSK], sfull, sempty, vfull[NVB], vempty[NVB], wready[2],
      pvdone[2], pvfree[2], wfree[2], fin;
  __shared__ uint32_t tmem_s;
  __shared__ int Fq[BM], Fv[DP];
  __shared__ unsigned char qfit[BM], qlon[BM];
  __shared__ int elist_n;   // SC epilogue: elements listed for canonical digits
  __shared__ int2 qlo[BM][NLO];
  __shared__ float mrow[BM];
  __shared__ long long denT[BM][3];
  constexpr int NVBL = 16;   // per compute warp: keys with V elements outside their window, handled after the tiles
  __shared__ float4 vbl_w[NCW][NVBL];
  __shared__ int vbl_j[NCW][NVBL], vbl_n[NCW];
  __shared__ uint32_t tbit[BM][NW];   // spill slot digits touched this pass: single columns, whole rows, DEN
  __shared__ int trow[BM], tden[BM];
  __shared__ idiv::Divisor fdiv[BM];   // fused finalize: each row's RN64(DEN) prepared as a divisor
  __shared__ double fden64[BM];
  __shared__ int fslow[BM];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // This CTA's work item: query-tile pair (causal) or query tile bx of head h, batch b, taken
  // from a.order when it is set (the heaviest items first; part 2 or 1: the pair's long or
  // short tile alone; an unused slot ends the CTA at once), else in launch order.
  const int ntq = (a.Sq + BM - 1) / BM;
  const int nx = a.causal ? (ntq + 1) / 2 : ntq;
  int item = (int)blockIdx.x, part = 0;
  if (a.order) {
    const int v = __ldg(a.order + blockIdx.x);
    if (v < 0) return;   // uniform over the CTA, before any barrier or TMEM allocation
    item = v & 0x1FFFFFFF;
    part = v >> 29;
  }
  const int bx = item % nx, h = (item / nx) % a.Hq, b = item / (nx * a.Hq), hk = h / (a.Hq / a.Hkv);
  __shared__ int s_hb[2];
  if (tid == 0) {
    s_hb[0] = h;
    s_hb[1] = b;
  }
  // Row, output and spill-slot addresses are recomputed where they are used (head and batch
  // read back through volatile shared-memory loads, which the compiler does not hoist), so the
  // compute warps do not hold them in registers across the tile loop.
  auto cta_y = [&]() { return (int64_t)*reinterpret_cast<volatile int*>(&s_hb[0]); };
  auto cta_z = [&]() { return (int64_t)*reinterpret_cast<volatile int*>(&s_hb[1]); };
  auto qrow = [&](int i) { return (const T*)a.q + cta_z() * a.qs[0] + cta_y() * a.qs[1] + (int64_t)i * a.qs[2]; };
  auto krow = [&](int j) {
    return (const T*)a.k + cta_z() * a.ks[0] + (cta_y() / (a.Hq / a.Hkv)) * a.ks[1] + (int64_t)j * a.ks[2];
  };
  auto vrow = [&](int j) {
    return (const T*)a.v + cta_z() * a.vs[0] + (cta_y() / (a.Hq / a.Hkv)) * a.vs[1] + (int64_t)j * a.vs[2];
  };
  auto out_row = [&](int i) { return (cta_z() * a.Hq + cta_y()) * a.Sq + i; };   // output row index
  auto slot_num = [&](int rl) {   // this SM's spill slot: NUM digits of row rl, [15][DP]
    uint32_t sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    return p.spill + (size_t)(sm < (uint32_t)SPILL_SLOTS ? sm : 0) * spill_slot_words(DP) + (size_t)rl * NUM_NDIG * DP;
  };
  auto slot_den = [&](int rl) { return slot_num(BM) + (size_t)rl * DEN_NDIG; };
  const int64_t krow0 = ((int64_t)b * a.Hkv + hk) * a.Skv;
  const unsigned char* ktc = p.ktc + (int64_t)(b * a.Hkv + hk) * p.ntk * NDS * KT_BLOCK;
  const unsigned char* vtc = p.vtc + (int64_t)(b * a.Hkv + hk) * p.ntk * NKB * VP_BLOCK;

  if (warp == 0) tc5::tmem_alloc(&tmem_s, L::TCOLS);
  if (tid == 0) {
    for (int s = 0; s < NSK; s++) {
      tc5::mbar_init(&kfull[s], 1);
      tc5::mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < NVB; s++) {
      tc5::mbar_init(&vfull[s], 1);
      tc5::mbar_init(&vempty[s], 1);
    }
    for (int s = 0; s < 2; s++) tc5::mbar_init(&wready[s], NCW);
    tc5::mbar_init(&sfull, 2);   // one commit per score issuer
    tc5::mbar_init(&sempty, NCW);
    for (int s = 0; s < 2; s++) {
      tc5::mbar_init(&pvdone[s], 1);
      tc5::mbar_init(&pvfree[s], NCW);
      tc5::mbar_init(&wfree[s], 1);   // SC: the MMAs that read weight-plane buffer s have completed
    }
    tc5::mbar_init(&fin, 3);   // the score issuers and the PV issuer
    s_abort = 0;
    tc5::mbar_fence_init();
  }
  for (int d = tid; d < DP; d += L::THREADS)   // biased exponent in [1, 254]: |Vint| < 2^23, digit offsets in range
    Fv[d] = min(max(p.vcol[((int64_t)b * a.Hkv + hk) * DP + d], 1), 254) - 149;
  for (int e = tid; e < 16 * 16 / 2; e += L::THREADS)   // f16 1.0 pairs: DEN's all-ones B operand
    reinterpret_cast<uint32_t*>(smem_p + L::one_off)[e] = 0x3C003C00u;
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  const uint32_t tmem = tmem_s;
  // every accumulator starts at zero; the compute warps zero what they read
  const int quarter = warp & 3, rg = warp >> 2;   // compute warp: TMEM lanes 32 quarter .., rows 4 rg .. 4 rg + 3
  const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
  if (warp < NCW) {
#pragma unroll
    for (int c = 0; c < 2 * L::NPD; c++) tc5::st_zero_x4(lane_base + L::PV_COL + c * BM + rg * 4);
#pragma unroll
    for (int c = 0; c < NDIAG; c++) tc5::st_zero_x4(lane_base + L::SC_COL + c * BM + rg * 4);
    tc5::st_zero_x4(lane_base + L::DEN_COL + rg * 4);
    tc5::st_wait();
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();

  int nf = 0, viol = 0;
  const int npass = (part == 0 && a.causal && bx != ntq - 1 - bx) ? 2 : 1;
  // Register split: the control warpgroup (copies, MMA issue) runs on 32 registers a thread,
  // the four compute warpgroups on 112 (640 x 96 at launch = 128 x 32 + 512 x 112).  Each
  // role runs its own pass loop; named barrier 2 opens a pass (query operand and per-pass
  // state ready), barrier 3 closes it.
  if (warp >= NCW) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 32;" ::: "memory");
    uint32_t tc = 0;   // key tiles of earlier passes
    uint32_t pc = 0;   // SC: PV buffer pairs of earlier passes
    for (int pass = 0; pass < npass; pass++) {
      const int q0 = (part == 1 || (part == 0 && pass == 1) ? bx : ntq - 1 - bx) * BM;
      const int hi = a.causal ? min(a.kv_hi, q0 + BM) : a.kv_hi;
      const int nkt = hi > a.kv_lo ? (hi - a.kv_lo + KTILE - 1) / KTILE : 0;
      tc5::bar_sync(2, L::THREADS);
      if (warp == L::LOADW) {   // ---------------- bulk copies ----------------
        if (lane == 0 && !SC) {   // key operand steps
          for (int ls = 0; ls < nkt * NDS && !s_abort; ls++) {
            const uint32_t g = tc * NDS + ls, st = g % NSK;
            if (g >= NSK && !tc5::mbar_wait(&kempty[st], ((g / NSK) - 1) & 1, &s_abort, 64)) break;
            tc5::mbar_expect_tx(&kfull[st], KT_BLOCK);
            tc5::bulk_g2s(Kst + st * KT_BLOCK, ktc + (size_t)ls * KT_BLOCK, KT_BLOCK, &kfull[st]);
          }
        } else if (lane == 1) {   // V digit blocks
          for (int lb = 0; lb < nkt * NKB && !s_abort; lb++) {
            const uint32_t g = tc * NKB + lb, sl = g % NVB;
            if (g >= NVB && !tc5::mbar_wait(&vempty[sl], ((g / NVB) - 1) & 1, &s_abort, 64)) break;
            tc5::mbar_expect_tx(&vfull[sl], VP_BLOCK);
            tc5::bulk_g2s(Vst + sl * VP_BLOCK, vtc + (size_t)lb * VP_BLOCK, VP_BLOCK, &vfull[sl]);
          }
        }
      } else {
        if ((warp == L::ISSW || warp == L::ISSW2) && lane == 0 && !SC) {   // ---------------- score MMAs: alternate steps ----------------
          for (int ls = warp == L::ISSW ? 0 : 1; ls < nkt * NDS && !s_abort; ls += 2) {
            const uint32_t g = tc * NDS + ls, st = g % NSK, tt = tc + ls / NDS;
            const int k = ls % NDS;
            if (!tc5::mbar_wait(&kfull[st], (g / NSK) & 1, &s_abort, 32)) break;
            if (k < 2 && tt >= 1 && !tc5::mbar_wait(&sempty, (tt - 1) & 1, &s_abort, 64)) break;
            tc5::fence_after();
            const uint64_t ka = tc5::desc(tc5::smem_addr(Kst + st * KT_BLOCK));
            const uint64_t qa = tc5::desc(tc5::smem_addr(Qs + k * L::q_step));
  #pragma unroll
            for (int sa = 0; sa < NSLICE; sa++)   // descriptor start addresses advance in 16-byte units
              tc5::mma_bf16(tmem + L::SC_COL + sa * BM, ka + (uint64_t)(sa * KTILE * 2), qa, IDESC_S, 1u);
            tc5::commit(&kempty[st]);
            if (k >= NDS - 2) tc5::commit(&sfull);   // this issuer's last step of the tile
          }
        } else if (warp == L::PISSW && lane == 0) {   // ---------------- PV and DEN MMAs ----------------
          const uint64_t ones = tc5::desc(tc5::smem_addr(smem_p + L::one_off));
          tc5::fence_after();   // the DEN accumulators were zeroed before the pass barrier
          for (int t = 0; t < nkt && !s_abort; t++) {
            const uint32_t tt = tc + t, bsel = tt & 1;
            // SC: PV sums of two tiles share one buffer (a pair: tiles 2 m and 2 m + 1 of the pass)
            const bool first = !SC || (t & 1) == 0, last = !SC || (t & 1) == 1 || t == nkt - 1;
            const uint32_t pb = SC ? (pc & 1) : bsel;
            const uint32_t pidx = SC ? pc : tt;   // pair (tile) index of the buffer's uses
            if (!tc5::mbar_wait(&wready[bsel], (tt >> 1) & 1, &s_abort, 64)) break;   // weight digits of tile tt
            if (first && pidx >= 2 && !tc5::mbar_wait(&pvfree[pb], ((pidx - 2) >> 1) & 1, &s_abort, 64)) break;   // buffer drained
            tc5::fence_after();
            for (int kb = 0; kb < NKB && !s_abort; kb++) {
              const uint32_t g = tt * NKB + kb, sl = g % NVB;
              if (!tc5::mbar_wait(&vfull[sl], (g / NVB) & 1, &s_abort, 32)) break;
              tc5::fence_after();
              pv_block_mmas(tmem + L::PV_COL + pb * L::PV_BUF, tmem + L::DEN_COL, Vst + sl * VP_BLOCK,
                            Wp + bsel * L::w_buf + (size_t)kb * NWP * L::w_blk, ones, IDESC_P, IDESC_D);
              tc5::commit(&vempty[sl]);
            }
            if (SC) tc5::commit(&wfree[bsel]);   // weight-plane buffer bsel may be rewritten once these complete
            if (last) {
              tc5::commit(&pvdone[pb]);
              if (SC) pc++;
            }
          }
        }
      }
      tc += nkt;
      tc5::bar_sync(3, L::THREADS);
    }
    if ((warp == L::ISSW || warp == L::PISSW || warp == L::ISSW2) && lane == 0) {   // every MMA has completed before TMEM is released
      tc5::commit(&fin);
      tc5::mbar_wait(&fin, 0, &s_abort);
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 96;" ::: "memory");
  } else {   // ---------------- compute warps ----------------
    asm volatile("setmaxnreg.inc.sync.aligned.u32 112;" ::: "memory");
    uint32_t tc = 0;   // key tiles of earlier passes
    uint32_t pcd = 0;   // SC: the next PV buffer pair to drain (pairs of earlier passes included)
    for (int pass = 0; pass < npass; pass++) {
      const int q0 = (part == 1 || (part == 0 && pass == 1) ? bx : ntq - 1 - bx) * BM;
      const int hi = a.causal ? min(a.kv_hi, q0 + BM) : a.kv_hi;
      const int nkt = hi > a.kv_lo ? (hi - a.kv_lo + KTILE - 1) / KTILE : 0;
      const int nrows = min(BM, a.Sq - q0);
      // ---- per pass: query slices (resident B operand of the scores), row maxima, cleared sums ----
      for (int r = warp; r < BM && !SC; r += NCW) {
        const int i = q0 + r;
        row_slices<DT, DP>(
            i < a.Sq ? qrow(i) : nullptr, a.D,
            [&](int q, int d, uint16_t v) {
              *reinterpret_cast<uint16_t*>(Qs + (d >> 4) * L::q_step + tc5::canon_off(q * BM + r, d & 15)) = v;
            },
            &Fq[r], &qfit[r], nf, lane, qlo[r], &qlon[r]);
      }
      for (int r = tid; r < BM; r += NCT) mrow[r] = (q0 + r < a.Sq) ? a.m_in[out_row(q0 + r)] : 0.0f;
      for (int e = tid; e < BM * 3; e += NCT) (&denT[0][0])[e] = 0;
      if (tid == 0) elist_n = 0;
      for (int e = tid; e < NCW; e += NCT) vbl_n[e] = 0;
      for (int e = tid; e < BM * NW; e += NCT) (&tbit[0][0])[e] = 0;
      for (int e = tid; e < BM; e += NCT) trow[e] = tden[e] = 0;
      tc5::fence_async_smem();
      tc5::bar_sync(2, L::THREADS);
        // Weight phase: this thread's key is TMEM lane dcol (rows 4 rg .. 4 rg + 3).  Drain: it
        // owns value column d = dcol; acc[r][k] is radix-2^32 digit k (lazily carried) in units
        // of 2^(Fv[d] - 79).
        const int dcol = 32 * quarter + lane;
        long long acc[4][3];
  #pragma unroll
        for (int r = 0; r < 4; r++)
  #pragma unroll
          for (int k = 0; k < 3; k++) acc[r][k] = 0;
        // lane 0 waits, the warp follows
        auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
          bool ok = true;
          if (lane == 0) ok = tc5::mbar_wait(bar, parity, &s_abort, 64);
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          tc5::fence_after();
          return ok;
        };
        // fold the PV accumulators of one tile (SC: of one pair of tiles) into the integer digits,
        // zero them, release them
        auto drain = [&](uint32_t tt) {
          drain_pv<SC>(acc, lane_base + L::PV_COL + (tt & 1) * L::PV_BUF + rg * 4, &pvdone[tt & 1], &pvfree[tt & 1],
                       (tt >> 1) & 1, &s_abort, lane);
        };
        // key meta and the V-bad words of this thread's key in tile t (zeros past the range)
        auto tile_meta = [&](int t, int& mv, uint4& vb) {
          mv = 0;
          vb = make_uint4(0u, 0u, 0u, 0u);
          if (t < nkt) {
            const int j = a.kv_lo + t * KTILE + dcol;
            if (j < hi) {
              if constexpr (!SC) mv = p.kmeta[krow0 + j];
              vb = *reinterpret_cast<const uint4*>(p.vbad + (krow0 + j) * NW);
            }
          }
        };
        int mv_n;
        uint4 vb_n;
        tile_meta(0, mv_n, vb_n);
        // score cache: this thread's key column of each block, rows 4 rg .. 4 rg + 3 (16 bytes),
        // one tile ahead; the blocks of one query tile are consecutive
        const float* sc_col = nullptr;
        float4 sc_n = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        float mr[4];
        if constexpr (SC) {
          sc_col = a.scores + sc_block(a, b * a.Hq + h, q0 / SC_ROWS, 0) * SC_BLOCK + dcol * SC_ROWS + 4 * rg;
          if (nkt > 0) sc_n = __ldcs(reinterpret_cast<const float4*>(sc_col));
#pragma unroll
          for (int e = 0; e < 4; e++) mr[e] = mrow[rg * 4 + e];
        }
        for (int t = 0; t < nkt; t++) {
          const int kt = a.kv_lo + t * KTILE;
          const uint32_t tt = tc + t, bsel = tt & 1;
          unsigned char* wbuf = Wp + bsel * L::w_buf;
          const int j = kt + dcol;
          const bool vj = j < hi;
          const int mv = mv_n;
          const uint4 vb = vb_n;
          tile_meta(t + 1, mv_n, vb_n);   // the next tile's, in flight meanwhile
          const int Fk = kmeta_F(mv), kf = kmeta_fit(mv);
          float w[4];
          uint32_t slow = 0;
          if constexpr (SC) {   // ---- weights from the cached exact scores ----
            const float4 sv = sc_n;
            if (t + 1 < nkt) sc_n = __ldcs(reinterpret_cast<const float4*>(sc_col + (size_t)(t + 1) * SC_BLOCK));
            const float scs[4] = {sv.x, sv.y, sv.z, sv.w};
  #pragma unroll
            for (int e = 0; e < 4; e++) {
              const int i = q0 + rg * 4 + e;
              const bool valid = vj && i < a.Sq && (!a.causal || j <= i);
              float x = __fsub_rn(scs[e], mr[e]);
              if (valid && x != x) nf |= ST_NONFINITE;
              if (valid && x > 0.0f) viol |= ST_VIOLATION;
              x = x != x ? neg_inf() : (x > 0.0f ? 0.0f : x);
              const float wf = exp32_det_nb(x);
              w[e] = valid ? wf : 0.0f;
            }
          } else {
          // ---- score diagonals of rows 4 rg .. 4 rg + 3 against this thread's key ----
          const bool ok = warp_wait(&sfull, tt & 1);
          long long Tq[4];   // the exact dot of each row's (truncated) digits with this key's
          if (ok) {
            float v[NDIAG][4];
  #pragma unroll
            for (int c = 0; c < NDIAG; c++) tc5::ld_x4(lane_base + L::SC_COL + c * BM + rg * 4, v[c]);
            tc5::ld_wait();
  #pragma unroll
            for (int e = 0; e < 4; e++) Tq[e] = combine_diag(v, e);
  #pragma unroll
            for (int c = 0; c < NDIAG; c++) tc5::st_zero_x4(lane_base + L::SC_COL + c * BM + rg * 4);
            tc5::st_wait();
          } else {
  #pragma unroll
            for (int e = 0; e < 4; e++) Tq[e] = 0;
          }
          tc5::fence_before();
          __syncwarp();
          if (lane == 0) tc5::mbar_arrive(&sempty);
          // ---- weights: one straight-line evaluation per row (the four interleave); pairs it
          // cannot take (a row outside its window, a score outside the normal range) go to `slow` ----
  #pragma unroll
          for (int e = 0; e < 4; e++) {
            const int rl = rg * 4 + e, i = q0 + rl;
            const bool valid = ok && vj && i < a.Sq && (!a.causal || j <= i);
            bool sp;
            const float c = cr32_scaled_cvt(Tq[e], Fq[rl] + Fk, sp);
            float x = __fsub_rn(__fmul_rn(a.scale32, c), mrow[rl]);
            const bool fast = valid && qfit[rl] && kf && !sp;
            if (fast && x != x) nf |= ST_NONFINITE;
            if (fast && x > 0.0f) viol |= ST_VIOLATION;
            x = x != x ? neg_inf() : (x > 0.0f ? 0.0f : x);
            const float wf = exp32_det_nb(x);
            w[e] = fast ? wf : 0.0f;
            if (valid && !fast) slow |= 1u << e;
          }
          if (slow) {
            for (int e = 0; e < 4; e++)
              if ((slow >> e) & 1u) {
                const int rl = rg * 4 + e;
                const SlowWeight r = slow_pair_weight<DT>(Tq[e], qrow(q0 + rl), Fq[rl], qfit[rl], qlo[rl], qlon[rl],
                                                          krow(j), Fk, kf, p.klo + (krow0 + j) * NLO, kmeta_lon(mv),
                                                          a.D, a.scale32, mrow[rl]);
                w[e] = r.w;
                nf |= r.flags & ST_NONFINITE;
                viol |= r.flags & ST_VIOLATION;
              }
          }
          }   // scores recomputed
          // ---- weight digits: W = w 2^79 = x 2^(8 b0), x < 2^32; words[e][q] = bytes 4q .. 4q + 3 of W ----
          uint32_t words[4][3];
          uint32_t tiny = 0;   // pairs with 0 < w < 2^-56: exact atomics below
  #pragma unroll
          for (int e = 0; e < 4; e++) {
            const uint32_t wb = __float_as_uint(w[e]);   // 0 <= w <= 1
            const int ex = (int)(wb >> 23);
            uint32_t x = 0;
            int b0 = 0;
            if (ex >= 71) {
              const int sh = ex - 71;   // <= 56
              b0 = sh >> 3;
              x = ((wb & 0x7FFFFFu) | 0x800000u) << (sh & 7);
            } else if (wb != 0u) {
              tiny |= 1u << e;
            }
            const uint64_t y = (uint64_t)x << (8 * (b0 & 3));
            const uint32_t lo = (uint32_t)y, hw = (uint32_t)(y >> 32);
            const bool low = b0 < 4;
            words[e][0] = low ? lo : 0u;
            words[e][1] = low ? hw : lo;
            words[e][2] = low ? 0u : hw;   // digits 8 and 9: below 2^16
          }
          if constexpr (SC) {
            // Balanced digits: W + sum_{s<9} 128 256^s, byte s minus 128 for s < 9 (in [-128, 127],
            // carries included), byte 9 as is (at most 129): the same W, products at most
            // 129 * 128, so two tiles of PV sums stay below 2^24 (the drains run every two tiles).
  #pragma unroll
            for (int e = 0; e < 4; e++) {
              const uint64_t lo64 = ((uint64_t)words[e][1] << 32) | words[e][0];
              const uint64_t b64 = lo64 + 0x8080808080808080ull;
              words[e][0] = (uint32_t)b64;
              words[e][1] = (uint32_t)(b64 >> 32);
              words[e][2] += 0x80u + (b64 < lo64 ? 1u : 0u);   // below 2^16 + 2^8
            }
  #pragma unroll
            for (int e = 0; e < 4; e++) {   // DEN digits 8-9: (byte 8 - 128) + 256 byte 9, one exact warp sum per row
              const int s89 = __reduce_add_sync(0xFFFFFFFFu, (int)(words[e][2] & 0xFFFFu) - 128);
              if (lane == 0 && s89) atomicAdd((unsigned long long*)&denT[rg * 4 + e][2], (unsigned long long)(long long)s89);
            }
          } else {
  #pragma unroll
            for (int e = 0; e < 4; e++) {   // DEN digits 8-9: one exact warp sum per row (32 x 2^16 < 2^21)
              const unsigned s89 = __reduce_add_sync(0xFFFFFFFFu, words[e][2]);
              if (lane == 0 && s89) atomicAdd((unsigned long long*)&denT[rg * 4 + e][2], (unsigned long long)s89);
            }
          }
          // SC: the buffer's previous tile (tt - 2) may still be read by its PV MMAs (drains run per pair)
          const bool wok = !SC || tt < 2 || warp_wait(&wfree[bsel], ((tt - 2) >> 1) & 1);
          if (wok) {   // plane s of this key's 4 rows: 4 f16 values, contiguous in the MN-major block (one 8-byte store)
            unsigned char* wdst = wbuf + (size_t)(dcol / VKEYS) * NWP * L::w_blk + tc5::mn_off(rg * 4, dcol % VKEYS);
  #pragma unroll
            for (int q = 0; q < 3; q++) {
              const uint32_t a01[2] = {__byte_perm(words[0][q], words[1][q], 0x5140),    // bytes 0, 1 of rows 0, 1
                                       __byte_perm(words[0][q], words[1][q], 0x7362)};   // bytes 2, 3
              const uint32_t a23[2] = {__byte_perm(words[2][q], words[3][q], 0x5140),
                                       __byte_perm(words[2][q], words[3][q], 0x7362)};
  #pragma unroll
              for (int k = 0; k < 4; k++) {
                const int s = 4 * q + k;
                if (s < NWP) {
                  const uint32_t sel = (k & 1) ? 0x4342u : 0x4140u;   // (0x64, byte of row 1, 0x64, byte of row 0)
                  const bool bal = SC && s < NWP - 1;   // digits 0-8 balanced, digit 9 as is
                  const uint32_t h01 = f16_pair_from_biased(__byte_perm(a01[k >> 1], 0x64646464u, sel), bal);
                  const uint32_t h23 = f16_pair_from_biased(__byte_perm(a23[k >> 1], 0x64646464u, sel), bal);
                  *reinterpret_cast<uint2*>(wdst + s * L::w_blk) = make_uint2(h01, h23);
                }
              }
            }
          }
          tc5::fence_async_smem();   // the weight digit planes are read by the tensor cores
          __syncwarp();
          if (lane == 0) tc5::mbar_arrive(&wready[bsel]);
          // ---- the previous tile's (SC: pair's) PV products are done by now (or soon): fold them in ----
          if constexpr (SC) {
            if (t >= 2 && (t & 1) == 0) drain(pcd++);   // the pair of tiles t - 2, t - 1
          } else {
            if (t >= 1) drain(tt - 1);
          }
          // ---- this warp's products outside the window: exact int64 atomics into the output digits ----
          if (__ballot_sync(0xFFFFFFFFu, tiny != 0)) {
  #pragma unroll
            for (int e = 0; e < 4; e++) {
              uint32_t pend = __ballot_sync(0xFFFFFFFFu, (tiny >> e) & 1u);
              if (!pend) continue;
              const int rl = rg * 4 + e;
              long long* nrow = slot_num(rl);
              if (lane == 0) {
                trow[rl] = 1;
                tden[rl] = 1;
              }
              long long sum[NW][3];
  #pragma unroll
              for (int c = 0; c < NW; c++) sum[c][0] = sum[c][1] = sum[c][2] = 0;
              // SC: the Vint rows of up to TB pending keys at a time are staged in this warp's part of
              // the element-list room (unused during the tile loop) by asynchronous copies issued
              // together, so a row whose weights are nearly all tiny pays one memory latency per TB keys
              constexpr int TB = 4;
              int* stg = SC ? reinterpret_cast<int*>(smem_p + L::e_off) + warp * (TB * DP) : nullptr;
              uint32_t staged = 0;   // the keys of the current batch (SC)
              for (; pend; pend &= pend - 1) {
                const int src = __ffs(pend) - 1, jj = kt + 32 * quarter + src;
                if constexpr (SC) {
                  if (!((staged >> src) & 1u)) {   // a new batch: the next TB pending keys
                    __syncwarp();                  // the previous batch's rows are read
                    staged = 0;
                    uint32_t q = pend;
  #pragma unroll
                    for (int u = 0; u < TB; u++) {
                      if (q) {
                        const int su = __ffs(q) - 1;
                        staged |= 1u << su;
                        cp_async16(stg + u * DP + 4 * lane, p.vint + (krow0 + kt + 32 * quarter + su) * DP + 4 * lane, 16);
                        q &= q - 1;
                      }
                    }
                    cp_async_wait_all();
                    __syncwarp();
                  }
                }
                const uint32_t wb = __float_as_uint(__shfl_sync(0xFFFFFFFFu, w[e], src));
                const Split sw = split_f32(wb);
                if (lane == 0) atomic_digits_add(slot_den(rl), 1, DEN_E0, sw.mant, 0, sw.lsb);
                const int ex = (int)(wb >> 23);
                if (ex >= 15) {   // W' = w 2^135 = x 2^(8 b0): words of W' against the prepared Vint
                  const int sh = ex - 15, b0 = sh >> 3;
                  const uint64_t y = (uint64_t)(((wb & 0x7FFFFFu) | 0x800000u) << (sh & 7)) << (8 * (b0 & 3));
                  const bool low = b0 < 4;
                  const long long w0 = low ? (long long)(uint32_t)y : 0, w1 = low ? (long long)(y >> 32) : (long long)(uint32_t)y,
                                  w2 = low ? 0 : (long long)(y >> 32);
                  const int* vrow = SC ? stg + __popc(staged & ((1u << src) - 1u)) * DP : p.vint + (krow0 + jj) * DP;
  #pragma unroll
                  for (int c = 0; c < NW; c++) {   // |Vint| < 2^23, words < 2^32: 32 products stay below 2^60
                    const long long vi = vrow[lane + 32 * c];
                    sum[c][0] += vi * w0;
                    sum[c][1] += vi * w1;
                    sum[c][2] += vi * w2;
                  }
                } else {   // w < 2^-112: the whole product w V_jd for every d
                  for (int d = lane; d < a.D; d += 32) {
                    const uint32_t u = In<DT>::bits(vrow(jj), d);
                    if (nonfinite_bits(u)) continue;
                    const Split sv = split_f32(u);
                    atomic_digits_add(nrow + d, DP, NUM_E0, (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
                  }
                }
              }
  #pragma unroll
              for (int c = 0; c < NW; c++) {
                const int d = lane + 32 * c;
                if (d < a.D)
  #pragma unroll
                  for (int q = 0; q < 3; q++)
                    if (sum[c][q] != 0)
                      atomic_digits_add(nrow + d, DP, NUM_E0,
                                        sum[c][q] < 0 ? 0ull - (unsigned long long)sum[c][q] : (unsigned long long)sum[c][q],
                                        sum[c][q] < 0, Fv[d] - 135 + 32 * q);
              }
            }
          }
          {   // keys with V elements outside their column window: listed, their products added after the tiles
            const bool bad = (vb.x | vb.y | vb.z | vb.w) != 0u && (w[0] != 0.0f || w[1] != 0.0f || w[2] != 0.0f || w[3] != 0.0f);
            const uint32_t bm = __ballot_sync(0xFFFFFFFFu, bad);
            if (bm) {
              const int base = vbl_n[warp];
              const int idx = base + __popc(bm & ((1u << lane) - 1u));
              if (bad && idx < NVBL) {
                vbl_w[warp][idx] = make_float4(w[0], w[1], w[2], w[3]);
                vbl_j[warp][idx] = j;
              }
              __syncwarp();
              if (lane == 0) vbl_n[warp] = base + __popc(bm);
              if (bad && idx >= NVBL) {   // list full: this lane adds its products now
                const uint32_t vw[4] = {vb.x, vb.y, vb.z, vb.w};
  #pragma unroll
                for (int tw = 0; tw < NW; tw++)
                  for (uint32_t m = vw[tw]; m; m &= m - 1) {
                    const int d = tw * 32 + __ffs(m) - 1;
                    const Split sv = split_f32(In<DT>::bits(vrow(j), d));
  #pragma unroll
                    for (int e = 0; e < 4; e++) {
                      const uint32_t wb = __float_as_uint(w[e]);
                      if (wb == 0u || (int)(wb >> 23) < 15) continue;   // zero, or a whole-product pair above
                      const Split sw = split_f32(wb);
                      atomic_digits_add(slot_num(rg * 4 + e) + d, DP, NUM_E0,
                                        (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
                      atomicOr(&tbit[rg * 4 + e][d >> 5], 1u << (d & 31));
                    }
                  }
              }
              __syncwarp();
            }
          }
        }
        if (nkt > 0) drain(SC ? pcd++ : tc + nkt - 1);
        if (lane < min(vbl_n[warp], NVBL)) {   // listed keys, one per lane: products of their V elements below the window
          const int jj = vbl_j[warp][lane];
          const float4 wl = vbl_w[warp][lane];
          const float wr[4] = {wl.x, wl.y, wl.z, wl.w};
          const uint4 vbr = *reinterpret_cast<const uint4*>(p.vbad + (krow0 + jj) * NW);
          const uint32_t vw[4] = {vbr.x, vbr.y, vbr.z, vbr.w};
  #pragma unroll
          for (int tw = 0; tw < NW; tw++)
            for (uint32_t m = vw[tw]; m; m &= m - 1) {
              const int d = tw * 32 + __ffs(m) - 1;
              const Split sv = split_f32(In<DT>::bits(vrow(jj), d));
  #pragma unroll
              for (int e = 0; e < 4; e++) {
                const uint32_t wb = __float_as_uint(wr[e]);
                if (wb == 0u || (int)(wb >> 23) < 15) continue;   // smaller weights took whole products
                const Split sw = split_f32(wb);
                atomic_digits_add(slot_num(rg * 4 + e) + d, DP, NUM_E0,
                                  (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
                atomicOr(&tbit[rg * 4 + e][d >> 5], 1u << (d & 31));
              }
            }
        }
        // ---- DEN digits 0-7 from TMEM (lane 16 s + row; every column holds the same sum) ----
        if (rg == 0) {
          if (nkt > 0) {
            const float dsum = tc5::ld_x1(lane_base + L::DEN_COL);
            tc5::ld_wait();
            const int sv = __float2int_rn(dsum);   // < 2^24
            const int s = 2 * quarter + (lane >> 4), rl = lane & 15;
            if (sv) atomicAdd((unsigned long long*)&denT[rl][s >> 2], (unsigned long long)sv << (8 * (s & 3)));
            tc5::st_zero_x8(lane_base + L::DEN_COL);
            tc5::st_zero_x8(lane_base + L::DEN_COL + 8);
            tc5::st_wait();
          }
          tc5::fence_before();
        }
        // ---- epilogue: canonical digits ----
        tc5::bar_sync(1, NCT);   // denT, the touched flags and every spill atomic of this pass complete
        {
          uint32_t sm;
          asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
          if (sm >= (uint32_t)SPILL_SLOTS) nf |= ST_HEADROOM;   // no spill slot for this SM: products outside the windows are missing
        }
        // canonical DEN digits of row rl: this pass's sum, the spill slot's (cleared after), the
        // stored digits with add_into; headroom checked
        auto den_digits = [&](int rl, long long (&t)[DEN_NDIG]) {
          const long long* drow = a.den + out_row(q0 + rl) * DEN_NDIG;
          long long dg[DEN_NDIG + 3];
  #pragma unroll
          for (int k = 0; k < DEN_NDIG + 3; k++) dg[k] = 0;
          if (a.add_into)
  #pragma unroll
            for (int k = 0; k < DEN_NDIG; k++) dg[k] = __ldcg(drow + k);
          if (tden[rl])
  #pragma unroll
            for (int k = 0; k < DEN_NDIG; k++) {
              dg[k] += __ldcg(slot_den(rl) + k);
              slot_den(rl)[k] = 0;
            }
          {
            unsigned __int128 M;
            bool neg;
            digits3_to_u128(denT[rl][0], denT[rl][1], denT[rl][2], M, neg);
            add_u128_at(dg, M, neg, -79 - DEN_E0);   // W units
          }
          carry_digits(dg);
          long long top = dg[DEN_NDIG + 2];
          bool bad = false;
#pragma unroll
          for (int k = DEN_NDIG + 1; k >= DEN_NDIG - 1; k--) {
            if (top > (1ll << 30) || top < -(1ll << 30)) bad = true;
            top = top * 4294967296ll + dg[k];
          }
          if (bad) nf |= ST_HEADROOM;
  #pragma unroll
          for (int k = 0; k < DEN_NDIG - 1; k++) t[k] = dg[k];
          t[DEN_NDIG - 1] = top;
        };
        const bool fused = a.out != nullptr;   // finalize here: o = RN32(RN64(RN64(NUM) / RN64(DEN)))
        const int d = dcol;
        // SC, phase 1a (needs no divisor, so it overlaps the divisors' preparation): an element
        // whose column of the spill slot was not touched holds NUM = X 2^(Fv - 79) exactly in its
        // three register digits; its RN64 comes from that 128-bit integer.  Touched elements are
        // listed for phase 2.
        uint64_t p1m[4];
        int p1e[4];
        uint32_t p1nz = 0, p1neg = 0, p1live = 0;
        if constexpr (SC) {
          EpiElem* elist = reinterpret_cast<EpiElem*>(smem_p + L::e_off);
  #pragma unroll
          for (int r = 0; r < 4; r++) {
            p1m[r] = 0;
            p1e[r] = 0;
            const int rl = rg * 4 + r, i = q0 + rl;
            const bool live = i < a.Sq && d < a.D;
            const bool touched = live && (trow[rl] || ((tbit[rl][d >> 5] >> (d & 31)) & 1u));
            const uint32_t tm = __ballot_sync(0xFFFFFFFFu, touched);   // one list slot reservation per warp and row
            if (tm) {
              int base = 0;
              if (lane == 0) base = atomicAdd(&elist_n, __popc(tm));
              base = __shfl_sync(0xFFFFFFFFu, base, 0);
              if (touched) elist[base + __popc(tm & ((1u << lane) - 1u))] = EpiElem{rl, d, acc[r][0], acc[r][1], acc[r][2]};
            }
            if (!live || touched) continue;
            const __int128 X = (__int128)acc[r][0] + (__int128)acc[r][1] * ((__int128)1 << 32) +
                               (__int128)acc[r][2] * ((__int128)1 << 64);
            bool neg;
            if (idiv::i128_split_rn64(X, Fv[d] - 79, neg, p1m[r], p1e[r])) p1nz |= 1u << r;
            if (neg) p1neg |= 1u << r;
            p1live |= 1u << r;
          }
        }
        if (fused) {
          for (int rl = tid; rl < nrows; rl += NCT) {
            long long t[DEN_NDIG];
            den_digits(rl, t);
            bool neg;
            uint64_t mm;
            int ee;
            const bool nz = idiv::digits_split_rn64<DEN_NDIG>(t, DEN_E0, neg, mm, ee);
            fslow[rl] = !nz || neg;   // a zero or negative DEN divides in binary64 (IEEE NaN / inf)
            fden64[rl] = nz ? idiv::make_f64(neg, mm, ee) : 0.0;
            if (nz && !neg) fdiv[rl] = idiv::make_divisor(mm, ee);
          }
          tc5::bar_sync(1, NCT);
        }
        // a pass with no key adds nothing: with canonical digits already there, leave them
        const bool keep = nkt == 0 && a.add_into && a.canon_in && !fused;
        if constexpr (SC) {   // phase 1b: the untouched elements' quotients
  #pragma unroll
          for (int r = 0; r < 4; r++) {
            if (!((p1live >> r) & 1u)) continue;
            const int rl = rg * 4 + r;
            const bool nz = (p1nz >> r) & 1u, neg = (p1neg >> r) & 1u;
            float o = 0.0f;   // RN64(NUM) = +0 over a positive DEN
            if (fslow[rl])
              o = __double2float_rn(__ddiv_rn(nz ? idiv::make_f64(neg, p1m[r], p1e[r]) : 0.0, fden64[rl]));
            else if (nz)
              o = __uint_as_float(idiv::div_rn32(p1m[r], p1e[r], fdiv[rl], neg));
            a.out[out_row(q0 + rl) * a.D + d] = o;
          }
          tc5::bar_sync(1, NCT);   // the element list is complete
        }
        // canonical digits of one element (row rl, column dd, register digits a0..a2): the stored
        // digits with add_into, the spill slot's touched digits (cleared after), the register
        // digits; then stored, or finalized
        auto canonical = [&](int rl, int dd, long long a0, long long a1, long long a2) {
          const int i = q0 + rl;
          if (i >= a.Sq || dd >= a.D || keep) return;
          const bool touched = trow[rl] || ((tbit[rl][dd >> 5] >> (dd & 31)) & 1u);
          long long* nrow = a.num + out_row(i) * NUM_NDIG * a.D;   // unused when fused
          long long dg[NUM_NDIG + 3];
  #pragma unroll
          for (int k = 0; k < NUM_NDIG + 3; k++) dg[k] = 0;
          if (a.add_into)
  #pragma unroll
            for (int k = 0; k < NUM_NDIG; k++) dg[k] = __ldcg(nrow + (int64_t)k * a.D + dd);
          if (touched) {   // this digit column of the slot was touched
            long long* sp = slot_num(rl) + dd;
  #pragma unroll
            for (int k = 0; k < NUM_NDIG; k++) {
              dg[k] += __ldcg(sp + (size_t)k * DP);
              sp[(size_t)k * DP] = 0;
            }
          }
          {
            unsigned __int128 M;
            bool neg;
            digits3_to_u128(a0, a1, a2, M, neg);
            add_u128_at(dg, M, neg, Fv[dd] - 79 - NUM_E0);   // the accumulator's unit is 2^(Fv - 79)
          }
          carry_digits(dg);
          long long top = dg[NUM_NDIG + 2];
          bool bad = false;
#pragma unroll
          for (int k = NUM_NDIG + 1; k >= NUM_NDIG - 1; k--) {
            if (top > (1ll << 30) || top < -(1ll << 30)) bad = true;
            top = top * 4294967296ll + dg[k];
          }
          if (bad) nf |= ST_HEADROOM;
          if (fused) {
            long long t[NUM_NDIG];
  #pragma unroll
            for (int k = 0; k < NUM_NDIG - 1; k++) t[k] = dg[k];
            t[NUM_NDIG - 1] = top;
            bool neg;
            uint64_t mm;
            int ee;
            const bool nz = idiv::digits_split_rn64<NUM_NDIG>(t, NUM_E0, neg, mm, ee);
            float o = 0.0f;   // RN64(NUM) = +0 over a positive DEN
            if (fslow[rl])
              o = __double2float_rn(__ddiv_rn(nz ? idiv::make_f64(neg, mm, ee) : 0.0, fden64[rl]));
            else if (nz)
              o = __uint_as_float(idiv::div_rn32(mm, ee, fdiv[rl], neg));
            a.out[out_row(i) * a.D + dd] = o;
          } else {
  #pragma unroll
            for (int k = 0; k < NUM_NDIG - 1; k++) nrow[(int64_t)k * a.D + dd] = dg[k];
            nrow[(int64_t)(NUM_NDIG - 1) * a.D + dd] = top;
          }
        };
        if constexpr (SC) {
          const EpiElem* el = reinterpret_cast<const EpiElem*>(smem_p + L::e_off);
          for (int e = tid; e < elist_n; e += NCT) canonical(el[e].rl, el[e].d, el[e].a0, el[e].a1, el[e].a2);
        } else {
  #pragma unroll
          for (int r = 0; r < 4; r++) canonical(rg * 4 + r, d, acc[r][0], acc[r][1], acc[r][2]);
        }
        if (!fused && !keep)
          for (int rl = tid; rl < nrows; rl += NCT) {
            long long t[DEN_NDIG];
            den_digits(rl, t);
            long long* drow = a.den + out_row(q0 + rl) * DEN_NDIG;
  #pragma unroll
            for (int k = 0; k < DEN_NDIG; k++) drow[k] = t[k];
          }
        __threadfence();   // the cleared slot digits reach L2 before the SM's next CTA adds into them
          tc += nkt;
      tc5::bar_sync(3, L::THREADS);
    }
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  if (warp == 0) tc5::tmem_dealloc(tmem, L::TCOLS);
  if (s_abort) nf |= ST_TIMEOUT;
  report(a.status, nf | viol);
}

template <int DT, bool SC>
static cudaError_t launch_acc_tp_t(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  using L = AccTpLayoutT<SC>;
  cudaError_t e =
      cudaFuncSetAttribute(accumulate_tp_kernel<DT, SC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
  if (e != cudaSuccess) return e;
  // the spill slots start clean (a CTA clears what it used; a kernel that gave up may not have)
  e = cudaMemsetAsync(p.spill, 0, (size_t)SPILL_SLOTS * spill_slot_words(L::DP) * sizeof(long long), st);
  if (e != cudaSuccess) return e;
  const int nt = (a.Sq + L::BM - 1) / L::BM;
  const int64_t nitems = (int64_t)(a.causal ? (nt + 1) / 2 : nt) * a.Hq * a.B;   // one CTA per work item
  const int64_t nblocks = nitems + (a.order ? a.order_extra : 0);
  accumulate_tp_kernel<DT, SC><<<(unsigned)nblocks, L::THREADS, L::bytes, st>>>(a, p);
  return cudaGetLastError();
}

// ---- work order ----
// A work item whose rows have a rowmax far above the rest of their scores has most of its
// weights below the 2^-56 window, and those take the exact per-pair path: such an item runs
// several times longer than the others.  Launched late it leaves the GPU idle behind it, so the
// items whose largest rowmax lies within 5 of the largest of the call go first.  The order
// only schedules the same work: the output does not depend on it.
static int tp_nx(const AttnArgs& a) {
  const int nt = (a.Sq + AccTpLayout::BM - 1) / AccTpLayout::BM;
  return a.causal ? (nt + 1) / 2 : nt;
}

__global__ void tp_item_keys_kernel(const AttnArgs a, int nx, int nitems, int* keys, int* gmax) {
  constexpr int BM = AccTpLayout::BM;
  const int it = blockIdx.x * blockDim.x + threadIdx.x;
  if (it >= nitems) return;
  const int ntq = (a.Sq + BM - 1) / BM;
  const int bx = it % nx, h = (it / nx) % a.Hq, b = it / (nx * a.Hq);
  const float* mr = a.m_in + ((int64_t)b * a.Hq + h) * a.Sq;
  int key = float_key(neg_inf());
  for (int pass = 0; pass < 2; pass++) {
    const int qt = pass == 0 ? (a.causal ? ntq - 1 - bx : bx) : bx;
    if (pass == 1 && (!a.causal || qt == ntq - 1 - bx)) break;
    for (int i = qt * BM; i < min(a.Sq, qt * BM + BM); i++) {
      const float m = mr[i];
      if (m == m) key = max(key, float_key(m));
    }
  }
  keys[it] = key;
  atomicMax(gmax, key);
}

// Then the light items; last, split in two, the k pairs of each (b, h) with the largest bx
// (their two tiles near the middle of the sequence, so the halves are near equal), long
// halves before short ones, so the end of the launch is made of the smallest items (k = half
// the SMs over the heads: about one wave of halves, at most a quarter of the pairs).
// Classes: 0 heavy, 1 light, 2 split.
__global__ void tp_item_class_kernel(const AttnArgs a, int nx, int nitems, int ksplit, const int* keys, int* counters,
                                     unsigned char* cls) {
  const int it = blockIdx.x * blockDim.x + threadIdx.x;
  if (it >= nitems) return;
  const int ntq = (a.Sq + AccTpLayout::BM - 1) / AccTpLayout::BM, bx = it % nx;
  const int thr = float_key(__fsub_rn(key_float(counters[0]), 5.0f));
  const int c = keys[it] >= thr ? 0 : (a.causal && bx >= nx - ksplit && bx != ntq - 1 - bx ? 2 : 1);
  cls[it] = (unsigned char)c;
  atomicAdd(&counters[1 + c], 1);
}

__global__ void tp_item_place_kernel(int nitems, int nslots, const unsigned char* cls, int* counters, int* order) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= nslots) return;
  const int nh = counters[1], nl = counters[2], ns = counters[3];
  if (t >= nitems + ns) order[t] = -1;   // an unused slot (fewer pairs split than reserved)
  if (t >= nitems) return;
  const int c = cls[t];
  if (c == 0) {
    order[atomicAdd(&counters[4], 1)] = t;
  } else if (c == 1) {
    order[nh + atomicAdd(&counters[5], 1)] = t;
  } else {
    const int q = atomicAdd(&counters[6], 1);
    order[nh + nl + q] = t | (1 << 30);        // the long tile
    order[nh + nl + ns + q] = t | (1 << 29);   // the short tile
  }
}

static int current_device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 1;
  return n;
}

static int tp_ksplit(const AttnArgs& a) {
  static const int sms = current_device_sms();   // initialised once, safe under concurrent first calls
  if (!a.causal) return 0;
  const int bh = a.Hq * a.B;
  return min(tp_nx(a) / 4, max(1, (sms + bh - 1) / bh / 2));
}

size_t tp_order_bytes(const AttnArgs& a) {
  const int64_t nitems = (int64_t)tp_nx(a) * a.Hq * a.B, nslots = nitems + (int64_t)tp_ksplit(a) * a.Hq * a.B;
  return 32 + (size_t)nitems * 4 + (((size_t)nitems + 15) & ~(size_t)15) + (size_t)nslots * 4;
}

cudaError_t launch_tp_order(AttnArgs& a, void* ws, cudaStream_t st) {
  const int64_t nitems = (int64_t)tp_nx(a) * a.Hq * a.B;
  const int ksplit = tp_ksplit(a);
  const int64_t nslots = nitems + (int64_t)ksplit * a.Hq * a.B;
  int* counters = (int*)ws;   // largest key (+0 to start); heavy, light, split counts; their positions taken
  int* keys = counters + 8;
  unsigned char* cls = (unsigned char*)(keys + nitems);
  int* order = (int*)(cls + ((nitems + 15) & ~(int64_t)15));
  cudaError_t e = cudaMemsetAsync(counters, 0, 32, st);
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)((nitems + 255) / 256), sblocks = (unsigned)((nslots + 255) / 256);
  tp_item_keys_kernel<<<blocks, 256, 0, st>>>(a, tp_nx(a), (int)nitems, keys, counters);
  tp_item_class_kernel<<<blocks, 256, 0, st>>>(a, tp_nx(a), (int)nitems, ksplit, keys, counters, cls);
  tp_item_place_kernel<<<sblocks, 256, 0, st>>>((int)nitems, (int)nslots, cls, counters, order);
  a.order = order;
  a.order_extra = (int)(nslots - nitems);
  return cudaGetLastError();
}

cudaError_t launch_accumulate_tp(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  if (a.scores) return a.dtype == 0 ? launch_acc_tp_t<0, true>(a, p, st) : launch_acc_tp_t<1, true>(a, p, st);
  return a.dtype == 0 ? launch_acc_tp_t<0, false>(a, p, st) : launch_acc_tp_t<1, false>(a, p, st);
}

}  // namespace detattn
