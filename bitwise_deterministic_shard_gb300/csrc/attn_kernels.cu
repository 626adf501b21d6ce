// det-attn kernels for sm_103a: rowmax (pass 1, tcgen05) and the exact accumulate for
// D = 256 (pass 2; D <= 128 runs accumulate_tc.cu).
//
// Page "det-attn", section "Method": rowmax_i = max_j (scale Q_i.K_j) is a max-reduce;
// NUM_id = sum_j exp(s_ij - rowmax_i) V_jd and DEN_i = sum_j exp(s_ij - rowmax_i) are
// exact integer sums in fixed bins, so any tiling, split or order gives the same bits.
//
// Exact scores come from integer-valued bf16 digit slices on the tensor cores (score_tc.cuh:
// mma.sync in the D = 256 accumulate kernel; tc5.cuh: tcgen05 in rowmax), rounded once.
//
// Exact PV.  The weight w in [0, 1] is held as W = w 2^92, three 31-bit limbs (exact for
// w >= 2^-69); V is fixed point per column over the call's key range, |Vint| < 2^23.  Per
// (i, d) three int64 accumulators take limb*Vint (< 2^54 each); every 256 keys the limbs
// carry into a fourth word in shared memory.  Products the window cannot hold (w < 2^-69,
// or a V element more than 15 binades below its column maximum) are added exactly with
// int64 atomics into the output digits; integer addition commutes, so this stays
// deterministic.  At the end each (i, d) is converted to canonical radix-2^32 digits.
#include "numerics.cuh"
#include "score_tc.cuh"
#include "tc5.cuh"
#include "attn_kernels.h"

namespace detattn {

// copy rows [kt, kt + nrow) of the prepared K slices into a smem slice tile; rows at or
// past hi are zero-filled (their pairs are masked)
template <int DP>
__device__ __forceinline__ void load_k_tile(const KvPrep& p, int64_t rowbase, int kt, int hi, int nrow, uint16_t* Ks,
                                            int LDS, int* Fk, unsigned char* kfit, int tid) {
  constexpr int CH = DP / 8;   // 16-byte chunks per slice row
  for (int c = tid; c < nrow * NSLICE * CH; c += 256) {
    const int r = c / (NSLICE * CH), q = (c / CH) % NSLICE, x = c % CH;
    const int j = kt + r;
    const bool ok = j < hi;
    const uint16_t* src = p.ksl + ((rowbase + (ok ? j : kt)) * NSLICE + q) * DP + 8 * x;
    cp_async16(Ks + q * nrow * LDS + r * LDS + 8 * x, src, ok ? 16 : 0);
  }
  for (int r = tid; r < nrow; r += 256) {
    const int j = kt + r;
    const int mv = j < hi ? p.kmeta[rowbase + j] : (1024 - 151) | (1 << 16);
    Fk[r] = kmeta_F(mv);
    kfit[r] = (unsigned char)kmeta_fit(mv);
  }
}

// =======================================================================================
// K1: rowmax on the tensor cores (tcgen05).
//
// The exact scores of a 128-key x 32-row block come from S^T = K Q^T on the 5th-generation
// tensor cores.  Per step of 16 dimensions, four MMAs of M = 128 keys x N = 128 x K = 16:
// A = key slice sa (the keys' bf16 digit slice sa, streamed from the prepared operand tiles
// by bulk copies into an 8-stage shared-memory ring), B = all four query slices stacked
// along N (row n = 32 sb + query row, resident), D_sa in TMEM (128 f32 columns each).  So
// D_sa[key][32 sb + row] = sum_d K_sa[key][d] Q_sb[row][d], an integer below 2^21; the seven
// diagonal sums A_c = sum_{sa+sb=c} D_sa[32 sb + row] are formed exactly in f32 by the
// epilogue (integers below 2^23), and the exact dot is sum_c 2^(7c) A_c.
//
// Roles (one CTA per SM): warp 16 lane 0 issues the bulk copies; warps 17 and 18 (lane 0)
// issue the MMAs of alternate steps (a tcgen05.commit holds its thread until that thread's
// MMAs are done, so the other issuer keeps the tensor pipe fed meanwhile).  Every MMA
// accumulates: warps 0-15 read TMEM (warp w: keys 32 (w % 4) .. +31 as its lanes, query rows
// 8 (w / 4) .. +7), zero what they read, release it, then score.
//
// Certified filter.  The diagonal sums are exact integers in f32, so T~ = Horner(A_c) in f32
// and B~ = Horner(|A_c|) bound the exact dot T: |T~ - T| <= 2^-21.3 B~, hence
// U = T~ + 2^-19 B~ (one fma) satisfies U >= T >= L = T~ - 2^-19 B~.  Both roundings of the
// score (to f32, then times scale) are monotone, so RN32(scale * U 2^E) bounds the exact score
// from above.  A pair whose bound does not exceed the row's running maximum (an exact score
// already found for that row, shared in shared memory after every key tile) cannot change
// the row maximum and skips the exact rounding;
// all others take the exact path (int64 dot, cr32_scaled).  A pair with a row outside the
// 26-bit window adds that row's few low limbs to the truncated dot (dot_lo, score_tc.cuh);
// a pair with a deep row is computed by its warp with the exact two-limb warp dot.  Every
// mbarrier wait is bounded; a wait that gives up sets DA_STATUS_TIMEOUT and the CTA winds
// down, freeing its TMEM.
// =======================================================================================
template <int DP>
struct RowmaxTcLayout {
  static constexpr int BM = 32, NDS = DP / 16, NST = 8, TCOLS = 512, NEPI = 16, NISS = 2;
  // warps: NEPI epilogue warps (four warpgroups) and one control warpgroup (the copy warp, NISS
  // MMA issuers, one idle warp).  The control warpgroup runs on 32 registers a thread, the
  // epilogue on 112 (640 x 96 at launch = 128 x 32 + 512 x 112); each role runs its own pass
  // loop, opened by named barrier 2 (query operand ready) and closed by barrier 3.
  static constexpr int LOADER = NEPI, ISS0 = NEPI + 1;
  static constexpr int THREADS = 32 * (NEPI + 4);
  static_assert(NISS <= 2, "the control warpgroup holds the copy warp and the issuers");
  static_assert(NDS % NISS == 0, "issuers split the steps of a tile evenly");
  static constexpr size_t q_step = (size_t)NSLICE * BM * 32;   // one B block: 4 slices x BM rows x 16 bf16
  static constexpr size_t q_bytes = (size_t)NDS * q_step;
  static constexpr size_t k_off = q_bytes;
  static constexpr size_t bytes = k_off + (size_t)NST * KT_BLOCK;
  static constexpr int SETC = NDIAG * BM;   // one set of diagonal sums: column BM c + row
  static_assert(2 * SETC <= TCOLS, "TMEM columns");
  static_assert(bytes <= 227 * 1024, "shared memory budget");
};

// true when the score RN32(scale * RN32(T 2^E)) cannot exceed `bound` and is finite
template <int N>
__device__ __forceinline__ bool score_below(const float (&v)[NDIAG][N], int r, int E, float scale, float bound) {
  if (E < -126 || E > 127) return false;
  float t = v[NDIAG - 1][r], m = fabsf(v[NDIAG - 1][r]);
#pragma unroll
  for (int c = NDIAG - 2; c >= 0; c--) {
    t = fmaf(t, 128.0f, v[c][r]);
    m = fmaf(m, 128.0f, fabsf(v[c][r]));
  }
  const float p2 = __int_as_float((E + 127) << 23);
  const float s1 = __fmul_rn(__fmul_rn(fmaf(m, 0x1p-19f, t), p2), scale);
  const float s2 = __fmul_rn(__fmul_rn(fmaf(m, -0x1p-19f, t), p2), scale);
  return fmaxf(s1, s2) <= bound && fminf(s1, s2) >= -3.4028235e38f;
}

// STORE: the score-cache variant (AttnArgs::scores).  Every valid pair's exact score is
// rounded (no filter) and written to its cache block; the row maximum is the maximum of
// those exact scores, so both variants produce the same rowmax.
template <int DT, int DP, bool STORE>
__global__ void __launch_bounds__(RowmaxTcLayout<DP>::THREADS, 1) rowmax_tc_kernel(const AttnArgs a, const KvPrep p) {
  using T = typename In<DT>::T;
  using L = RowmaxTcLayout<DP>;
  constexpr int BM = L::BM, NDS = L::NDS, NST = L::NST, NEPI = L::NEPI, NISS = L::NISS;
  constexpr int NQ = NSLICE * BM;   // MMA N: the stacked query slices
  constexpr uint32_t IDESC = tc5::idesc_bf16(KTILE, NQ);
  extern __shared__ __align__(1024) unsigned char smem_t[];
  unsigned char* Qs = smem_t;
  unsigned char* Kst = smem_t + L::k_off;
  __shared__ __align__(8) uint64_t full[NST], empty[NST], tfull[2], tempty[2], fin;
  __shared__ uint32_t tmem_s;
  __shared__ int Fq[BM], rkey[BM];
  __shared__ unsigned char qlon[BM];
  __shared__ int2 qlo[BM][NLO];
  __shared__ unsigned char qfit[BM];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // One query tile per CTA, the longest first: with causal masking tile q has q + 1 key
  // tiles, and the blocks start roughly in index order, so the longest tiles of every head
  // start first and the short ones fill the end of the launch (pairs of a long and a short
  // tile, equal in work, left the last partial wave of the launch idle behind them).
  const int ntq = (a.Sq + BM - 1) / BM, nbh = a.Hq * a.B;
  const int tq = (int)blockIdx.x / nbh, bh = (int)blockIdx.x % nbh;
  const int qtile = a.causal ? ntq - 1 - tq : tq;
  const int h = bh % a.Hq, b = bh / a.Hq, hk = h / (a.Hq / a.Hkv);
  const T* qbase = (const T*)a.q + b * a.qs[0] + h * a.qs[1];
  const T* kbase = (const T*)a.k + b * a.ks[0] + hk * a.ks[1];
  const int64_t krow0 = ((int64_t)b * a.Hkv + hk) * a.Skv;
  const unsigned char* ktc = p.ktc + (int64_t)(b * a.Hkv + hk) * p.ntk * NDS * KT_BLOCK;

  if (warp == 0) tc5::tmem_alloc(&tmem_s, L::TCOLS);
  if (tid == 0) {
    for (int s = 0; s < NST; s++) {
      tc5::mbar_init(&full[s], 1);
      tc5::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; s++) {   // two diagonal sets: one tile's MMAs run while the epilogue reads the last
      tc5::mbar_init(&tfull[s], NISS);
      tc5::mbar_init(&tempty[s], NEPI);
    }
    tc5::mbar_init(&fin, NISS);
    s_abort = 0;
    tc5::mbar_fence_init();
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  const uint32_t tmem = tmem_s;
  // every MMA accumulates: the epilogue warps keep their TMEM region zero between key tiles
  const uint32_t lbase = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (warp >> 2) * 8;
  if (warp < NEPI) {
#pragma unroll
    for (int c = 0; c < 2 * NDIAG; c++) tc5::st_zero_x8(lbase + c * BM);
    tc5::st_wait();
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();

  int nf = 0;
  uint32_t g_base = 0, tcount = 0;   // ring steps of earlier passes; key tiles seen by this thread's role
  const int npass = 1;
  if (warp >= NEPI) {   // ---------------- control warpgroup ----------------
    asm volatile("setmaxnreg.dec.sync.aligned.u32 32;" ::: "memory");
    for (int pass = 0; pass < npass; pass++) {
      const int q0 = qtile * BM;
      const int hi = a.causal ? min(a.kv_hi, q0 + BM) : a.kv_hi;
      const int nkt = hi > a.kv_lo ? (hi - a.kv_lo + KTILE - 1) / KTILE : 0;
      const uint32_t nsteps = (uint32_t)nkt * NDS;
      tc5::bar_sync(2, L::THREADS);
      if (warp == L::LOADER) {   // ---------------- bulk copies of the key operand tiles ----------------
        if (lane == 0)
          for (uint32_t ls = 0; ls < nsteps && !s_abort; ls++) {
            const uint32_t g_step = g_base + ls, st = g_step % NST;
            if (g_step >= NST && !tc5::mbar_wait(&empty[st], ((g_step / NST) - 1) & 1, &s_abort, 64)) break;
            tc5::mbar_expect_tx(&full[st], KT_BLOCK);
            tc5::bulk_g2s(Kst + st * KT_BLOCK, ktc + (size_t)ls * KT_BLOCK, KT_BLOCK, &full[st]);
          }
      } else if (warp < L::ISS0 + NISS) {   // ---------------- MMA issuers: steps ii, ii + NISS, ... ----------------
        if (lane == 0) {
          const uint32_t ii = warp - L::ISS0;
          for (uint32_t ls = ii; ls < nsteps && !s_abort; ls += NISS) {
            const uint32_t g_step = g_base + ls, st = g_step % NST;
            const int k = (int)(ls % NDS);
            if (!tc5::mbar_wait(&full[st], (g_step / NST) & 1, &s_abort, 32)) break;
            const uint32_t set = tcount & 1;
            if (k == (int)ii && tcount >= 2 && !tc5::mbar_wait(&tempty[set], ((tcount - 2) >> 1) & 1, &s_abort, 64)) break;
            tc5::fence_after();
            const uint64_t ka = tc5::desc(tc5::smem_addr(Kst + st * KT_BLOCK));
            const uint64_t qa = tc5::desc(tc5::smem_addr(Qs + k * L::q_step));
#pragma unroll
            for (int sa = 0; sa < NSLICE; sa++)   // D offset by BM per key slice: the diagonals add themselves
              tc5::mma_bf16(tmem + set * L::SETC + sa * BM, ka + (uint64_t)(sa * KTILE * 2), qa, IDESC, 1u);
            tc5::commit(&empty[st]);
            if (k + NISS >= NDS) {   // this issuer's last step of the tile
              tc5::commit(&tfull[set]);
              tcount++;
            }
          }
        }
      }
      g_base += nsteps;
      tc5::bar_sync(3, L::THREADS);
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 96;" ::: "memory");
  } else {   // ---------------- epilogue warps: thread = key, 8 query rows ----------------
    asm volatile("setmaxnreg.inc.sync.aligned.u32 112;" ::: "memory");
    for (int pass = 0; pass < npass; pass++) {
      const int q0 = qtile * BM;
      const int hi = a.causal ? min(a.kv_hi, q0 + BM) : a.kv_hi;
      const int nkt = hi > a.kv_lo ? (hi - a.kv_lo + KTILE - 1) / KTILE : 0;
    // ---- query slices into the resident B operand ----
    for (int r = warp; r < BM; r += NEPI) {
      const int i = q0 + r;
      row_slices<DT, DP>(
          i < a.Sq ? qbase + (int64_t)i * a.qs[2] : nullptr, a.D,
          [&](int q, int d, uint16_t v) {
            *reinterpret_cast<uint16_t*>(Qs + (d >> 4) * L::q_step + tc5::canon_off(q * BM + r, d & 15)) = v;
          },
          &Fq[r], &qfit[r], nf, lane, qlo[r], &qlon[r]);
    }
    for (int r = tid; r < BM; r += NEPI * 32) rkey[r] = float_key(neg_inf());
    tc5::fence_async_smem();
    tc5::bar_sync(2, L::THREADS);
    {
      const int quarter = warp & 3, rg = warp >> 2;
      const int jl = 32 * quarter + lane;
      // STORE: this thread's 8 rows all exist and fit their windows (then a tile whose keys all
      // fit and lie at or below every one of these rows takes the short path below)
      bool rows_clean = q0 + rg * 8 + 7 < a.Sq && fabsf(a.scale32) <= 1.0f;
      int fqr[8], fqmin = 1 << 20, fqmax = -(1 << 20);
#pragma unroll
      for (int r = 0; r < 8; r++) {
        rows_clean = rows_clean && qfit[rg * 8 + r];
        fqr[r] = Fq[rg * 8 + r];
        fqmin = min(fqmin, fqr[r]);
        fqmax = max(fqmax, fqr[r]);
      }
      float mrun[8];
#pragma unroll
      for (int r = 0; r < 8; r++) mrun[r] = neg_inf();
      // key meta words one tile ahead (the load's latency stays off the tile's path)
      int mv_n = (nkt > 0 && a.kv_lo + jl < hi) ? p.kmeta[krow0 + a.kv_lo + jl] : 0;
      for (int t = 0; t < nkt; t++) {
        const int j = a.kv_lo + t * KTILE + jl;
        const bool vj = j < hi;
        const int mv = mv_n;
        mv_n = (t + 1 < nkt && j + KTILE < hi) ? p.kmeta[krow0 + j + KTILE] : 0;
        const uint32_t set = tcount & 1;
        bool tok = true;
        if (lane == 0) tok = tc5::mbar_wait(&tfull[set], (tcount >> 1) & 1, &s_abort, 128);
        if (!__shfl_sync(0xFFFFFFFFu, tok, 0)) break;   // warp-uniform
        tc5::fence_after();
        float thr[8];   // the rows' running maxima so far (exact scores)
        if constexpr (!STORE) {
#pragma unroll
          for (int r = 0; r < 8; r++) thr[r] = fmaxf(mrun[r], key_float(rkey[rg * 8 + r]));
        }
        const int Fk = kmeta_F(mv), kf = kmeta_fit(mv);
        uint32_t defer = 0;   // rows whose pair with this key needs the exact fallback
        // score cache: this thread's 8 rows lie in query tile qt16 (rows rr0 .. rr0 + 7 of it);
        // under causal masking that tile may have one key tile fewer than the 32-row tile
        const int qt16 = q0 / SC_ROWS + (rg >> 1), rr0 = (rg & 1) * 8;
        bool sc_ok = false;
        float* sc_blk = nullptr;
        if constexpr (STORE) {
          const int hi16 = a.causal ? min(a.kv_hi, qt16 * SC_ROWS + SC_ROWS) : a.kv_hi;
          sc_ok = qt16 * SC_ROWS < a.Sq && t * KTILE < hi16 - a.kv_lo;
          if (sc_ok) sc_blk = a.scores + sc_block(a, b * a.Hq + h, qt16, t) * SC_BLOCK + jl * SC_ROWS + rr0;
        }
        // short path (STORE): every row and every key of this warp's tile that takes part is in its
        // window, and every E = Fq + Fk lies in [-126, 64]: then RN32(T) 2^E is a normal binary32
        // for every nonzero T (|T| < 2^63), so the score is RN32(scale * RN32(T) 2^E) with no
        // special case, and with |scale| <= 1 it is finite.  Masked pairs (a key past the range
        // or, under causal masking, after the row) store 0 and leave the maximum alone.
        const bool clean = STORE && __all_sync(0xFFFFFFFFu, rows_clean && (!vj || (kf && fqmin + Fk >= -126 && fqmax + Fk <= 64)));
        const bool all_valid = a.kv_lo + t * KTILE + KTILE <= hi &&
                               (!a.causal || a.kv_lo + t * KTILE + KTILE - 1 <= q0 + rg * 8);   // warp-uniform
        if (clean) {
#pragma unroll
          for (int hf = 0; hf < 2; hf++) {
            float v[NDIAG][4];
#pragma unroll
            for (int c = 0; c < NDIAG; c++) tc5::ld_x4(lbase + set * L::SETC + c * BM + 4 * hf, v[c]);
            tc5::ld_wait();
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
              const int r = 4 * hf + e;
              const int E = fqr[r] + Fk;
              const float c = __fmul_rn(__ll2float_rn(combine_diag(v, e)), __uint_as_float((uint32_t)(E + 127) << 23));
              float sc = __fmul_rn(a.scale32, c);
              if (!all_valid && !(vj && (!a.causal || j <= q0 + rg * 8 + r))) sc = 0.0f;   // masked (the row exists)
              else mrun[r] = sc > mrun[r] ? sc : mrun[r];
              o[e] = sc;
            }
            if (sc_ok) *reinterpret_cast<float4*>(sc_blk + 4 * hf) = make_float4(o[0], o[1], o[2], o[3]);
          }
        } else
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {   // rows 4 hf .. 4 hf + 3: half the diagonal sums live at a time
          float v[NDIAG][4];   // diagonal sums of these 4 rows, exact
#pragma unroll
          for (int c = 0; c < NDIAG; c++) tc5::ld_x4(lbase + set * L::SETC + c * BM + 4 * hf, v[c]);
          tc5::ld_wait();
          if constexpr (STORE) {   // every valid pair: its exact score, rounded once, into the cache
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
              const int r = 4 * hf + e, rl = rg * 8 + r, i = q0 + rl;
              float sc = 0.0f;
              if (vj && i < a.Sq && (!a.causal || j <= i)) {
                if (qfit[rl] && kf) {
                  const int E = Fq[rl] + Fk;
                  const long long T = combine_diag(v, e);
                  bool special;
                  float c = cr32_scaled_cvt(T, E, special);
                  if (special) c = cr32_scaled(T, E);   // subnormal or overflowing: the general rounding
                  sc = __fmul_rn(a.scale32, c);
                } else if (qlon[rl] != LO_DEEP && kmeta_lon(mv) != KLO_DEEP) {   // truncated dot + low limbs
                  sc = __fmul_rn(a.scale32, dot_lo<DT>(combine_diag(v, e), qbase + (int64_t)i * a.qs[2], Fq[rl],
                                                        qlo[rl], qlon[rl], kbase + (int64_t)j * a.ks[2], Fk,
                                                        p.klo + (krow0 + j) * NLO, kmeta_lon(mv)));
                } else {
                  defer |= 1u << rl;   // a deep row: the warp's exact dot below stores it
                }
                if (!((defer >> rl) & 1u)) {
                  if (!(fabsf(sc) <= 3.4028235e38f)) nf |= ST_NONFINITE;
                  mrun[r] = sc > mrun[r] ? sc : mrun[r];
                }
              }
              o[e] = sc;
            }
            if (sc_ok) *reinterpret_cast<float4*>(sc_blk + 4 * hf) = make_float4(o[0], o[1], o[2], o[3]);
          } else {
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const int r = 4 * hf + e, rl = rg * 8 + r, i = q0 + rl;
            if (vj && i < a.Sq && (!a.causal || j <= i)) {
              if (qfit[rl] && kf) {
                const int E = Fq[rl] + Fk;
                if (!score_below(v, e, E, a.scale32, thr[r])) {
                  const float sc = __fmul_rn(a.scale32, cr32_scaled(combine_diag(v, e), E));
                  if (!(fabsf(sc) <= 3.4028235e38f)) nf |= ST_NONFINITE;
                  mrun[r] = sc > mrun[r] ? sc : mrun[r];
                }
              } else if (qlon[rl] != LO_DEEP && kmeta_lon(mv) != KLO_DEEP) {   // truncated dot + low limbs
                const float sc = __fmul_rn(
                    a.scale32, dot_lo<DT>(combine_diag(v, e), qbase + (int64_t)i * a.qs[2], Fq[rl], qlo[rl], qlon[rl],
                                          kbase + (int64_t)j * a.ks[2], Fk, p.klo + (krow0 + j) * NLO, kmeta_lon(mv)));
                if (!(fabsf(sc) <= 3.4028235e38f)) nf |= ST_NONFINITE;
                mrun[r] = sc > mrun[r] ? sc : mrun[r];
              } else {
                defer |= 1u << rl;   // a deep row: the warp's exact dot below
              }
            }
          }
          }   // filter
        }
#pragma unroll
        for (int c = 0; c < NDIAG; c++) tc5::st_zero_x8(lbase + set * L::SETC + c * BM);
        tc5::st_wait();
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) tc5::mbar_arrive(&tempty[set]);
        tcount++;
        // deferred pairs of this warp, one at a time with the whole warp
        for (uint32_t pend = __ballot_sync(0xFFFFFFFFu, defer != 0); pend; pend = __ballot_sync(0xFFFFFFFFu, defer != 0)) {
          const int src = __ffs(pend) - 1;
          const uint32_t dm = __shfl_sync(0xFFFFFFFFu, defer, src);
          const int rl = __ffs(dm) - 1;
          const int jj = a.kv_lo + t * KTILE + 32 * quarter + src;
          const float sc = __fmul_rn(a.scale32, exact_dot_warp<DT>(qbase + (int64_t)(q0 + rl) * a.qs[2],
                                                                  kbase + (int64_t)jj * a.ks[2], a.D, lane));
          if (!(fabsf(sc) <= 3.4028235e38f)) nf |= ST_NONFINITE;
          if (lane == 0 && sc == sc) atomicMax(&rkey[rl], float_key(sc));
          if constexpr (STORE) {   // the lane that owns the key stored the pair's placeholder: overwrite it
            if (lane == src && sc_ok) sc_blk[rl - rg * 8] = sc;
          }
          if (lane == src) defer &= defer - 1;
        }
        if constexpr (!STORE) {
#pragma unroll
          for (int r = 0; r < 8; r++) {   // publish this tile's maxima
            const int km = __reduce_max_sync(0xFFFFFFFFu, float_key(mrun[r]));
            if (lane == 0 && key_float(km) > thr[r]) atomicMax(&rkey[rg * 8 + r], km);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 8; r++) {
        const int kmax = __reduce_max_sync(0xFFFFFFFFu, float_key(mrun[r]));
        if (lane == 0) atomicMax(&rkey[rg * 8 + r], kmax);
      }
    }
    tc5::bar_sync(1, NEPI * 32);   // every epilogue warp's maxima are in rkey
    if (tid < BM) {
      const int i = q0 + tid;
      float v = key_float(rkey[tid]);
      if (i < a.Sq) {
        if (v == 0.0f) v = __int_as_float(0);   // -0 -> +0
        a.m_out[((int64_t)b * a.Hq + h) * a.Sq + i] = v;
      }
    }
    tc5::bar_sync(3, L::THREADS);
    }
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
  }
  if (warp >= L::ISS0 && warp < L::ISS0 + NISS && lane == 0) {   // every MMA issued has completed before TMEM is released
    tc5::commit(&fin);
    tc5::mbar_wait(&fin, 0, &s_abort);
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  if (warp == 0) tc5::tmem_dealloc(tmem, L::TCOLS);
  if (s_abort) nf |= ST_TIMEOUT;
  report(a.status, nf);
}

// =======================================================================================
// K2: exact accumulate.
// =======================================================================================
template <int DP> struct AccCfg;
// RP x CP accumulators per thread; MINB CTAs per SM (register and shared-memory budget)
template <> struct AccCfg<64>  { static constexpr int RP = 4, CP = 2, MINB = 2; };
template <> struct AccCfg<128> { static constexpr int RP = 2, CP = 4, MINB = 2; };
template <> struct AccCfg<256> { static constexpr int RP = 2, CP = 8, MINB = 1; };

template <int DP>
struct AccLayout {
  static constexpr int RP = AccCfg<DP>::RP, CP = AccCfg<DP>::CP;
  static constexpr int BM = 8 * RP, BN = 32, LD = DP + 4, LDS = DP + 8, LDW = BM + 4;
  static constexpr size_t q_off = 0;                                          // bf16 [4][BM][LDS]
  static constexpr size_t k_off = q_off + sizeof(uint16_t) * NSLICE * BM * LDS;  // bf16 [4][BN][LDS]
  static constexpr size_t v_off = k_off + sizeof(uint16_t) * NSLICE * BN * LDS;  // int32 [BN][LD]
  static constexpr size_t w_off = v_off + sizeof(int) * BN * LD;                 // int32 [3][BN][LDW]
  static constexpr size_t wf_off = w_off + sizeof(int) * 3 * BN * LDW;           // float [BN][BM]
  static constexpr size_t p3_off = wf_off + sizeof(float) * BN * BM;             // int64 [BM][DP]
  static constexpr size_t vm_off = p3_off + sizeof(long long) * BM * DP;         // uint32 [BN][DP/32]
  static constexpr size_t ps_off = vm_off + sizeof(uint32_t) * BN * (DP / 32);    // uint16 [BN*BM] tiny weights
  static constexpr size_t ls_off = ps_off + sizeof(uint16_t) * BN * BM;           // uint16 [BN*BM] low limb set
  static constexpr size_t bytes = ls_off + sizeof(uint16_t) * BN * BM;
  static_assert(sizeof(long long) * BM * DP * 3 <= wf_off, "epilogue staging must fit in the tile area");
  static_assert(bytes <= 227 * 1024, "shared memory budget");
  static_assert(AccCfg<DP>::MINB == 1 || bytes + 8 * 1024 <= 113 * 1024, "two CTAs per SM");
};

// add a signed 64-bit X * 2^o into lazily carried radix-2^32 digits dg[]
__device__ __forceinline__ void digits_add_i64(long long* dg, long long X, int o) {
  unsigned long long lo = (unsigned long long)X & 0xFFFFFFFFull;
  long long hi = X >> 32;
  int k = o >> 5, r = o & 31;
  unsigned long long u = lo << r;
  dg[k] += (long long)(u & 0xFFFFFFFFull);
  dg[k + 1] += (long long)(u >> 32);
  long long v = hi * (1ll << r);
  dg[k + 1] += (long long)((unsigned long long)v & 0xFFFFFFFFull);
  dg[k + 2] += v >> 32;
}

template <int DT, int DP>
__global__ void __launch_bounds__(256, AccCfg<DP>::MINB) accumulate_kernel(const AttnArgs a, const KvPrep p) {
  using T = typename In<DT>::T;
  using L = AccLayout<DP>;
  constexpr int RP = L::RP, CP = L::CP, BM = L::BM, BN = L::BN, LD = L::LD, LDS = L::LDS, LDW = L::LDW;
  constexpr int NW = DP / 32, NT = (BM / 16) * (BN / 8);
  extern __shared__ __align__(16) unsigned char smem_b[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem_b + L::q_off);
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem_b + L::k_off);
  int* Vx = reinterpret_cast<int*>(smem_b + L::v_off);
  int* Wl = reinterpret_cast<int*>(smem_b + L::w_off);
  float* Wf = reinterpret_cast<float*>(smem_b + L::wf_off);
  long long* P3 = reinterpret_cast<long long*>(smem_b + L::p3_off);
  uint32_t* vmask = reinterpret_cast<uint32_t*>(smem_b + L::vm_off);
  uint16_t* plist = reinterpret_cast<uint16_t*>(smem_b + L::ps_off);
  uint16_t* llist = reinterpret_cast<uint16_t*>(smem_b + L::ls_off);
  __shared__ int Fq[BM], Fk[BN], Fv[DP];
  __shared__ unsigned char qfit[BM], kfit[BN];
  __shared__ float mrow[BM];
  __shared__ long long denT[BM][3];
  __shared__ int s_np, s_nl, s_nfix, s_vany, s_zeroed;
  __shared__ uint16_t flist[BM * BN];   // pairs outside the fixed-point window, this tile

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y, b = blockIdx.z, hk = h / (a.Hq / a.Hkv);
  // causal: CTA x takes query tiles x and T-1-x, so every CTA sees about the same keys
  const int ntiles = (a.Sq + BM - 1) / BM;
  const int npass = (a.causal && blockIdx.x != ntiles - 1 - blockIdx.x) ? 2 : 1;
  for (int pass = 0; pass < npass; pass++) {
  const int q0 = (pass == 0 ? ntiles - 1 - (int)blockIdx.x : (int)blockIdx.x) * BM;
  if (pass) __syncthreads();
  const T* qbase = (const T*)a.q + b * a.qs[0] + h * a.qs[1];
  const T* kbase = (const T*)a.k + b * a.ks[0] + hk * a.ks[1];
  const T* vbase = (const T*)a.v + b * a.vs[0] + hk * a.vs[1];
  const int64_t rowbase = ((int64_t)b * a.Hq + h) * a.Sq;
  long long* numb = a.num + rowbase * NUM_NDIG * a.D;
  long long* denb = a.den + rowbase * DEN_NDIG;
  const int nrows = min(BM, a.Sq - q0);
  int nf = 0, viol = 0;
  int lo = a.kv_lo, hi = a.kv_hi;
  if (a.causal) hi = min(hi, q0 + BM);

  // ---- set-up: Q tile, rowmax, per-column V exponent over [lo, hi) ----
  for (int r = warp; r < BM; r += 8) {
    int i = q0 + r;
    convert_row_slices<DT, DP>(i < a.Sq ? qbase + (int64_t)i * a.qs[2] : nullptr, a.D, Qs + r * LDS, BM * LDS, &Fq[r],
                               &qfit[r], nf, lane);
  }
  for (int r = tid; r < BM; r += 256) mrow[r] = (q0 + r < a.Sq) ? a.m_in[rowbase + q0 + r] : 0.0f;
  for (int e = tid; e < BM * DP; e += 256) P3[e] = 0;
  if (tid == 0) { s_zeroed = 0; }
  for (int d = tid; d < DP; d += 256)   // biased exponent in [1, 254]: |Vint| < 2^23, digit offsets in range
    Fv[d] = min(max(p.vcol[((int64_t)b * a.Hkv + hk) * DP + d], 1), 254) - 149;
  __syncthreads();

  // ---- accumulators ----
  long long acc[RP][CP][3];
#pragma unroll
  for (int r = 0; r < RP; r++)
#pragma unroll
    for (int c = 0; c < CP; c++)
#pragma unroll
      for (int l = 0; l < 3; l++) acc[r][c][l] = 0;
  if (tid < BM * 3) (&denT[0][0])[tid] = 0;
  const int g = lane >> 2, t = lane & 3;     // MMA fragment coordinates
  const int pr = warp, pc = lane;            // PV layout: rows pr*RP + r, cols pc*CP + c
  int tiles_since_carry = 0;

  auto carry_into_p3 = [&]() {
#pragma unroll
    for (int r = 0; r < RP; r++)
#pragma unroll
      for (int c = 0; c < CP; c++) {
        long long c0 = acc[r][c][0] >> 31;
        acc[r][c][0] -= c0 * (1ll << 31);
        acc[r][c][1] += c0;
        long long c1 = acc[r][c][1] >> 31;
        acc[r][c][1] -= c1 * (1ll << 31);
        acc[r][c][2] += c1;
        long long c2 = acc[r][c][2] >> 31;
        acc[r][c][2] -= c2 * (1ll << 31);
        P3[(pr * RP + r) * DP + pc * CP + c] += c2;
      }
  };

  const int64_t krow0 = ((int64_t)b * a.Hkv + hk) * a.Skv;
  auto weight_of = [&](float sc, float m, int& nfl, int& vio) -> float {
    float x = __fsub_rn(sc, m);
    if (x != x) { nfl |= ST_NONFINITE; x = neg_inf(); }
    if (x > 0.0f) { vio |= ST_VIOLATION; x = 0.0f; }
    return exp32_det(x);
  };
  // weight w of pair (rl, cl) -> limbs of W = w 2^92 in the Wl planes, the float in Wf,
  // its denominator limbs into dp; weights outside the limb window go to the lists
  auto store_weight = [&](float w, int rl, int cl, long long (&dp)[3]) {
    uint32_t wb = __float_as_uint(w);
    int ex = (int)(wb >> 23);
    int l0 = 0, l1 = 0, l2 = 0;
    if (wb != 0u) {
      if (ex >= 58) {
        unsigned __int128 W = ((unsigned __int128)((wb & 0x7FFFFFu) | 0x800000u)) << (ex - 58);
        l0 = (int)((uint64_t)W & 0x7FFFFFFFull);
        l1 = (int)((uint64_t)(W >> 31) & 0x7FFFFFFFull);
        l2 = (int)(uint64_t)(W >> 62);
        if (l0 != 0) llist[atomicAdd(&s_nl, 1)] = (uint16_t)(cl * BM + rl);   // w < 2^-38 (rare)
        dp[0] += l0;
        dp[1] += l1;
        dp[2] += l2;
      } else {
        plist[atomicAdd(&s_np, 1)] = (uint16_t)(cl * BM + rl);
      }
    }
    Wl[(0 * BN + cl) * LDW + rl] = l0;
    Wl[(1 * BN + cl) * LDW + rl] = l1;
    Wl[(2 * BN + cl) * LDW + rl] = l2;
    Wf[cl * BM + rl] = w;
  };

  for (int kt = lo; kt < hi; kt += BN) {
    __syncthreads();   // previous tile fully consumed
    // ---- K and V tiles: prepared rows, copied asynchronously ----
    load_k_tile<DP>(p, krow0, kt, hi, BN, Ks, LDS, Fk, kfit, tid);
    for (int c = tid; c < BN * (DP / 4); c += 256) {
      const int r = c / (DP / 4), x = c % (DP / 4), j = kt + r;
      const bool ok = j < hi;
      cp_async16(Vx + r * LD + 4 * x, p.vint + (krow0 + (ok ? j : kt)) * DP + 4 * x, ok ? 16 : 0);
    }
    for (int c = tid; c < BN * NW; c += 256) {
      const int r = c / NW, j = kt + r;
      vmask[c] = j < hi ? p.vbad[(krow0 + j) * NW + c % NW] : 0u;
    }
    cp_async_wait_all();
    if (tid == 0) { s_np = 0; s_nl = 0; s_nfix = 0; s_vany = 0; }
    __syncthreads();
    // ---- exact scores on the tensor cores, then weights ----
    for (int ot = warp; ot < NT; ot += 8) {
      const int r0 = 16 * (ot / (BN / 8)), n0 = 8 * (ot % (BN / 8));
      float sacc[NDIAG][4];
      score_tile_mma<DP>(sacc, Qs, BM * LDS, Ks, BN * LDS, LDS, r0, n0, g, t);
      long long dpart[2][3] = {{0, 0, 0}, {0, 0, 0}};
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int rl = r0 + g + 8 * (e >> 1), cl = n0 + 2 * t + (e & 1);
        const int i = q0 + rl, j = kt + cl;
        float w = 0.0f;
        if (i < a.Sq && j < hi && (!a.causal || j <= i)) {
          if (!(qfit[rl] && kfit[cl])) {   // a row outside the window: deferred to one warp below
            flist[atomicAdd(&s_nfix, 1)] = (uint16_t)(cl * BM + rl);
            continue;
          }
          float sc = __fmul_rn(a.scale32, cr32_scaled(combine_diag(sacc, e), Fq[rl] + Fk[cl]));
          w = weight_of(sc, mrow[rl], nf, viol);
        }
        store_weight(w, rl, cl, dpart[e >> 1]);
      }
#pragma unroll
      for (int hh = 0; hh < 2; hh++)
#pragma unroll
        for (int l = 0; l < 3; l++) {
          long long v = dpart[hh][l];
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
          if (t == 0 && v) atomicAdd((unsigned long long*)&denT[r0 + g + 8 * hh][l], (unsigned long long)v);
        }
    }
    if (lane == 0) {
      bool any = false;
      for (int e = warp; e < BN * NW; e += 8) any = any || (vmask[e] != 0u);
      if (any) s_vany = 1;
    }
    __syncthreads();
    if (s_nfix > 0) {   // deferred pairs: one warp each computes the exact score, then the weight
      for (int fe = warp; fe < s_nfix; fe += 8) {
        const int cl = flist[fe] / BM, rl = flist[fe] % BM;
        const float sc = __fmul_rn(a.scale32, exact_dot_warp<DT>(qbase + (int64_t)(q0 + rl) * a.qs[2],
                                                                kbase + (int64_t)(kt + cl) * a.ks[2], a.D, lane));
        if (lane == 0) {
          long long dp[3] = {0, 0, 0};
          store_weight(weight_of(sc, mrow[rl], nf, viol), rl, cl, dp);
#pragma unroll
          for (int l = 0; l < 3; l++)
            if (dp[l]) atomicAdd((unsigned long long*)&denT[rl][l], (unsigned long long)dp[l]);
        }
      }
      __syncthreads();
    }
    // ---- exact PV on the integer pipe: limbs 1 and 2 of every weight ----
#pragma unroll 2
    for (int j = 0; j < BN; j++) {
      int wv[2][RP];
      int vv[CP];
#pragma unroll
      for (int l = 0; l < 2; l++) {
        const int* wp = Wl + ((l + 1) * BN + j) * LDW + pr * RP;
        if constexpr (RP == 4) {
          int4 t4 = *reinterpret_cast<const int4*>(wp);
          wv[l][0] = t4.x; wv[l][1] = t4.y; wv[l][2] = t4.z; wv[l][3] = t4.w;
        } else {
          int2 t2 = *reinterpret_cast<const int2*>(wp);
          wv[l][0] = t2.x; wv[l][1] = t2.y;
        }
      }
      const int* vp = Vx + j * LD + pc * CP;
      if constexpr (CP == 2) {
        int2 t2 = *reinterpret_cast<const int2*>(vp);
        vv[0] = t2.x; vv[1] = t2.y;
      } else {
#pragma unroll
        for (int c4 = 0; c4 < CP; c4 += 4) {
          int4 t4 = *reinterpret_cast<const int4*>(vp + c4);
          vv[c4] = t4.x; vv[c4 + 1] = t4.y; vv[c4 + 2] = t4.z; vv[c4 + 3] = t4.w;
        }
      }
#pragma unroll
      for (int r = 0; r < RP; r++)
#pragma unroll
        for (int c = 0; c < CP; c++)
#pragma unroll
          for (int l = 0; l < 2; l++) mad_wide(acc[r][c][l + 1], wv[l][r], vv[c]);
    }
    // ---- limb 0 is nonzero only for weights below 2^-38: the listed pairs of this tile ----
    {
      const int nl = s_nl;
      for (int e = 0; e < nl; e++) {
        const int cl = llist[e] / BM, rl = llist[e] % BM;
        if (rl / RP != pr) continue;   // another warp's row
        const int w0 = Wl[(0 * BN + cl) * LDW + rl];
        const int* vp = Vx + cl * LD + pc * CP;
#pragma unroll
        for (int r = 0; r < RP; r++)
          if (rl == pr * RP + r)
#pragma unroll
            for (int c = 0; c < CP; c++) mad_wide(acc[r][c][0], w0, vp[c]);
      }
    }
    if (++tiles_since_carry == 256 / BN) {   // 256 keys: limb sums stay below 2^62
      carry_into_p3();
      tiles_since_carry = 0;
    }
    // ---- products outside the window: exact int64 atomics into the output digits ----
    if (s_np > 0 || s_vany) {
      if (!s_zeroed) {
        if (!a.add_into) {
          for (int64_t e = tid; e < (int64_t)nrows * NUM_NDIG * a.D; e += 256) numb[(int64_t)q0 * NUM_NDIG * a.D + e] = 0;
          for (int e = tid; e < nrows * DEN_NDIG; e += 256) denb[(int64_t)q0 * DEN_NDIG + e] = 0;
        }
        __syncthreads();
        if (tid == 0) s_zeroed = 1;
      }
      const int np = s_np;
      for (int e = warp; e < np; e += 8) {
        const int cl = plist[e] / BM, rl = plist[e] % BM;
        const int i = q0 + rl, j = kt + cl;
        Split sw = split_f32(__float_as_uint(Wf[cl * BM + rl]));
        long long* nrow = numb + (int64_t)i * NUM_NDIG * a.D;
        for (int d = lane; d < a.D; d += 32) {
          uint32_t u = In<DT>::bits(vbase + (int64_t)j * a.vs[2], d);
          if (nonfinite_bits(u)) continue;
          Split sv = split_f32(u);
          atomic_digits_add(nrow + d, a.D, NUM_E0, (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
        }
        if (lane == 0) atomic_digits_add(denb + (int64_t)i * DEN_NDIG, 1, DEN_E0, sw.mant, 0, sw.lsb);
      }
      if (s_vany) {
        for (int e = tid; e < BN * NW; e += 256) {
          uint32_t m = vmask[e];
          const int cl = e / NW, t = e % NW, j = kt + cl;
          while (m) {
            const int bit = __ffs(m) - 1;
            m &= m - 1;
            const int d = t * 32 + bit;
            Split sv = split_f32(In<DT>::bits(vbase + (int64_t)j * a.vs[2], d));
            for (int rl = 0; rl < BM; rl++) {
              uint32_t wb = __float_as_uint(Wf[cl * BM + rl]);
              if (wb == 0u || (int)(wb >> 23) < 58) continue;   // zero, or already a pair spill
              Split sw = split_f32(wb);
              atomic_digits_add(numb + (int64_t)(q0 + rl) * NUM_NDIG * a.D + d, a.D, NUM_E0,
                                (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
            }
          }
        }
      }
    }
  }

  // ---- epilogue: canonical digits ----
  carry_into_p3();
  __syncthreads();   // tiles consumed; the tile area becomes the staging area below
  long long* stage = reinterpret_cast<long long*>(smem_b);   // [BM][DP][3], fits in the Q/K/V/W tiles
#pragma unroll
  for (int r = 0; r < RP; r++)
#pragma unroll
    for (int c = 0; c < CP; c++)
#pragma unroll
      for (int l = 0; l < 3; l++) stage[((pr * RP + r) * DP + pc * CP + c) * 3 + l] = acc[r][c][l];
  __syncthreads();   // staging, P3, denT and every spill atomic complete
  const bool rmw = a.add_into || s_zeroed;
  for (int e = tid; e < BM * DP; e += 256) {
    const int rl = e / DP, d = e % DP, i = q0 + rl;
    if (i >= a.Sq || d >= a.D) continue;
    long long* nrow = numb + (int64_t)i * NUM_NDIG * a.D;
    long long dg[NUM_NDIG + 3];
#pragma unroll
    for (int k = 0; k < NUM_NDIG + 3; k++) dg[k] = 0;
    if (rmw)
#pragma unroll
      for (int k = 0; k < NUM_NDIG; k++) dg[k] = __ldcg(nrow + (int64_t)k * a.D + d);
    const int off = Fv[d] - 92 - NUM_E0;   // bit position of the accumulator's unit
    digits_add_i64(dg, stage[e * 3 + 0], off);
    digits_add_i64(dg, stage[e * 3 + 1], off + 31);
    digits_add_i64(dg, stage[e * 3 + 2], off + 62);
    digits_add_i64(dg, P3[e], off + 93);
    kul_carry(dg, NUM_NDIG + 3);
    long long top = dg[NUM_NDIG + 2];
    bool bad = false;
    for (int k = NUM_NDIG + 1; k >= NUM_NDIG - 1; k--) {
      if (top > (1ll << 30) || top < -(1ll << 30)) bad = true;
      top = top * 4294967296ll + dg[k];
    }
    if (bad) nf |= ST_HEADROOM;
#pragma unroll
    for (int k = 0; k < NUM_NDIG - 1; k++) nrow[(int64_t)k * a.D + d] = dg[k];
    nrow[(int64_t)(NUM_NDIG - 1) * a.D + d] = top;
  }
  for (int rl = tid; rl < nrows; rl += 256) {
    long long* drow = denb + (int64_t)(q0 + rl) * DEN_NDIG;
    long long dg[DEN_NDIG + 3];
#pragma unroll
    for (int k = 0; k < DEN_NDIG + 3; k++) dg[k] = 0;
    if (rmw)
#pragma unroll
      for (int k = 0; k < DEN_NDIG; k++) dg[k] = __ldcg(drow + k);
    const int off = -92 - DEN_E0;
    digits_add_i64(dg, denT[rl][0], off);
    digits_add_i64(dg, denT[rl][1], off + 31);
    digits_add_i64(dg, denT[rl][2], off + 62);
    kul_carry(dg, DEN_NDIG + 3);
    long long top = dg[DEN_NDIG + 2];
    bool bad = false;
    for (int k = DEN_NDIG + 1; k >= DEN_NDIG - 1; k--) {
      if (top > (1ll << 30) || top < -(1ll << 30)) bad = true;
      top = top * 4294967296ll + dg[k];
    }
    if (bad) nf |= ST_HEADROOM;
#pragma unroll
    for (int k = 0; k < DEN_NDIG - 1; k++) drow[k] = dg[k];
    drow[DEN_NDIG - 1] = top;
  }
  report(a.status, nf | viol);
  nf = 0;
  viol = 0;
  }   // pass
}

// ---------------------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------------------
template <int DT, int DP, bool STORE>
static cudaError_t launch_rowmax_t(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  using L = RowmaxTcLayout<DP>;
  const size_t smem = L::bytes;
  cudaError_t e =
      cudaFuncSetAttribute(rowmax_tc_kernel<DT, DP, STORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int nt = (a.Sq + L::BM - 1) / L::BM;
  const int64_t nblocks = (int64_t)nt * a.Hq * a.B;   // one query tile per CTA
  rowmax_tc_kernel<DT, DP, STORE><<<(unsigned)nblocks, L::THREADS, smem, st>>>(a, p);
  return cudaGetLastError();
}

template <int DT, int DP>
static cudaError_t launch_rowmax_t(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  if constexpr (DP == 128) {
    if (a.scores) return launch_rowmax_t<DT, DP, true>(a, p, st);
  }
  return launch_rowmax_t<DT, DP, false>(a, p, st);
}

size_t score_cache_bytes(int B, int Hq, int Sq, int Skv, int causal, int* sc_nkt, int64_t* sc_per_bh) {
  const int64_t nqt = (Sq + SC_ROWS - 1) / SC_ROWS;
  int64_t per_bh;
  *sc_nkt = (Skv + KTILE - 1) / KTILE;
  if (causal) {
    if (Sq != Skv) return 0;
    const int64_t q = nqt - 1, g = q >> 3, r = q & 7;
    per_bh = nqt == 0 ? 0 : q + 4 * g * (g - 1) + r * g + (Sq + KTILE - 1) / KTILE;
  } else {
    per_bh = nqt * *sc_nkt;
  }
  *sc_per_bh = per_bh;
  return (size_t)B * Hq * per_bh * SC_BLOCK * sizeof(float);
}

template <int DT, int DP>
static cudaError_t launch_accumulate_t(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  using L = AccLayout<DP>;
  const size_t smem = L::bytes;
  cudaError_t e =
      cudaFuncSetAttribute(accumulate_kernel<DT, DP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int nt = (a.Sq + L::BM - 1) / L::BM;
  dim3 grid(a.causal ? (nt + 1) / 2 : nt, a.Hq, a.B);
  accumulate_kernel<DT, DP><<<grid, 256, smem, st>>>(a, p);
  return cudaGetLastError();
}

// D <= 128 runs on the 128-wide tensor-core kernels (the padding columns are zero: the exact
// sums are unchanged, and the per-pair work, not the MMA width, sets their time), D <= 256 on
// the 256-wide ones
static int padded_d(int D) { return D <= 128 ? 128 : 256; }

cudaError_t launch_rowmax(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  const int dp = padded_d(a.D);
  if (a.dtype == 0) {
    if (dp == 64) return launch_rowmax_t<0, 64>(a, p, st);
    if (dp == 128) return launch_rowmax_t<0, 128>(a, p, st);
    return launch_rowmax_t<0, 256>(a, p, st);
  }
  if (dp == 64) return launch_rowmax_t<1, 64>(a, p, st);
  if (dp == 128) return launch_rowmax_t<1, 128>(a, p, st);
  return launch_rowmax_t<1, 256>(a, p, st);
}

bool accumulate_is_tp(const AttnArgs& a, const KvPrep& p) {
  return padded_d(a.D) == 128 && p.vtc != nullptr && (a.kv_hi - a.kv_lo + KTILE - 1) / KTILE <= ACC_TP_MAX_TILES;
}

cudaError_t launch_accumulate(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  const int dp = padded_d(a.D);
  if (accumulate_is_tp(a, p)) return launch_accumulate_tp(a, p, st);
  if (a.out) return cudaErrorInvalidValue;   // only the tensor-PV kernel finalizes in its epilogue
  if (dp <= 128) return launch_accumulate_tc(a, p, st);
  return a.dtype == 0 ? launch_accumulate_t<0, 256>(a, p, st) : launch_accumulate_t<1, 256>(a, p, st);
}

}  // namespace detattn
