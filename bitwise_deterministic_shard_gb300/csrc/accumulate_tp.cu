// K2 with both products on the tensor cores (sm_103a): exact accumulate of NUM / DEN
// digits for 64 < D <= 128.
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
// A_c = sum_{sa+sb=c} sum_d K_sa Q_sb (integers below 2^22, exact in f32).
//
// PV.  Every weight w >= 2^-56 is held as W = w 2^79, an integer below 2^80, split into
// ten base-256 digits W_s (bytes, exact in f16); V is fixed point per column, |Vint| < 2^23,
// split into three balanced base-256 digits V_t (|V_t| <= 128, prepared once per call).
// The ten weight digit planes of a 16-key block lie next to each other along N (n = 16 s +
// row, MN-major), so one MMA of M = 128 value columns x N = 160 x K = 16 multiplies V digit
// t by all ten; written at column offset 16 t it adds V_t W_s into the diagonal sum
// P_c (c = s + t) at column 16 c + row.  Three MMAs per 16 keys, plus one with an all-ones
// A operand whose rows all receive DEN's digit sums sum_k W_s.  A product is at most
// 255 * 128 and a diagonal holds at most 3 per key, so over one 128-key tile every partial
// sum is an integer below 128 * 3 * 32640 < 2^24: exact.  After each tile the compute warps
// fold sum_c P_c 2^(8c) into three radix-2^32 int64 digits per (row, column) and the DEN
// planes into int32 sums, then zero the accumulators.  The weight digit planes are
// double-buffered, so the PV MMAs of one tile run while the next tile's weights are
// computed.  Products outside the window (w < 2^-56, or a V element below its column
// window) are added with exact int64 atomics into the output digits.
//
// Roles: warp 16 copies (lane 0: key operand steps, 4-stage ring; lane 1: V digit blocks,
// 3-stage ring), warp 17 lane 0 issues the score MMAs, warp 18 lane 0 the PV and DEN MMAs.
// Warps 0-15 read the score diagonals, compute weights, write the weight digit planes and
// drain the PV accumulators; each zeroes the TMEM it read before releasing it, so every MMA
// accumulates.  Every mbarrier wait is bounded; one that gives up sets DA_STATUS_TIMEOUT,
// and a failed wait in the compute warps only skips work so every named barrier is still
// passed.  The three int64 state digits stay exact for up to ACC_TP_MAX_TILES key tiles per
// pass; longer key ranges take the integer-pipe kernel.
#include "numerics.cuh"
#include "score_tc.cuh"
#include "tc5.cuh"
#include "attn_kernels.h"

namespace detattn {

struct AccTpLayout {
  static constexpr int DP = 128, BM = 16, NDS = DP / 16, NSK = 4, NVB = 3, NCW = 16;
  static constexpr int LOADW = NCW, SISS = NCW + 1, PISS = NCW + 2, THREADS = 32 * (NCW + 3);
  static constexpr int NWP = 10, NVP = 3, NPD = NWP + NVP - 1, NKB = KTILE / VKEYS;
  static constexpr int NQ = NSLICE * BM;                              // score MMA N: the stacked query slices
  static constexpr int NW16 = NWP * BM;                               // PV MMA N: the stacked weight digits
  // TMEM columns: PV diagonals P_c at 16 c, DEN digit sums at 16 s, score diagonals at 16 c
  static constexpr int PV_COL = 0, DEN_COL = PV_COL + NPD * BM, SC_COL = DEN_COL + NWP * BM, TCOLS = 512;
  static constexpr size_t q_step = (size_t)NQ * 32;                    // one B block: 64 rows (16 sb + r) x 16 bf16
  static constexpr size_t q_bytes = (size_t)NDS * q_step;
  static constexpr size_t k_off = q_bytes;                             // NSK key operand steps
  static constexpr size_t v_off = k_off + (size_t)NSK * KT_BLOCK;      // NVB V digit blocks
  static constexpr size_t w_blk = (size_t)BM * VKEYS * 2;              // one weight digit plane: 16 rows x 16 keys
  static constexpr size_t w_buf = (size_t)NKB * NWP * w_blk;           // one tile's weight digit planes [kb][s]
  static constexpr size_t w_off = v_off + (size_t)NVB * VP_BLOCK;      // two buffers
  static constexpr size_t one_off = w_off + 2 * w_buf;                 // 128 x 16 f16 ones (DEN's A operand)
  static constexpr size_t wf_off = one_off + (size_t)DP * 16 * 2;      // float [KTILE][BM] weights
  static constexpr size_t ps_off = wf_off + (size_t)BM * KTILE * 4;    // uint16 pairs below 2^-56
  static constexpr size_t bytes = ps_off + (size_t)KTILE * BM * 2;
  static constexpr int NBAD = 1024;
  static_assert(SC_COL + NDIAG * BM <= TCOLS, "TMEM columns");
  static_assert(NW16 <= 256 && NW16 % 16 == 0, "one PV MMA covers every weight digit");
  static_assert(KTILE * (DP / 32) == 32 * NCW, "one V-bad word per compute thread");
  static_assert(bytes <= 213 * 1024, "shared memory budget (plus about 8 KB static)");
};

// one 16-key block: V digit t (A) times the ten stacked weight digits (B) into P_{s+t}, and
// the ones block times the weight digits into the DEN sums
__device__ __forceinline__ void pv_block_mmas(uint32_t tmem, const unsigned char* vblk, const unsigned char* wblk,
                                              uint64_t ones, uint32_t idesc) {
  using L = AccTpLayout;
  const uint64_t va = tc5::desc(tc5::smem_addr(vblk));
  const uint64_t wa = tc5::desc(tc5::smem_addr(wblk));
#pragma unroll
  for (int t = 0; t < L::NVP; t++)   // descriptor start addresses advance in 16-byte units
    tc5::mma_bf16(tmem + L::PV_COL + t * L::BM, va + (uint64_t)(t * (VP_BLOCK / 3) / 16), wa, idesc, 1u);
  tc5::mma_bf16(tmem + L::DEN_COL, ones, wa, idesc, 1u);
}

// two f16 values b0, b1 in [0, 255] from the pattern (0x64 b1 0x64 b0): (1024 + b) - 1024
__device__ __forceinline__ uint32_t f16_pair_from_biased(uint32_t h) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64006400u));
  return r;
}

__device__ __forceinline__ void add_i64_at_tp(long long* dg, long long X, int o) {
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

template <int DT>
__global__ void __launch_bounds__(AccTpLayout::THREADS, 1) accumulate_tp_kernel(const AttnArgs a, const KvPrep p) {
  using T = typename In<DT>::T;
  using L = AccTpLayout;
  constexpr int DP = L::DP, BM = L::BM, NDS = L::NDS, NSK = L::NSK, NVB = L::NVB, NCW = L::NCW;
  constexpr int NKB = L::NKB, NWP = L::NWP, NW = DP / 32;
  constexpr int NCT = 32 * NCW;
  constexpr int NQ = L::NQ;
  constexpr uint32_t IDESC_S = tc5::idesc_bf16(KTILE, NQ);        // scores: 128 keys x (4 slices x 16 rows)
  constexpr uint32_t IDESC_P = tc5::idesc_f16(DP, L::NW16, true);   // PV: 128 columns x (10 digits x 16 rows)
  extern __shared__ __align__(1024) unsigned char smem_p[];
  unsigned char* Qs = smem_p;
  unsigned char* Kst = smem_p + L::k_off;
  unsigned char* Vst = smem_p + L::v_off;
  unsigned char* Wp = smem_p + L::w_off;
  float* Wf = reinterpret_cast<float*>(smem_p + L::wf_off);
  uint16_t* plist = reinterpret_cast<uint16_t*>(smem_p + L::ps_off);
  __shared__ __align__(8) uint64_t kfull[NSK], kempty[NSK], sfull, sempty, vfull[NVB], vempty[NVB], wready[2], pvdone,
      pvfree, fin;
  __shared__ uint32_t tmem_s;
  __shared__ int Fq[BM], Fv[DP];
  __shared__ unsigned char qfit[BM], qlon[BM];
  __shared__ int2 qlo[BM][NLO];
  __shared__ float mrow[BM];
  __shared__ long long denT[BM][3];
  __shared__ uint32_t vmask[KTILE * NW];
  __shared__ uint32_t badl[L::NBAD];
  __shared__ int s_np[2], s_nbad[2], s_vany[2], s_zeroed;   // per tile parity
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y, b = blockIdx.z, hk = h / (a.Hq / a.Hkv);
  const T* qbase = (const T*)a.q + b * a.qs[0] + h * a.qs[1];
  const T* kbase = (const T*)a.k + b * a.ks[0] + hk * a.ks[1];
  const T* vbase = (const T*)a.v + b * a.vs[0] + hk * a.vs[1];
  const int64_t krow0 = ((int64_t)b * a.Hkv + hk) * a.Skv;
  const unsigned char* ktc = p.ktc + (int64_t)(b * a.Hkv + hk) * p.ntk * NDS * KT_BLOCK;
  const unsigned char* vtc = p.vtc + (int64_t)(b * a.Hkv + hk) * p.ntk * NKB * VP_BLOCK;
  const int64_t rowbase = ((int64_t)b * a.Hq + h) * a.Sq;
  long long* numb = a.num + rowbase * NUM_NDIG * a.D;
  long long* denb = a.den + rowbase * DEN_NDIG;

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
    tc5::mbar_init(&sfull, 1);
    tc5::mbar_init(&sempty, NCW);
    tc5::mbar_init(&pvdone, 1);
    tc5::mbar_init(&pvfree, NCW);
    tc5::mbar_init(&fin, 2);   // the score issuer and the PV issuer
    s_abort = 0;
    tc5::mbar_fence_init();
  }
  for (int d = tid; d < DP; d += L::THREADS)   // biased exponent in [1, 254]: |Vint| < 2^23, digit offsets in range
    Fv[d] = min(max(p.vcol[((int64_t)b * a.Hkv + hk) * DP + d], 1), 254) - 149;
  for (int e = tid; e < DP * 16 / 2; e += L::THREADS)   // f16 1.0 pairs: DEN's all-ones A operand
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
    for (int c = 0; c < L::NPD; c++) tc5::st_zero_x4(lane_base + L::PV_COL + c * BM + rg * 4);
#pragma unroll
    for (int c = 0; c < NWP; c++) tc5::st_zero_x4(lane_base + L::DEN_COL + c * BM + rg * 4);
#pragma unroll
    for (int c = 0; c < NDIAG; c++) tc5::st_zero_x4(lane_base + L::SC_COL + c * BM + rg * 4);
    tc5::st_wait();
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();

  int nf = 0, viol = 0;
  uint32_t tc = 0;   // key tiles of earlier passes
  const int ntq = (a.Sq + BM - 1) / BM;
  const int npass = (a.causal && (int)blockIdx.x != ntq - 1 - (int)blockIdx.x) ? 2 : 1;
  for (int pass = 0; pass < npass; pass++) {
    const int q0 = (pass == 0 ? ntq - 1 - (int)blockIdx.x : (int)blockIdx.x) * BM;
    const int hi = a.causal ? min(a.kv_hi, q0 + BM) : a.kv_hi;
    const int nkt = hi > a.kv_lo ? (hi - a.kv_lo + KTILE - 1) / KTILE : 0;
    const int nrows = min(BM, a.Sq - q0);
    // ---- per pass: query slices (resident B operand of the scores), row maxima, cleared sums ----
    for (int r = warp; r < BM; r += L::THREADS / 32) {
      const int i = q0 + r;
      row_slices<DT, DP>(
          i < a.Sq ? qbase + (int64_t)i * a.qs[2] : nullptr, a.D,
          [&](int q, int d, uint16_t v) {
            *reinterpret_cast<uint16_t*>(Qs + (d >> 4) * L::q_step + tc5::canon_off(q * BM + r, d & 15)) = v;
          },
          &Fq[r], &qfit[r], nf, lane, qlo[r], &qlon[r]);
    }
    for (int r = tid; r < BM; r += L::THREADS) mrow[r] = (q0 + r < a.Sq) ? a.m_in[rowbase + q0 + r] : 0.0f;
    for (int e = tid; e < BM * 3; e += L::THREADS) (&denT[0][0])[e] = 0;
    if (tid < 2) { s_np[tid] = 0; s_nbad[tid] = 0; s_vany[tid] = 0; }
    if (tid == 0) s_zeroed = 0;
    tc5::fence_async_smem();
    __syncthreads();

    if (warp == L::LOADW) {   // ---------------- bulk copies ----------------
      if (lane == 0) {   // key operand steps
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
    } else if (warp == L::SISS) {   // ---------------- score MMAs ----------------
      if (lane == 0)
        for (int ls = 0; ls < nkt * NDS && !s_abort; ls++) {
          const uint32_t g = tc * NDS + ls, st = g % NSK, tt = tc + ls / NDS;
          const int k = ls % NDS;
          if (!tc5::mbar_wait(&kfull[st], (g / NSK) & 1, &s_abort, 32)) break;
          if (k == 0 && tt >= 1 && !tc5::mbar_wait(&sempty, (tt - 1) & 1, &s_abort, 64)) break;
          tc5::fence_after();
          const uint64_t ka = tc5::desc(tc5::smem_addr(Kst + st * KT_BLOCK));
          const uint64_t qa = tc5::desc(tc5::smem_addr(Qs + k * L::q_step));
#pragma unroll
          for (int sa = 0; sa < NSLICE; sa++)   // descriptor start addresses advance in 16-byte units
            tc5::mma_bf16(tmem + L::SC_COL + sa * BM, ka + (uint64_t)(sa * KTILE * 2), qa, IDESC_S, 1u);
          tc5::commit(&kempty[st]);
          if (k == NDS - 1) tc5::commit(&sfull);
        }
    } else if (warp == L::PISS) {   // ---------------- PV and DEN MMAs ----------------
      if (lane == 0) {
        const uint64_t ones = tc5::desc(tc5::smem_addr(smem_p + L::one_off));
        for (int t = 0; t < nkt && !s_abort; t++) {
          const uint32_t tt = tc + t, bsel = tt & 1;
          if (!tc5::mbar_wait(&wready[bsel], (tt >> 1) & 1, &s_abort, 64)) break;   // weight digits of tile tt
          if (tt >= 1 && !tc5::mbar_wait(&pvfree, (tt - 1) & 1, &s_abort, 64)) break;   // accumulators drained
          tc5::fence_after();
          for (int kb = 0; kb < NKB && !s_abort; kb++) {
            const uint32_t g = tt * NKB + kb, sl = g % NVB;
            if (!tc5::mbar_wait(&vfull[sl], (g / NVB) & 1, &s_abort, 32)) break;
            tc5::fence_after();
            pv_block_mmas(tmem, Vst + sl * VP_BLOCK, Wp + bsel * L::w_buf + (size_t)kb * NWP * L::w_blk, ones, IDESC_P);
            tc5::commit(&vempty[sl]);
          }
          tc5::commit(&pvdone);
        }
      }
    } else {   // ---------------- compute warps ----------------
      // Weight phase: this thread's key is TMEM lane dcol (rows 4 rg .. 4 rg + 3).  Drain: it
      // owns value column d = dcol; acc[r][k] is radix-2^32 digit k (lazily carried) in units
      // of 2^(Fv[d] - 79).
      const int dcol = 32 * quarter + lane;
      long long acc[4][3];
#pragma unroll
      for (int r = 0; r < 4; r++)
#pragma unroll
        for (int k = 0; k < 3; k++) acc[r][k] = 0;
      auto weight_of = [&](float sc, float m) -> float {
        float x = __fsub_rn(sc, m);
        if (x != x) { nf |= ST_NONFINITE; x = neg_inf(); }
        if (x > 0.0f) { viol |= ST_VIOLATION; x = 0.0f; }
        return exp32_det(x);
      };
      // lane 0 waits, the warp follows
      auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        bool ok = true;
        if (lane == 0) ok = tc5::mbar_wait(bar, parity, &s_abort, 64);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        tc5::fence_after();
        return ok;
      };
      // fold the PV and DEN accumulators of one tile into the integer sums, zero them, release them
      auto drain = [&](uint32_t tt) {
        if (warp_wait(&pvdone, tt & 1)) {
#pragma unroll
          for (int g3 = 0; g3 < 3; g3++) {   // diagonals 4 g3 .. 4 g3 + 3 -> digit g3
            float pv[4][4];
#pragma unroll
            for (int c = 0; c < 4; c++) tc5::ld_x4(lane_base + L::PV_COL + (4 * g3 + c) * BM + rg * 4, pv[c]);
            tc5::ld_wait();
#pragma unroll
            for (int r = 0; r < 4; r++) {
              long long s = 0;
#pragma unroll
              for (int c = 0; c < 4; c++) s += (long long)__float2int_rn(pv[c][r]) * (1ll << (8 * c));   // |P_c| < 2^24
              acc[r][g3] += s;
            }
          }
          // DEN: this warp folds planes quarter + 4 k (every lane holds the same sums); plane
          // s weighs 2^(8 s) = 2^(32 k + 8 quarter) in units of 2^-79
          float dv[3][4];
#pragma unroll
          for (int k = 0; k < 3; k++)
            if (quarter + 4 * k < NWP) tc5::ld_x4(lane_base + L::DEN_COL + (quarter + 4 * k) * BM + rg * 4, dv[k]);
          tc5::ld_wait();
          if (lane == 0)
#pragma unroll
            for (int k = 0; k < 3; k++)
              if (quarter + 4 * k < NWP)
#pragma unroll
                for (int r = 0; r < 4; r++) {
                  const int sv = __float2int_rn(dv[k][r]);   // < 2^15
                  if (sv) atomicAdd((unsigned long long*)&denT[rg * 4 + r][k], (unsigned long long)sv << (8 * quarter));
                }
#pragma unroll
          for (int c = 0; c < L::NPD; c++) tc5::st_zero_x4(lane_base + L::PV_COL + c * BM + rg * 4);
#pragma unroll
          for (int c = 0; c < NWP; c++) tc5::st_zero_x4(lane_base + L::DEN_COL + c * BM + rg * 4);
          tc5::st_wait();
        }
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) tc5::mbar_arrive(&pvfree);
      };
      // key meta of this thread's key and V-bad word tid of tile t (zeros past the range)
      auto tile_meta = [&](int t, int& mv, uint32_t& vb) {
        mv = 0;
        vb = 0u;
        if (t < nkt) {
          const int kt = a.kv_lo + t * KTILE, r = tid / NW;
          if (kt + dcol < hi) mv = p.kmeta[krow0 + kt + dcol];
          if (kt + r < hi) vb = p.vbad[(krow0 + kt + r) * NW + tid % NW];
        }
      };
      int mv_n;
      uint32_t vb_n;
      tile_meta(0, mv_n, vb_n);
      for (int t = 0; t < nkt; t++) {
        const int kt = a.kv_lo + t * KTILE, cp = t & 1;
        const uint32_t tt = tc + t, bsel = tt & 1;
        unsigned char* wbuf = Wp + bsel * L::w_buf;
        const int j = kt + dcol;
        const bool vj = j < hi;
        const int mv = mv_n;
        const uint32_t vb = vb_n;
        tile_meta(t + 1, mv_n, vb_n);   // the next tile's, in flight meanwhile
        const int Fk = kmeta_F(mv), kf = kmeta_fit(mv);
        if (tid == 0) { s_np[cp ^ 1] = 0; s_nbad[cp ^ 1] = 0; s_vany[cp ^ 1] = 0; }   // the next tile's counters
        {   // V elements outside the column window (key tid / NW, word tid % NW)
          uint32_t m = vb;
          vmask[tid] = m;
          if (m) s_vany[cp] = 1;
          while (m) {
            const int bit = __ffs(m) - 1, slot = atomicAdd(&s_nbad[cp], 1);
            m &= m - 1;
            if (slot < L::NBAD) badl[slot] = ((uint32_t)(tid / NW) << 16) | (uint32_t)((tid % NW) * 32 + bit);
          }
        }
        // ---- score diagonals of rows 4 rg .. 4 rg + 3 against this thread's key ----
        const bool ok = warp_wait(&sfull, tt & 1);
        float v[NDIAG][4];
        if (ok) {
#pragma unroll
          for (int c = 0; c < NDIAG; c++) tc5::ld_x4(lane_base + L::SC_COL + c * BM + rg * 4, v[c]);
          tc5::ld_wait();
#pragma unroll
          for (int c = 0; c < NDIAG; c++) tc5::st_zero_x4(lane_base + L::SC_COL + c * BM + rg * 4);
          tc5::st_wait();
        } else {
#pragma unroll
          for (int c = 0; c < NDIAG; c++)
#pragma unroll
            for (int e = 0; e < 4; e++) v[c][e] = 0.0f;
        }
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) tc5::mbar_arrive(&sempty);
        // ---- weights ----
        float w[4];
        uint32_t defer = 0;
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int rl = rg * 4 + e, i = q0 + rl;
          w[e] = 0.0f;
          if (ok && vj && i < a.Sq && (!a.causal || j <= i)) {
            if (qfit[rl] && kf) {
              w[e] = weight_of(__fmul_rn(a.scale32, cr32_scaled(combine_diag(v, e), Fq[rl] + Fk)), mrow[rl]);
            } else if (qlon[rl] != LO_DEEP && kmeta_lon(mv) != KLO_DEEP) {   // truncated dot + low limbs
              const float dot = dot_lo<DT>(combine_diag(v, e), qbase + (int64_t)i * a.qs[2], Fq[rl], qlo[rl], qlon[rl],
                                           kbase + (int64_t)j * a.ks[2], Fk, p.klo + (krow0 + j) * NLO, kmeta_lon(mv));
              w[e] = weight_of(__fmul_rn(a.scale32, dot), mrow[rl]);
            } else {
              defer |= 1u << e;   // a deep row: the general exact dot below fills this pair
            }
          }
        }
        // pairs with a deep row: each thread computes its own exactly
        if (defer) {
          const T* krow = kbase + (int64_t)j * a.ks[2];
#pragma unroll
          for (int e = 0; e < 4; e++)
            if ((defer >> e) & 1u) {
              const int rl = rg * 4 + e;
              const T* qrow = qbase + (int64_t)(q0 + rl) * a.qs[2];
              float dot;
              if (!qfit[rl] && kf)
                dot = exact_dot_lane<DT, true, false>(qrow, Fq[rl], krow, Fk, a.D);
              else if (qfit[rl])
                dot = exact_dot_lane<DT, false, true>(qrow, Fq[rl], krow, Fk, a.D);
              else
                dot = exact_dot_lane<DT, true, true>(qrow, Fq[rl], krow, Fk, a.D);
              w[e] = weight_of(__fmul_rn(a.scale32, dot), mrow[rl]);
            }
        }
        // ---- weight digits: W = w 2^79 = x 2^(8 b0), x < 2^32; words[e][q] = bytes 4q .. 4q + 3 of W ----
        uint32_t words[4][3];
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
            plist[atomicAdd(&s_np[cp], 1)] = (uint16_t)(dcol * BM + rg * 4 + e);   // w < 2^-56: exact atomics
          }
          const uint64_t y = (uint64_t)x << (8 * (b0 & 3));
          const uint32_t lo = (uint32_t)y, hw = (uint32_t)(y >> 32);
          const bool low = b0 < 4;
          words[e][0] = low ? lo : 0u;
          words[e][1] = low ? hw : lo;
          words[e][2] = low ? 0u : hw;
        }
        *reinterpret_cast<float4*>(Wf + dcol * BM + rg * 4) = make_float4(w[0], w[1], w[2], w[3]);
        {   // plane s of this key's 4 rows: 4 f16 values, contiguous in the MN-major block (one 8-byte store)
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
                const uint32_t h01 = f16_pair_from_biased(__byte_perm(a01[k >> 1], 0x64646464u, sel));
                const uint32_t h23 = f16_pair_from_biased(__byte_perm(a23[k >> 1], 0x64646464u, sel));
                *reinterpret_cast<uint2*>(wdst + s * L::w_blk) = make_uint2(h01, h23);
              }
            }
          }
        }
        tc5::fence_async_smem();   // the weight digit planes are read by the tensor cores
        __syncwarp();
        if (lane == 0) tc5::mbar_arrive(&wready[bsel]);
        // ---- the previous tile's PV products are done by now (or soon): fold them in ----
        if (t >= 1) drain(tt - 1);
        // ---- products outside the window: exact int64 atomics into the output digits ----
        tc5::bar_sync(1, NCT);   // lists, spill counters and the float weights complete
        if (s_np[cp] > 0 || s_vany[cp]) {
          if (!s_zeroed) {
            if (!a.add_into) {
              for (int64_t e = tid; e < (int64_t)nrows * NUM_NDIG * a.D; e += NCT)
                numb[(int64_t)q0 * NUM_NDIG * a.D + e] = 0;
              for (int e = tid; e < nrows * DEN_NDIG; e += NCT) denb[(int64_t)q0 * DEN_NDIG + e] = 0;
            }
            tc5::bar_sync(1, NCT);
            if (tid == 0) s_zeroed = 1;
          }
          const int np = s_np[cp];
          for (int e = warp; e < np; e += NCW) {
            const int cl = plist[e] / BM, rl = plist[e] % BM;
            const int i = q0 + rl, jj = kt + cl;
            const uint32_t wb = __float_as_uint(Wf[cl * BM + rl]);
            const Split sw = split_f32(wb);
            long long* nrow = numb + (int64_t)i * NUM_NDIG * a.D;
            for (int d = lane; d < a.D; d += 32) {
              uint32_t u = In<DT>::bits(vbase + (int64_t)jj * a.vs[2], d);
              if (nonfinite_bits(u)) continue;
              Split sv = split_f32(u);
              atomic_digits_add(nrow + d, a.D, NUM_E0, (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
            }
            if (lane == 0) atomic_digits_add(denb + (int64_t)i * DEN_NDIG, 1, DEN_E0, sw.mant, 0, sw.lsb);
          }
          const int nbad = s_nbad[cp];
          for (int it = tid; it < min(nbad, L::NBAD) * BM; it += NCT) {   // one (element, row) product each
            const int rl = it % BM;
            const uint32_t ent = badl[it / BM];
            const int cl = (int)(ent >> 16), d = (int)(ent & 0xFFFFu);
            const uint32_t wb = __float_as_uint(Wf[cl * BM + rl]);
            if (wb == 0u || (int)(wb >> 23) < 71) continue;   // zero, or already a pair spill
            const Split sv = split_f32(In<DT>::bits(vbase + (int64_t)(kt + cl) * a.vs[2], d));
            const Split sw = split_f32(wb);
            atomic_digits_add(numb + (int64_t)(q0 + rl) * NUM_NDIG * a.D + d, a.D, NUM_E0,
                              (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
          }
          if (nbad > L::NBAD) {   // list overflow: the elements past it, one thread per mask word
            for (int e = tid; e < KTILE * NW; e += NCT) {
              uint32_t m = vmask[e];
              const int cl = e / NW, tw = e % NW, jj = kt + cl;
              while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1;
                const int d = tw * 32 + bit;
                bool listed = false;
                for (int q = 0; q < L::NBAD && !listed; q++) listed = badl[q] == (((uint32_t)cl << 16) | (uint32_t)d);
                if (listed) continue;
                Split sv = split_f32(In<DT>::bits(vbase + (int64_t)jj * a.vs[2], d));
                for (int rl = 0; rl < BM; rl++) {
                  uint32_t wb = __float_as_uint(Wf[cl * BM + rl]);
                  if (wb == 0u || (int)(wb >> 23) < 71) continue;
                  Split sw = split_f32(wb);
                  atomic_digits_add(numb + (int64_t)(q0 + rl) * NUM_NDIG * a.D + d, a.D, NUM_E0,
                                    (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
                }
              }
            }
          }
        }
        if ((t & 1023) == 1023) {   // carry the lower digits up
#pragma unroll
          for (int r = 0; r < 4; r++) {
            long long c0 = acc[r][0] >> 32;
            acc[r][0] -= c0 * (1ll << 32);
            acc[r][1] += c0;
            long long c1 = acc[r][1] >> 32;
            acc[r][1] -= c1 * (1ll << 32);
            acc[r][2] += c1;
          }
        }
        tc5::bar_sync(1, NCT);   // tile consumed: float weights, lists and V masks are free
      }
      if (nkt > 0) drain(tc + nkt - 1);
      // ---- epilogue: canonical digits ----
      tc5::bar_sync(1, NCT);   // denT and every spill atomic complete
      const bool rmw = a.add_into || s_zeroed;
      const int d = dcol;
#pragma unroll
      for (int r = 0; r < 4; r++) {
        const int rl = rg * 4 + r, i = q0 + rl;
        if (i >= a.Sq || d >= a.D) continue;
        long long* nrow = numb + (int64_t)i * NUM_NDIG * a.D;
        long long dg[NUM_NDIG + 3];
#pragma unroll
        for (int k = 0; k < NUM_NDIG + 3; k++) dg[k] = 0;
        if (rmw)
#pragma unroll
          for (int k = 0; k < NUM_NDIG; k++) dg[k] = __ldcg(nrow + (int64_t)k * a.D + d);
        const int off = Fv[d] - 79 - NUM_E0;   // bit position of the accumulator's unit
        add_i64_at_tp(dg, acc[r][0], off);
        add_i64_at_tp(dg, acc[r][1], off + 32);
        add_i64_at_tp(dg, acc[r][2], off + 64);
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
      for (int rl = tid; rl < nrows; rl += NCT) {
        long long* drow = denb + (int64_t)(q0 + rl) * DEN_NDIG;
        long long dg[DEN_NDIG + 3];
#pragma unroll
        for (int k = 0; k < DEN_NDIG + 3; k++) dg[k] = 0;
        if (rmw)
#pragma unroll
          for (int k = 0; k < DEN_NDIG; k++) dg[k] = __ldcg(drow + k);
        const int off = -79 - DEN_E0;   // W units
        add_i64_at_tp(dg, denT[rl][0], off);
        add_i64_at_tp(dg, denT[rl][1], off + 32);
        add_i64_at_tp(dg, denT[rl][2], off + 64);
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
    }
    tc += nkt;
    __syncthreads();
  }   // pass
  if ((warp == L::SISS || warp == L::PISS) && lane == 0) {   // every MMA has completed before TMEM is released
    tc5::commit(&fin);
    tc5::mbar_wait(&fin, 0, &s_abort);
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  if (warp == 0) tc5::tmem_dealloc(tmem, L::TCOLS);
  if (s_abort) nf |= ST_TIMEOUT;
  report(a.status, nf | viol);
}

template <int DT>
static cudaError_t launch_acc_tp_t(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  using L = AccTpLayout;
  cudaError_t e = cudaFuncSetAttribute(accumulate_tp_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
  if (e != cudaSuccess) return e;
  const int nt = (a.Sq + L::BM - 1) / L::BM;
  dim3 grid(a.causal ? (nt + 1) / 2 : nt, a.Hq, a.B);
  accumulate_tp_kernel<DT><<<grid, L::THREADS, L::bytes, st>>>(a, p);
  return cudaGetLastError();
}

cudaError_t launch_accumulate_tp(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  return a.dtype == 0 ? launch_acc_tp_t<0>(a, p, st) : launch_acc_tp_t<1>(a, p, st);
}

}  // namespace detattn
