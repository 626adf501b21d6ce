// K2 on the tensor cores (sm_103a): exact accumulate of NUM / DEN digits, D <= 128.
//
// Page "det-attn", section "Method": NUM_id = sum_j exp(s_ij - rowmax_i) V_jd and
// DEN_i = sum_j exp(s_ij - rowmax_i) are exact integer sums in fixed bins.
//
// CTA = 32 query rows of one (b, h), key tiles of 128 keys, one CTA per SM.
//
// Scores.  The exact scores of a tile come from S^T = K Q^T on the tensor cores (tcgen05):
// per 16-dimension step, 16 MMAs of M = 128 keys x N = 32 rows x K = 16, key slice sa times
// query slice sb accumulated into the diagonal sum A_c, c = sa + sb (7 f32 accumulators of
// 32 columns; all partial sums are integers below 2^24, so exact).  Two accumulator sets
// (2 x 224 TMEM columns): the MMAs of tile t + 1 run while the CUDA cores work on tile t.
//
// Weights.  Warps 0-15 read the diagonal sums (warp w: keys 32 (w % 4) .. +31 as its lanes,
// query rows 8 (w / 4) .. +7), rebuild each exact int64 dot, round it once (cr32_scaled),
// scale it, and form w = exp32_det(RN32(s - m)).  W = w 2^92 goes to shared memory as three
// 31-bit limbs (exact for w >= 2^-69); DEN takes the limbs through warp reductions.
//
// PV.  The same 16 warps then add W * V exactly on the integer pipe: warp w owns query rows
// 2w, 2w + 1 and lane l the value columns CP l .. CP l + CP - 1; per (i, d) three int64
// accumulators hold limb * Vint (V as fixed point per column, |Vint| < 2^23); limbs 1 and 2
// carry the weights w >= 2^-38 and limbs 0 and 1 those below 2^-30, so each warp runs its two
// rows through the two limbs the tile needs (all three only when both kinds occur).  Every
// 256 keys the limbs carry into a fourth word in shared memory.  Products outside the window (w < 2^-69, or a V element below
// its column window) are added with exact int64 atomics into the output digits, one
// (element, row) product per thread.
//
// Roles: warp 16 lane 0 copies key operand tiles (bulk copies, 2-stage ring), warp 17 lane 0
// issues the MMAs, warp 18 lane 0 copies 16-key chunks of the prepared V rows (2-stage
// ring).  Every mbarrier wait is bounded; one that gives up sets DA_STATUS_TIMEOUT.  In the
// compute warps a failed wait only skips work, so all of them still pass every named
// barrier, and the CTA winds down, freeing its TMEM.
#include "numerics.cuh"
#include "score_tc.cuh"
#include "tc5.cuh"
#include "attn_kernels.h"

namespace detattn {

template <int DP>
struct AccTcLayout {
  static constexpr int BM = 32, NDS = DP / 16, NST = 2, VCH = 16, NVB = 2, NCW = 16;
  static constexpr int KLOAD = NCW, ISSUER = NCW + 1, VLOAD = NCW + 2, THREADS = 32 * (NCW + 3);
  static constexpr int RP = 2, CP = DP / 32, NW = DP / 32, LDW = KTILE + 4, NCH = KTILE / VCH;
  static constexpr int TCOLS = 512, BUF = 256;
  static constexpr size_t q_bytes = (size_t)NDS * NSLICE * BM * 32;   // B blocks [step][slice], BM x 16 bf16
  static constexpr size_t k_off = q_bytes;                              // NST key operand stages
  static constexpr size_t v_off = k_off + (size_t)NST * KT_BLOCK;       // NVB V chunks
  static constexpr size_t v_chunk = (size_t)VCH * DP * 4;               //   int32 [VCH][DP]
  static constexpr size_t w_off = v_off + NVB * v_chunk;                // int32 [3][BM][LDW] weight limbs
  static constexpr size_t wf_off = w_off + (size_t)3 * BM * LDW * 4;    // float [BM][KTILE] weights
  static constexpr size_t p3_off = wf_off + (size_t)KTILE * BM * 4;     // int64 [BM][DP] carried limbs
  static constexpr size_t ps_off = p3_off + (size_t)BM * DP * 8;        // uint16 pairs below 2^-69
  static constexpr int NBAD = 1024;                                     // listed V elements outside the window
  static constexpr size_t bytes = ps_off + (size_t)KTILE * BM * 2;
  static_assert(NDIAG * BM <= BUF && 2 * BUF <= TCOLS, "TMEM columns");
  static_assert(bytes <= 220 * 1024, "shared memory budget");
  static_assert(RP * NCW == BM && CP * 32 == DP, "PV thread mapping");
};

// add a signed 64-bit X * 2^o into lazily carried radix-2^32 digits dg[]
__device__ __forceinline__ void add_i64_at(long long* dg, long long X, int o) {
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

// warp sum of a 31-bit limb per lane, exact (two 16-bit halves through redux)
__device__ __forceinline__ long long warp_sum31(int x) {
  const unsigned lo = __reduce_add_sync(0xFFFFFFFFu, (unsigned)x & 0xFFFFu);
  const unsigned hi = __reduce_add_sync(0xFFFFFFFFu, (unsigned)x >> 16);
  return (long long)lo + ((long long)hi << 16);
}

// PV of one V chunk through limbs L0 .. L0 + NLB - 1: acc[r][c][l] += W_l(row, key) * Vint(key, col).
// Limb planes are [limb][row][key] (row stride LDW); two keys per step, one 64-bit load per
// (limb, row).
template <int L0, int NLB, int RP, int CP, int DP, int LDW, int VCH>
__device__ __forceinline__ void pv_chunk(long long (&acc)[RP][CP][3], const int* Wl, const int* vsl, int key0, int pr,
                                         int pc) {
#pragma unroll 1
  for (int jj = 0; jj < VCH; jj += 2) {
    int wv[NLB][RP][2], vv[2][CP];
#pragma unroll
    for (int l = 0; l < NLB; l++)
#pragma unroll
      for (int r = 0; r < RP; r++) {
        const int2 t2 = *reinterpret_cast<const int2*>(Wl + ((L0 + l) * (RP * 16) + pr * RP + r) * LDW + key0 + jj);
        wv[l][r][0] = t2.x;
        wv[l][r][1] = t2.y;
      }
#pragma unroll
    for (int k2 = 0; k2 < 2; k2++) {
      const int* vp = vsl + (jj + k2) * DP + pc * CP;
      if constexpr (CP == 2) {
        const int2 t2 = *reinterpret_cast<const int2*>(vp);
        vv[k2][0] = t2.x;
        vv[k2][1] = t2.y;
      } else {
#pragma unroll
        for (int c4 = 0; c4 < CP; c4 += 4) {
          const int4 t4 = *reinterpret_cast<const int4*>(vp + c4);
          vv[k2][c4] = t4.x;
          vv[k2][c4 + 1] = t4.y;
          vv[k2][c4 + 2] = t4.z;
          vv[k2][c4 + 3] = t4.w;
        }
      }
    }
#pragma unroll
    for (int k2 = 0; k2 < 2; k2++)
#pragma unroll
      for (int r = 0; r < RP; r++)
#pragma unroll
        for (int c = 0; c < CP; c++)
#pragma unroll
          for (int l = 0; l < NLB; l++) mad_wide(acc[r][c][L0 + l], wv[l][r][k2], vv[k2][c]);
  }
}

template <int DT, int DP>
__global__ void __launch_bounds__(AccTcLayout<DP>::THREADS, 1) accumulate_tc_kernel(const AttnArgs a, const KvPrep p) {
  using T = typename In<DT>::T;
  using L = AccTcLayout<DP>;
  constexpr int BM = L::BM, NDS = L::NDS, NST = L::NST, NVB = L::NVB, NCW = L::NCW, VCH = L::VCH, NCH = L::NCH;
  constexpr int RP = L::RP, CP = L::CP, NW = L::NW, LDW = L::LDW;
  constexpr int NCT = 32 * NCW;   // compute threads
  constexpr uint32_t IDESC = tc5::idesc_bf16(KTILE, BM);
  extern __shared__ __align__(1024) unsigned char smem_a[];
  unsigned char* Qs = smem_a;
  unsigned char* Kst = smem_a + L::k_off;
  int* Vs = reinterpret_cast<int*>(smem_a + L::v_off);
  int* Wl = reinterpret_cast<int*>(smem_a + L::w_off);
  float* Wf = reinterpret_cast<float*>(smem_a + L::wf_off);
  long long* P3 = reinterpret_cast<long long*>(smem_a + L::p3_off);
  uint16_t* plist = reinterpret_cast<uint16_t*>(smem_a + L::ps_off);
  __shared__ __align__(8) uint64_t kfull[NST], kempty[NST], tfull[2], tempty[2], vfull[NVB], vempty[NVB], fin;
  __shared__ uint32_t tmem_s;
  __shared__ int Fq[BM], Fv[DP];
  __shared__ unsigned char qfit[BM];
  __shared__ float mrow[BM];
  __shared__ long long denT[BM][3];
  __shared__ uint32_t vmask[KTILE * NW];
  __shared__ int s_np, s_nbad, s_vany, s_zeroed;
  __shared__ int rlimb[BM];   // per row of this tile: bit 0 some weight has a nonzero limb 0, bit 1 limb 2
  __shared__ uint32_t badl[L::NBAD];   // (key << 16) | column of V elements outside the window
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y, b = blockIdx.z, hk = h / (a.Hq / a.Hkv);
  const T* qbase = (const T*)a.q + b * a.qs[0] + h * a.qs[1];
  const T* kbase = (const T*)a.k + b * a.ks[0] + hk * a.ks[1];
  const T* vbase = (const T*)a.v + b * a.vs[0] + hk * a.vs[1];
  const int64_t krow0 = ((int64_t)b * a.Hkv + hk) * a.Skv;
  const unsigned char* ktc = p.ktc + (int64_t)(b * a.Hkv + hk) * p.ntk * NDS * KT_BLOCK;
  const int64_t rowbase = ((int64_t)b * a.Hq + h) * a.Sq;
  long long* numb = a.num + rowbase * NUM_NDIG * a.D;
  long long* denb = a.den + rowbase * DEN_NDIG;

  if (warp == 0) tc5::tmem_alloc(&tmem_s, L::TCOLS);
  if (tid == 0) {
    for (int s = 0; s < NST; s++) {
      tc5::mbar_init(&kfull[s], 1);
      tc5::mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < 2; s++) {
      tc5::mbar_init(&tfull[s], 1);
      tc5::mbar_init(&tempty[s], NCW);
    }
    for (int s = 0; s < NVB; s++) {
      tc5::mbar_init(&vfull[s], 1);
      tc5::mbar_init(&vempty[s], NCW);
    }
    tc5::mbar_init(&fin, 1);
    s_abort = 0;
    tc5::mbar_fence_init();
  }
  for (int d = tid; d < DP; d += L::THREADS)   // biased exponent in [1, 254]: |Vint| < 2^23, digit offsets in range
    Fv[d] = min(max(p.vcol[((int64_t)b * a.Hkv + hk) * DP + d], 1), 254) - 149;
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  const uint32_t tmem = tmem_s;

  int nf = 0, viol = 0;
  uint32_t g_base = 0, tc = 0;   // key-operand ring steps of earlier passes; key tiles seen by this role
  const int ntq = (a.Sq + BM - 1) / BM;
  const int npass = (a.causal && (int)blockIdx.x != ntq - 1 - (int)blockIdx.x) ? 2 : 1;
  for (int pass = 0; pass < npass; pass++) {
    const int q0 = (pass == 0 ? ntq - 1 - (int)blockIdx.x : (int)blockIdx.x) * BM;
    const int hi = a.causal ? min(a.kv_hi, q0 + BM) : a.kv_hi;
    const int nkt = hi > a.kv_lo ? (hi - a.kv_lo + KTILE - 1) / KTILE : 0;
    const uint32_t nsteps = (uint32_t)nkt * NDS;
    const int nrows = min(BM, a.Sq - q0);
    // ---- per pass: query slices (resident B operand), row maxima, cleared sums ----
    for (int r = warp; r < BM; r += L::THREADS / 32) {
      const int i = q0 + r;
      row_slices<DT, DP>(
          i < a.Sq ? qbase + (int64_t)i * a.qs[2] : nullptr, a.D,
          [&](int q, int d, uint16_t v) {
            *reinterpret_cast<uint16_t*>(Qs + ((d >> 4) * NSLICE + q) * (BM * 32) + tc5::canon_off(r, d & 15)) = v;
          },
          &Fq[r], &qfit[r], nf, lane);
    }
    for (int r = tid; r < BM; r += L::THREADS) mrow[r] = (q0 + r < a.Sq) ? a.m_in[rowbase + q0 + r] : 0.0f;
    for (int e = tid; e < BM * DP; e += L::THREADS) P3[e] = 0;
    for (int e = tid; e < BM * 3; e += L::THREADS) (&denT[0][0])[e] = 0;
    if (tid == 0) s_zeroed = 0;
    tc5::fence_async_smem();
    __syncthreads();

    if (warp == L::KLOAD) {   // ---------------- key operand tiles ----------------
      if (lane == 0)
        for (uint32_t ls = 0; ls < nsteps && !s_abort; ls++) {
          const uint32_t g = g_base + ls, st = g % NST;
          if (g >= NST && !tc5::mbar_wait(&kempty[st], ((g / NST) - 1) & 1, &s_abort, 64)) break;
          tc5::mbar_expect_tx(&kfull[st], KT_BLOCK);
          tc5::bulk_g2s(Kst + st * KT_BLOCK, ktc + (size_t)ls * KT_BLOCK, KT_BLOCK, &kfull[st]);
        }
    } else if (warp == L::ISSUER) {   // ---------------- MMAs ----------------
      if (lane == 0)
        for (uint32_t ls = 0; ls < nsteps && !s_abort; ls++) {
          const uint32_t g = g_base + ls, st = g % NST, bsel = tc & 1;
          const int k = (int)(ls % NDS);
          if (!tc5::mbar_wait(&kfull[st], (g / NST) & 1, &s_abort, 32)) break;
          if (k == 0 && tc >= 2 && !tc5::mbar_wait(&tempty[bsel], ((tc >> 1) - 1) & 1, &s_abort, 64)) break;
          tc5::fence_after();
          const uint64_t ka = tc5::desc(tc5::smem_addr(Kst + st * KT_BLOCK));
          const uint64_t qa = tc5::desc(tc5::smem_addr(Qs + k * NSLICE * BM * 32));
          const uint32_t dbase = tmem + bsel * L::BUF;
#pragma unroll
          for (int sa = 0; sa < NSLICE; sa++)
#pragma unroll
            for (int sb = 0; sb < NSLICE; sb++) {
              const int c = sa + sb;
              const uint32_t accum = (k > 0 || sa != (c > 3 ? c - 3 : 0)) ? 1u : 0u;
              // descriptor start addresses advance in 16-byte units
              tc5::mma_bf16(dbase + c * BM, ka + (uint64_t)(sa * KTILE * 2), qa + (uint64_t)(sb * BM * 2), IDESC,
                            accum);
            }
          tc5::commit(&kempty[st]);
          if (k == NDS - 1) {
            tc5::commit(&tfull[bsel]);
            tc++;
          }
        }
    } else if (warp == L::VLOAD) {   // ---------------- V chunks ----------------
      if (lane == 0)
        for (int t = 0; t < nkt && !s_abort; t++)
          for (int ch = 0; ch < NCH && !s_abort; ch++) {
            const uint32_t g = (tc + t) * NCH + ch, sl = g % NVB;
            if (g >= NVB && !tc5::mbar_wait(&vempty[sl], ((g / NVB) - 1) & 1, &s_abort, 64)) break;
            const int j0 = a.kv_lo + t * KTILE + ch * VCH, rows = min(VCH, hi - j0);
            if (rows > 0) {
              tc5::mbar_expect_tx(&vfull[sl], (uint32_t)(rows * DP * 4));
              tc5::bulk_g2s(Vs + sl * (VCH * DP), p.vint + (krow0 + j0) * DP, (uint32_t)(rows * DP * 4), &vfull[sl]);
            } else {
              tc5::mbar_arrive(&vfull[sl]);
            }
          }
    } else {   // ---------------- compute warps: weights, PV, spills ----------------
      const int quarter = warp & 3, rg = warp >> 2, jl = 32 * quarter + lane;
      const int pr = warp, pc = lane;   // PV: rows pr * RP + r, columns pc * CP + c
      long long acc[RP][CP][3];
#pragma unroll
      for (int r = 0; r < RP; r++)
#pragma unroll
        for (int c = 0; c < CP; c++)
#pragma unroll
          for (int l = 0; l < 3; l++) acc[r][c][l] = 0;
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
      // weight of one pair -> limb planes, float plane, lists; returns its limbs
      auto store_weight = [&](float w, int rl, int cl, int (&lb)[3]) {
        const uint32_t wb = __float_as_uint(w);
        const int ex = (int)(wb >> 23);
        int l0 = 0, l1 = 0, l2 = 0;
        if (wb != 0u) {
          if (ex >= 58) {   // W = mant << (ex - 58) < 2^93, split into 31-bit limbs with 64-bit shifts
            const uint64_t mant = (wb & 0x7FFFFFu) | 0x800000u;
            const int sh = ex - 58;
            if (sh <= 38) {
              const uint64_t W = mant << sh;   // < 2^62
              l0 = (int)(W & 0x7FFFFFFFull);
              l1 = (int)(W >> 31);
            } else {
              const uint64_t W1 = mant << (sh - 31);   // W >> 31, exact: the low 31 bits of W are zero
              l1 = (int)(W1 & 0x7FFFFFFFull);
              l2 = (int)(W1 >> 31);
            }
          } else {
            plist[atomicAdd(&s_np, 1)] = (uint16_t)(cl * BM + rl);             // w < 2^-69: exact atomics
          }
        }
        Wl[(0 * BM + rl) * LDW + cl] = l0;
        Wl[(1 * BM + rl) * LDW + cl] = l1;
        Wl[(2 * BM + rl) * LDW + cl] = l2;
        Wf[rl * KTILE + cl] = w;
        lb[0] = l0;
        lb[1] = l1;
        lb[2] = l2;
      };
      auto weight_of = [&](float sc, float m) -> float {
        float x = __fsub_rn(sc, m);
        if (x != x) { nf |= ST_NONFINITE; x = neg_inf(); }
        if (x > 0.0f) { viol |= ST_VIOLATION; x = 0.0f; }
        return exp32_det(x);
      };
      int tiles_since_carry = 0;
      for (int t = 0; t < nkt; t++) {
        const int kt = a.kv_lo + t * KTILE;
        const int j = kt + jl;
        const bool vj = j < hi;
        const int mv = vj ? p.kmeta[krow0 + j] : 0;
        if (tid < BM) rlimb[tid] = 0;
        if (tid == 0) { s_np = 0; s_nbad = 0; s_vany = 0; }
        tc5::bar_sync(1, NCT);
        for (int e = tid; e < KTILE * NW; e += NCT) {   // V elements outside the column window
          const int r = e / NW;
          uint32_t m = (kt + r < hi) ? p.vbad[(krow0 + kt + r) * NW + e % NW] : 0u;
          vmask[e] = m;
          if (m) s_vany = 1;
          while (m) {
            const int bit = __ffs(m) - 1, slot = atomicAdd(&s_nbad, 1);
            m &= m - 1;
            if (slot < L::NBAD) badl[slot] = ((uint32_t)r << 16) | (uint32_t)((e % NW) * 32 + bit);
          }
        }
        // ---- weights from the exact scores in TMEM ----
        const uint32_t bsel = tc & 1;
        // a failed wait only skips work: every compute warp still passes every barrier below
        const bool live = __all_sync(0xFFFFFFFFu, tc5::mbar_wait(&tfull[bsel], (tc >> 1) & 1, &s_abort, 64));
        tc5::fence_after();
        const int Fk = kmeta_F(mv), kf = kmeta_fit(mv);
        const uint32_t tbase = tmem + ((uint32_t)(32 * quarter) << 16) + bsel * L::BUF + rg * 8;
        uint32_t defer = 0;
#pragma unroll
        for (int rr = 0; rr < 8; rr += 2) {
          float v[NDIAG][2];
          if (live) {
#pragma unroll
            for (int c = 0; c < NDIAG; c++) tc5::ld_x2(tbase + c * BM + rr, v[c][0], v[c][1]);
            tc5::ld_wait();
          } else {
#pragma unroll
            for (int c = 0; c < NDIAG; c++) v[c][0] = v[c][1] = 0.0f;
          }
#pragma unroll
          for (int e = 0; e < 2; e++) {
            const int rl = rg * 8 + rr + e, i = q0 + rl;
            float w = 0.0f;
            if (live && vj && i < a.Sq && (!a.causal || j <= i)) {
              if (qfit[rl] && kf) {
                long long Tsum = 0;
#pragma unroll
                for (int c = NDIAG - 1; c >= 0; c--) Tsum = Tsum * 128 + small_f2i(v[c][e]);
                const float sc = __fmul_rn(a.scale32, cr32_scaled(Tsum, Fq[rl] + Fk));
                w = weight_of(sc, mrow[rl]);
              } else {
                defer |= 1u << (rr + e);   // the exact fallback below fills this pair
              }
            }
            int lb[3];
            store_weight(w, rl, jl, lb);
#pragma unroll
            for (int l = 0; l < 3; l++) {
              const long long s = warp_sum31(lb[l]);
              if (lane == 0 && s) atomicAdd((unsigned long long*)&denT[rl][l], (unsigned long long)s);
            }
            const int fl = (__any_sync(0xFFFFFFFFu, lb[0] != 0) ? 1 : 0) | (__any_sync(0xFFFFFFFFu, lb[2] != 0) ? 2 : 0);
            if (lane == 0 && fl) atomicOr(&rlimb[rl], fl);
          }
        }
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) tc5::mbar_arrive(&tempty[bsel]);
        tc++;
        // pairs outside the fixed-point window: the whole warp computes each exact dot
        for (uint32_t pend = __ballot_sync(0xFFFFFFFFu, defer != 0); pend;
             pend = __ballot_sync(0xFFFFFFFFu, defer != 0)) {
          const int src = __ffs(pend) - 1;
          const uint32_t dm = __shfl_sync(0xFFFFFFFFu, defer, src);
          const int rl = rg * 8 + __ffs(dm) - 1, cl = 32 * quarter + src;
          const float sc = __fmul_rn(a.scale32, exact_dot_warp<DT>(qbase + (int64_t)(q0 + rl) * a.qs[2],
                                                                  kbase + (int64_t)(kt + cl) * a.ks[2], a.D, lane));
          if (lane == 0) {
            int lb[3];
            store_weight(weight_of(sc, mrow[rl]), rl, cl, lb);
#pragma unroll
            for (int l = 0; l < 3; l++)
              if (lb[l]) atomicAdd((unsigned long long*)&denT[rl][l], (unsigned long long)lb[l]);
            atomicOr(&rlimb[rl], (lb[0] != 0 ? 1 : 0) | (lb[2] != 0 ? 2 : 0));
          }
          if (lane == src) defer &= defer - 1;
        }
        tc5::bar_sync(1, NCT);   // weight planes complete
        // ---- exact PV on the integer pipe: the two limbs this warp's rows need (three if both kinds) ----
        const int need = rlimb[pr * RP] | rlimb[pr * RP + 1];   // warp-uniform
        for (int ch = 0; ch < NCH; ch++) {
          const uint32_t g = (tc - 1) * NCH + ch, sl = g % NVB;
          const bool vok = __all_sync(0xFFFFFFFFu, tc5::mbar_wait(&vfull[sl], (g / NVB) & 1, &s_abort, 32));
          if (vok && kt + ch * VCH < hi) {
            const int* vsl = Vs + sl * (VCH * DP);
            if (need == 3)
              pv_chunk<0, 3, RP, CP, DP, LDW, VCH>(acc, Wl, vsl, ch * VCH, pr, pc);
            else if (need == 1)
              pv_chunk<0, 2, RP, CP, DP, LDW, VCH>(acc, Wl, vsl, ch * VCH, pr, pc);
            else
              pv_chunk<1, 2, RP, CP, DP, LDW, VCH>(acc, Wl, vsl, ch * VCH, pr, pc);
          }
          __syncwarp();
          if (lane == 0) tc5::mbar_arrive(&vempty[sl]);
        }
        if (++tiles_since_carry == 256 / KTILE) {   // 256 keys: limb sums stay below 2^62
          carry_into_p3();
          tiles_since_carry = 0;
        }
        // ---- products outside the window: exact int64 atomics into the output digits ----
        if (s_np > 0 || s_vany) {
          if (!s_zeroed) {
            if (!a.add_into) {
              for (int64_t e = tid; e < (int64_t)nrows * NUM_NDIG * a.D; e += NCT)
                numb[(int64_t)q0 * NUM_NDIG * a.D + e] = 0;
              for (int e = tid; e < nrows * DEN_NDIG; e += NCT) denb[(int64_t)q0 * DEN_NDIG + e] = 0;
            }
            tc5::bar_sync(1, NCT);
            if (tid == 0) s_zeroed = 1;
          }
          const int np = s_np;
          for (int e = warp; e < np; e += NCW) {
            const int cl = plist[e] / BM, rl = plist[e] % BM;
            const int i = q0 + rl, jj = kt + cl;
            Split sw = split_f32(__float_as_uint(Wf[rl * KTILE + cl]));
            long long* nrow = numb + (int64_t)i * NUM_NDIG * a.D;
            for (int d = lane; d < a.D; d += 32) {
              uint32_t u = In<DT>::bits(vbase + (int64_t)jj * a.vs[2], d);
              if (nonfinite_bits(u)) continue;
              Split sv = split_f32(u);
              atomic_digits_add(nrow + d, a.D, NUM_E0, (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
            }
            if (lane == 0) atomic_digits_add(denb + (int64_t)i * DEN_NDIG, 1, DEN_E0, sw.mant, 0, sw.lsb);
          }
          const int nbad = s_nbad;
          for (int it = tid; it < min(nbad, L::NBAD) * BM; it += NCT) {   // one (element, row) product each
            const int rl = it % BM;
            const uint32_t ent = badl[it / BM];
            const int cl = (int)(ent >> 16), d = (int)(ent & 0xFFFFu);
            const uint32_t wb = __float_as_uint(Wf[rl * KTILE + cl]);
            if (wb == 0u || (int)(wb >> 23) < 58) continue;   // zero, or already a pair spill
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
                Split sv = split_f32(In<DT>::bits(vbase + (int64_t)jj * a.vs[2], d));
                bool listed = false;   // the first NBAD listed elements are done above
                for (int q = 0; q < L::NBAD && !listed; q++) listed = badl[q] == (((uint32_t)cl << 16) | (uint32_t)d);
                if (listed) continue;
                for (int rl = 0; rl < BM; rl++) {
                  uint32_t wb = __float_as_uint(Wf[rl * KTILE + cl]);
                  if (wb == 0u || (int)(wb >> 23) < 58) continue;   // zero, or already a pair spill
                  Split sw = split_f32(wb);
                  atomic_digits_add(numb + (int64_t)(q0 + rl) * NUM_NDIG * a.D + d, a.D, NUM_E0,
                                    (unsigned long long)sw.mant * sv.mant, sv.neg, sw.lsb + sv.lsb);
                }
              }
            }
          }
        }
        tc5::bar_sync(1, NCT);   // tile consumed: weight planes and lists are free
      }
      // ---- epilogue: canonical digits ----
      carry_into_p3();
      tc5::bar_sync(1, NCT);   // P3, denT and every spill atomic complete
      const bool rmw = a.add_into || s_zeroed;
#pragma unroll
      for (int r = 0; r < RP; r++) {
        const int rl = pr * RP + r, i = q0 + rl;
        if (i >= a.Sq) continue;
        long long* nrow = numb + (int64_t)i * NUM_NDIG * a.D;
#pragma unroll
        for (int c = 0; c < CP; c++) {
          const int d = pc * CP + c;
          if (d >= a.D) continue;
          long long dg[NUM_NDIG + 3];
#pragma unroll
          for (int k = 0; k < NUM_NDIG + 3; k++) dg[k] = 0;
          if (rmw)
#pragma unroll
            for (int k = 0; k < NUM_NDIG; k++) dg[k] = __ldcg(nrow + (int64_t)k * a.D + d);
          const int off = Fv[d] - 92 - NUM_E0;   // bit position of the accumulator's unit
          add_i64_at(dg, acc[r][c][0], off);
          add_i64_at(dg, acc[r][c][1], off + 31);
          add_i64_at(dg, acc[r][c][2], off + 62);
          add_i64_at(dg, P3[rl * DP + d], off + 93);
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
      }
      for (int rl = tid; rl < nrows; rl += NCT) {
        long long* drow = denb + (int64_t)(q0 + rl) * DEN_NDIG;
        long long dg[DEN_NDIG + 3];
#pragma unroll
        for (int k = 0; k < DEN_NDIG + 3; k++) dg[k] = 0;
        if (rmw)
#pragma unroll
          for (int k = 0; k < DEN_NDIG; k++) dg[k] = __ldcg(drow + k);
        const int off = -92 - DEN_E0;
        add_i64_at(dg, denT[rl][0], off);
        add_i64_at(dg, denT[rl][1], off + 31);
        add_i64_at(dg, denT[rl][2], off + 62);
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
    g_base += nsteps;
    if (warp == L::VLOAD) tc += nkt;   // the V loader counts tiles without consuming them
    __syncthreads();
  }   // pass
  if (tid == 32 * L::ISSUER) {   // every MMA issued has completed before TMEM is released
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

template <int DT, int DP>
static cudaError_t launch_acc_tc_t(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  using L = AccTcLayout<DP>;
  cudaError_t e =
      cudaFuncSetAttribute(accumulate_tc_kernel<DT, DP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
  if (e != cudaSuccess) return e;
  const int nt = (a.Sq + L::BM - 1) / L::BM;
  dim3 grid(a.causal ? (nt + 1) / 2 : nt, a.Hq, a.B);
  accumulate_tc_kernel<DT, DP><<<grid, L::THREADS, L::bytes, st>>>(a, p);
  return cudaGetLastError();
}

cudaError_t launch_accumulate_tc(const AttnArgs& a, const KvPrep& p, cudaStream_t st) {
  if (a.dtype == 0) return p.DP == 64 ? launch_acc_tc_t<0, 64>(a, p, st) : launch_acc_tc_t<0, 128>(a, p, st);
  return p.DP == 64 ? launch_acc_tc_t<1, 64>(a, p, st) : launch_acc_tc_t<1, 128>(a, p, st);
}

}  // namespace detattn
