// Internal kernel interface of libdetattn (not part of the C ABI).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace detattn {

struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  int64_t qs[4], ks[4], vs[4];   // element strides of [B, H, S, D]; qs[3] == ks[3] == vs[3] == 1
  int dtype;                     // 0 = f32, 1 = bf16
  int B, Hq, Hkv, Sq, Skv, D;
  int causal;
  float scale32;
  int kv_lo, kv_hi;
  float* m_out;                  // rowmax output [B, Hq, Sq]
  const float* m_in;             // global rowmax input [B, Hq, Sq]
  long long* num;                // [B, Hq, Sq, 15, D]
  long long* den;                // [B, Hq, Sq, 6]
  int add_into;
  int canon_in;                  // with add_into: the digits already there are canonical, so a row with
                                 // no key in [kv_lo, kv_hi) may be left as it is (no read-modify-write)
  int* status;                   // device status word (may be null)
  float* out;                    // non-null: the tensor-PV accumulate finalizes into out [B, Hq, Sq, D]
                                 // instead of writing digits (one key range, add_into == 0)
  float* scores;                 // non-null: the score cache (below); rowmax writes it, the tensor-PV
                                 // accumulate reads it instead of recomputing the scores
  int64_t sc_per_bh;             // score-cache blocks per (b, query head)
  int sc_nkt;                    // non-causal: key tiles per query tile
  const int* order;              // tensor-PV accumulate: its work items in this order (null: launch order);
                                 // an entry is a pair index, with bit 30 for its long tile alone or bit
                                 // 29 for its short tile alone, or -1 for an unused slot
  int order_extra;               // CTAs the order holds beyond one per pair (split pairs, unused slots)
};

// Score cache of one whole-range call (kv_lo = 0, kv_hi = Skv; causal needs Sq = Skv): the
// exact score s_ij of every (query, key) pair of every processed tile, f32, in blocks of
// SC_ROWS query rows x KTILE keys laid out [key][row], one block per (b, h, query tile of
// SC_ROWS rows, key tile).  Causal: query tile q has ceil(min(Sq, SC_ROWS (q + 1)) / KTILE)
// key tiles, so the tiles of query tiles below q (all full) number
// q + 8 g (g - 1) / 2 + (q % 8) g with g = q / 8; non-causal: sc_nkt per query tile.
constexpr int SC_ROWS = 16;
__host__ __device__ inline int64_t sc_block(const AttnArgs& a, int bh, int qt, int kt) {
  const int64_t g = qt >> 3, r = qt & 7;
  const int64_t before = a.causal ? qt + 4 * g * (g - 1) + r * g : (int64_t)qt * a.sc_nkt;
  return (int64_t)bh * a.sc_per_bh + before + kt;
}
constexpr int SC_BLOCK = SC_ROWS * 128;   // floats per block (KTILE keys)
size_t score_cache_bytes(int B, int Hq, int Sq, int Skv, int causal, int* sc_nkt, int64_t* sc_per_bh);

// Prepared keys/values of one call's key range (prep_kernels.cu), rows indexed as
// (b * Hkv + hk) * Skv + j.
struct KvPrep {
  uint16_t* ksl;     // bf16 digit slices [rows][4][DP] (DP == 256 only)
  unsigned char* ktc;   // the same slices as tensor-core operand tiles (below)
  int ntk;           // key tiles of KTILE rows per (b, hk) in ktc
  int* kmeta;        // [rows]: (F + 1024) | (fit << 16) | (low-limb count, or 15 for deep, << 17)
  int2* klo;         // [rows][NLO] low limbs (d, X_lo) of rows outside the 26-bit window
  long long* spill;  // DP == 128 with V: SPILL_SLOTS per-SM scratch slots (below), zero between uses
  unsigned char* vtc;   // DP == 128: V as tensor-core operand digit planes (below), else null
  int* vcol;         // [B * Hkv][DP] largest V biased exponent per column over the range
  int* vint;         // [rows][DP] V fixed point, |Vint| < 2^23
  uint32_t* vbad;    // [rows][DP / 32] elements outside the V window
  int DP;
  int do_v;
};
// ktc: per (b, hk), key tiles of KTILE keys starting at the call's kv_lo; per tile, per
// 16-wide step of d, one 16 KiB block = 4 slices x (KTILE x 16 bf16 in the canonical
// K-major operand layout of tc5.cuh).  Rows past kv_hi are zero.
constexpr int KTILE = 128;
constexpr int KT_BLOCK = 4 * KTILE * 16 * 2;
// vtc (DP == 128): per (b, hk), blocks of 16 keys from kv_lo (padded to whole key tiles);
// per block 3 planes = the balanced base-256 digits of Vint (each exact in f16), each a
// 128 (d) x 16 (keys) operand block in the canonical K-major layout of tc5.cuh.
constexpr int VKEYS = 16;
// spill: one slot per SM (one tensor-PV CTA fits on an SM at a time), indexed by %smid: the
// products outside the fixed-point windows of the CTA's 16 rows, [16][15][DP] NUM digits then
// [16][6] DEN digits; the CTA's epilogue reads what it touched and clears it again
constexpr int SPILL_SLOTS = 256, SPILL_ROWS = 16;
__host__ __device__ constexpr size_t spill_slot_words(int dp) { return (size_t)SPILL_ROWS * (15 * dp + 6); }
constexpr int VP_BLOCK = 3 * 128 * VKEYS * 2;
size_t kv_prep_bytes(int B, int Hkv, int Skv, int D);
KvPrep kv_prep_layout(void* ws, int B, int Hkv, int Skv, int D, int do_v);
cudaError_t launch_kv_prep(const AttnArgs& a, const KvPrep& p, cudaStream_t st);

cudaError_t launch_rowmax(const AttnArgs& a, const KvPrep& p, cudaStream_t st);   // a.scores: also store scores
cudaError_t launch_accumulate(const AttnArgs& a, const KvPrep& p, cudaStream_t st);
cudaError_t launch_accumulate_tc(const AttnArgs& a, const KvPrep& p, cudaStream_t st);   // D <= 128
cudaError_t launch_accumulate_tp(const AttnArgs& a, const KvPrep& p, cudaStream_t st);   // D <= 128
// the tensor-PV accumulate's work items, heaviest first, into ws (tp_order_bytes): a.order set
size_t tp_order_bytes(const AttnArgs& a);
cudaError_t launch_tp_order(AttnArgs& a, void* ws, cudaStream_t st);
constexpr int ACC_TP_MAX_TILES = 512;   // key tiles per pass the tensor-PV kernel's state holds exactly
bool accumulate_is_tp(const AttnArgs& a, const KvPrep& p);   // launch_accumulate takes the tensor-PV kernel

cudaError_t launch_compose_max(float* dst, const float* src, int64_t n, cudaStream_t st);
cudaError_t launch_compose_add(long long* dst, const long long* src, int64_t n, cudaStream_t st);
cudaError_t launch_normalize(long long* dg, int64_t nrows, int ndig, int64_t inner, int* status, cudaStream_t st);
cudaError_t launch_finalize(const long long* num, const long long* den, int64_t rows, int D, float* out, int* status,
                            cudaStream_t st);

struct DceArgs {
  const void* x;
  int dtype;
  int64_t N, V, rs;     // rows, columns, row stride (elements)
  int64_t v_lo, v_hi;
  const float* m_in;
  float* m_out;
  long long* den;
  int add_into;
  const int64_t* targets;
  float* loss;
  double* denom;
  int* status;
  // vocabulary shards: the matrix holds columns [v_base, v_base + V) of a vocabulary of v_total
  // columns (0 and V for a whole vocabulary); targets are global column indices
  int64_t v_base, v_total;
};
cudaError_t launch_dce_rowmax(const DceArgs& a, cudaStream_t st);
cudaError_t launch_dce_denom(const DceArgs& a, cudaStream_t st);
cudaError_t launch_dce_backward(const DceArgs& a, const float* grad, int reduction, void* dlogits, cudaStream_t st);
cudaError_t launch_dce_reduce(const float* loss, int64_t N, int reduction, float* out, cudaStream_t st);
cudaError_t launch_dce_finalize(const DceArgs& a, cudaStream_t st);

}  // namespace detattn
