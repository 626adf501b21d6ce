/*
 * libdetattn: C ABI of the exact, order-invariant softmax reduction (sm_103a).
 *
 * Sources (page title, section):
 *   "det-attn" - "API" (det_attn, rowmax, accumulate, finalize, det_attn_sharded),
 *                "Method" (global rowmax by a max-reduce; exact Kulisch sums NUM/DEN of
 *                signed int64 digits; KV shards compose by max and by digit add),
 *                "Correctness" and "Requirements and limits" (causal / non-causal,
 *                MHA / GQA, f32 / bf16 inputs, D <= 256, f32 output).
 *   "det-cross-entropy" - "API" (rowmax, denom_digits, finalize), "Usage" (vocab shards
 *                combine by max and by digit add), "Method".
 *
 * Numerical contract (every rounding is IEEE round-to-nearest-even with gradual underflow):
 *   score     s_ij = RN32(scale32 * RN32(sum_d q_id k_jd))      (exact dot, rounded once)
 *   rowmax    m_i  = max over valid keys j of s_ij; -0 -> +0; no valid key -> -inf
 *   weight    w_ij = exp32_det(RN32(s_ij - m_i)), a fixed binary32 routine
 *                    (Cody-Waite reduction + degree-7 Taylor polynomial)
 *   digits    NUM_id = sum_j w_ij v_jd, DEN_i = sum_j w_ij, exactly, as
 *             value = sum_k digit_k * 2^(E0 + 32 k); NUM: E0 = -320, 15 digits;
 *             DEN: E0 = -160, 6 digits.  Canonical form: digits 0..n-2 in [0, 2^32),
 *             the top digit signed.  Digit arrays compose by plain int64 addition (up to
 *             2^31 canonical arrays without overflow) and normalize back to canonical form.
 *   finalize  o_id = RN32(RN64(RN64(NUM_id) / RN64(DEN_i)))
 *   DCE       m_i = max_v x_iv; den_i = sum_v exp32_det(RN32(x_iv - m_i)) (DEN format);
 *             loss_i = RN32(RN64(log64_det(RN64(den_i)) + RN64(m_i - x_{i,t_i}))),
 *             denom_i = RN64(den_i); log64_det is a fixed binary64 routine.
 *
 * Conventions for every entry point:
 *   - Every device pointer is caller-owned device memory; the library allocates nothing
 *     and keeps no state between calls.  Work is enqueued on `stream` (NULL = the legacy
 *     default stream) and the call returns without synchronizing.
 *   - Host-side argument checks happen before any launch; on failure nothing is enqueued
 *     and a DA_E* code is returned.  A failed launch returns DA_ECUDA.
 *   - Data-dependent conditions are OR-ed into the optional device word `dev_status`
 *     (DA_STATUS_* bits); read it after synchronizing the stream.  Kernels never trap.
 *     When a status bit is set the affected outputs are unspecified.
 *   - Causal masking keeps key j for query i when j <= i (global positions, so it does
 *     not depend on how the keys are split) and requires Sq == Skv.
 *   - GQA: query head h reads key/value head h / (Hq / Hkv) (contiguous groups).
 */
#ifndef DETATTN_H
#define DETATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* da_stream_t; /* a cudaStream_t */

/* return codes */
#define DA_OK 0
#define DA_EINVAL 1      /* bad argument value (null pointer, range, scale, order) */
#define DA_ESHAPE 2      /* inconsistent shapes or strides */
#define DA_EDTYPE 3      /* unsupported or mismatched dtype */
#define DA_EALIGN 4      /* pointer not aligned to its element type */
#define DA_EWORKSPACE 5  /* workspace missing or too small */
#define DA_ECUDA 6       /* a CUDA launch failed */

/* device status bits */
#define DA_STATUS_NONFINITE 1        /* a non-finite input, score or intermediate was met */
#define DA_STATUS_ROWMAX_VIOLATION 2 /* a score above the supplied rowmax (weight clamped to 1) */
#define DA_STATUS_DIGIT_HEADROOM 4   /* a digit sum left the representable range */
#define DA_STATUS_BAD_TARGET 8       /* a target index outside [0, V) (its loss is NaN) */
#define DA_STATUS_TIMEOUT 16         /* a bounded wait inside a kernel gave up; outputs unspecified */

/* element types */
#define DA_F32 0
#define DA_BF16 1

#define DA_NUM_NDIG 15
#define DA_DEN_NDIG 6
#define DA_NUM_E0 (-320)
#define DA_DEN_E0 (-160)

/* A [B, H, S, D] tensor view: element strides, stride[3] must be 1. */
typedef struct {
  const void* ptr;
  int32_t dtype; /* DA_F32 or DA_BF16 */
  int64_t B, H, S, D;
  int64_t stride[4];
} da_tensor;

/* One attention problem.  q: [B, Hq, Sq, D]; k, v: [B, Hkv, Skv, D], same dtype;
 * 1 <= D <= 256; Hq % Hkv == 0; scale: NaN selects RN32(1/sqrt(D)), otherwise finite. */
typedef struct {
  da_tensor q, k, v;
  int32_t causal;
  float scale;
  int32_t* dev_status; /* optional device int32, OR-ed with DA_STATUS_* bits */
} da_attn_desc;

/* A [rows, cols] matrix view with a row stride in elements (columns contiguous). */
typedef struct {
  const void* ptr;
  int32_t dtype;
  int64_t rows, cols, row_stride;
} da_matrix;

/* ABI version (incremented on any incompatible change). */
int da_abi_version(void);

/* Static text for a DA_* return code. */
const char* da_status_string(int code);

/* Bytes of the key/value workspace da_rowmax and da_accumulate need: each call first
 * rewrites the keys (and values) of its range [kv_lo, kv_hi) there in the form its
 * kernels read (fixed-point digit slices), once per call rather than once per block of
 * query rows.  Device memory, 256-byte aligned, caller-owned; contents need no
 * initialization and are not meaningful after the call. */
size_t da_kv_workspace_bytes(const da_attn_desc* desc);

/* det-attn "API", rowmax: m[b,h,i] = max over keys j in [kv_lo, kv_hi) (causal: j <= i)
 * of s_ij.  m: device f32 [B, Hq, Sq], contiguous.  Rows with no valid key get -inf.
 * Shards combine with da_compose_max.  ws: at least da_kv_workspace_bytes(desc). */
int da_rowmax(const da_attn_desc* desc, int64_t kv_lo, int64_t kv_hi, float* m, void* ws, size_t ws_bytes,
              da_stream_t stream);

/* det-attn "API", accumulate: exact NUM/DEN digits over keys [kv_lo, kv_hi) with the
 * GLOBAL rowmax m (device f32 [B, Hq, Sq]).  num: device int64 [B, Hq, Sq, 15, D];
 * den: device int64 [B, Hq, Sq, 6], both contiguous.  add_into = 0 overwrites them with
 * the canonical digits of this range; add_into = 1 adds this range's sums to the
 * (canonical or plainly added) digits already there and leaves canonical digits.  A score
 * above m sets DA_STATUS_ROWMAX_VIOLATION.  ws: at least da_kv_workspace_bytes(desc). */
int da_accumulate(const da_attn_desc* desc, const float* m, int64_t kv_lo, int64_t kv_hi, int64_t* num,
                  int64_t* den, int add_into, void* ws, size_t ws_bytes, da_stream_t stream);

/* det-attn "Method", pass 2 and finalize over the whole key range in one call:
 * out = RN32(RN64(RN64(NUM) / RN64(DEN))) for NUM/DEN over keys [0, Skv) with the global
 * rowmax m (device f32 [B, Hq, Sq]).  out: device f32 [B, Hq, Sq, D], contiguous.  Equal bit
 * for bit to da_accumulate(.., 0, Skv, .., add_into = 0) followed by da_finalize; where the
 * tensor-PV kernel applies (D <= 128, at most 65,536 keys) it finalizes in its epilogue
 * and the NUM digits never reach device memory.  ws: at least da_workspace_bytes(desc, 1)
 * (the digits are kept there on the other paths). */
int da_accumulate_finalize(const da_attn_desc* desc, const float* m, float* out, void* ws, size_t ws_bytes,
                           da_stream_t stream);

/* det-attn "Method", shard composition: dst[i] = max(dst[i], src[i]) (f32, -0 -> +0). */
int da_compose_max(float* dst, const float* src, int64_t n, da_stream_t stream);

/* det-attn "Method", shard composition: dst[i] += src[i] (int64 digit add; exact). */
int da_compose_add(int64_t* dst, const int64_t* src, int64_t n, da_stream_t stream);

/* Canonical form of digit arrays laid out [nrows, ndig, inner] (NUM: ndig = 15,
 * inner = D; DEN and cross-entropy: ndig = 6, inner = 1), in place.  ndig must be 15 or 6.
 * A value outside the range sets DA_STATUS_DIGIT_HEADROOM. */
int da_normalize(int64_t* digits, int64_t nrows, int ndig, int64_t inner, int32_t* dev_status, da_stream_t stream);

/* det-attn "API", finalize: out[b,h,i,d] = RN32(RN64(RN64(NUM)/RN64(DEN))); accepts any
 * non-overflowing digits (canonical or plainly added).  out: device f32 [B, Hq, Sq, D]. */
int da_finalize(const int64_t* num, const int64_t* den, int64_t B, int64_t Hq, int64_t Sq, int64_t D, float* out,
                int32_t* dev_status, da_stream_t stream);

/* Bytes of workspace da_det_attn (nsplits <= 1) or da_det_attn_sharded needs. */
size_t da_workspace_bytes(const da_attn_desc* desc, int nsplits);

/* det-attn "API", det_attn: da_rowmax_cached, then da_accumulate_finalize_cached (below).
 * out: device f32 [B, Hq, Sq, D] contiguous; ws: device workspace of at least
 * da_workspace_bytes(desc, 1).  Bit-identical to da_det_attn_sharded for every split and
 * order. */
int da_det_attn(const da_attn_desc* desc, float* out, void* ws, size_t ws_bytes, da_stream_t stream);

/* det_attn with HOST buffers (the call of a program whose tensors live in host memory):
 * desc's q, k, v point to host memory holding [B, H, S, D] contiguous tensors (strides
 * D*S*H, D*S, D, 1), out to host f32 [B, Hq, Sq, D] contiguous.  The call copies the inputs
 * to the device workspace, runs da_det_attn there and copies the output back, in ngroups
 * groups of whole (batch, KV head) units (clamped to [1, B * Hkv]), each on an internal
 * stream of its own that waits for the work already queued on `stream`: one group's copies
 * overlap another's kernels, and the groups' kernels fill each other's tails.
 * Pinned host memory lets the copies proceed asynchronously; pageable memory works but the
 * driver stages it.  Returns once the work is queued; the output is in `out` when `stream`
 * has run it (synchronize `stream`), and the inputs must stay valid until then.  ws: device
 * workspace of at least da_det_attn_host_workspace_bytes(desc, ngroups) (the device copies
 * of Q, K, V and the output, and a da_det_attn workspace per group), 256-byte aligned.
 * Bit-identical to da_det_attn on device copies of the same tensors.  DA_ESHAPE for
 * non-contiguous tensors, DA_EINVAL for ngroups < 1; da_det_attn_host_workspace_bytes
 * returns 0 for an invalid descriptor. */
size_t da_det_attn_host_workspace_bytes(const da_attn_desc* desc, int ngroups);
int da_det_attn_host(const da_attn_desc* desc, float* out, int ngroups, void* ws, size_t ws_bytes,
                     da_stream_t stream);

/* The two passes of det_attn (det-attn "Method": a max-reduce, then the exact sums with the
 * global rowmax) over all keys, with the score cache.  The score of a pair is a fixed function
 * of its query and key rows, so pass 1 can hand every exact score it computes to pass 2:
 * for D <= 128 (at most 65,536 keys, and a cache of at most 16 GiB) da_rowmax_cached
 * prepares keys and values once, writes m (device f32 [B, Hq, Sq]) and stores every score it
 * rounds in the workspace's cache; da_accumulate_finalize_cached then reads the scores
 * instead of recomputing them and writes the f32 output, bit for bit what
 * da_accumulate_finalize gives.  Otherwise they are da_rowmax over [0, Skv) and
 * da_accumulate_finalize.  Both take the workspace of da_workspace_bytes(desc, 1); the
 * second call reads what the first left in it, so issue them in this order on one stream
 * with the same descriptor and workspace.  da_score_cache_bytes: the cache's share of that
 * workspace (0 when the scores are recomputed). */
size_t da_score_cache_bytes(const da_attn_desc* desc);
int da_rowmax_cached(const da_attn_desc* desc, float* m, void* ws, size_t ws_bytes, da_stream_t stream);
int da_accumulate_finalize_cached(const da_attn_desc* desc, const float* m, float* out, void* ws, size_t ws_bytes,
                                  da_stream_t stream);

/* det-attn "API", det_attn_sharded: the keys split into nsplits contiguous shards of
 * kv_splits[k] keys (host array, sum = Skv, entries >= 0), visited in the order
 * order[0..nsplits-1] (host array, a permutation; NULL = 0, 1, ...).  Rowmax of every
 * shard composed by max, then the digits of every shard (with the global rowmax)
 * composed by add, then finalize.  Bit-identical to da_det_attn for any split and order. */
int da_det_attn_sharded(const da_attn_desc* desc, const int64_t* kv_splits, int nsplits, const int32_t* order,
                        float* out, void* ws, size_t ws_bytes, da_stream_t stream);

/* det-cross-entropy "API", rowmax: m[i] = max over v in [v_lo, v_hi) of logits[i, v];
 * -0 -> +0; empty range -> -inf.  m: device f32 [rows]. */
int dce_rowmax(const da_matrix* logits, int64_t v_lo, int64_t v_hi, float* m, int32_t* dev_status,
               da_stream_t stream);

/* det-cross-entropy "API", denom_digits: exact digits of sum over v in [v_lo, v_hi) of
 * exp32_det(RN32(logits[i, v] - m[i])), m the GLOBAL rowmax (device f32 [rows]).
 * den: device int64 [rows, 6]; add_into as for da_accumulate. */
int dce_denom_digits(const da_matrix* logits, const float* m, int64_t v_lo, int64_t v_hi, int64_t* den,
                     int add_into, int32_t* dev_status, da_stream_t stream);

/* det-cross-entropy "API", finalize: loss[i] (device f32 [rows]) and denom[i] = RN64(den_i)
 * (device f64 [rows]) from composed digits (any non-overflowing form), the full logits,
 * targets (device int64 [rows]) and the global rowmax.  A target outside [0, cols) gives
 * a NaN loss and DA_STATUS_BAD_TARGET. */
int dce_finalize(const int64_t* den, const da_matrix* logits, const int64_t* targets, const float* m, float* loss,
                 double* denom, int32_t* dev_status, da_stream_t stream);

/* det-cross-entropy "API", the deterministic dLogits of cross_entropy ("Method": the
 * gradient softmax(x_i) - onehot(t_i)), from forward's state (rowmax m, denom; targets):
 *   p = RN32(RN64(exp32_det(RN32(logits[i, v] - m[i])) / denom[i])),
 *   g = RN32(p - [v == targets[i]]),  dlogits[i, v] = RN32(go_i * g),
 * go_i = grad[i] for reduction 0 ("none", grad: device f32 [rows]), grad[0] for 1 ("sum"),
 * RN32(RN64(grad[0] / rows)) for 2 ("mean") (grad: device f32 [1]).  The pages fix the
 * value; the rounding sequence is this library's reading.  dlogits: device [rows, cols],
 * contiguous, of the logits' dtype (bf16 logits: the f32 value rounded to nearest even).
 * A logit above m sets DA_STATUS_ROWMAX_VIOLATION and is clamped as in the forward; a
 * target outside [0, cols) subtracts nothing.  Bit-identical for any vocab split of the
 * forward (its m and denom are). */
int dce_backward(const da_matrix* logits, const int64_t* targets, const float* m, const double* denom,
                 const float* grad, int reduction, void* dlogits, int32_t* dev_status, da_stream_t stream);

/* Vocabulary-parallel forms (det-cross-entropy, "Usage": the vocabulary sharded over ranks
 * composes by a max and a digit add; the logit of a row's target lives on one shard).
 * logits holds columns [v_base, v_base + cols) of a vocabulary of v_total columns; targets
 * are global column indices; den, m and denom are the composed (global) values.
 *   dce_finalize_shard: denom as dce_finalize; loss_i = the full loss for a row whose target
 *   lies in this shard, +0 for a row whose target lies in another shard, NaN with
 *   DA_STATUS_BAD_TARGET for a target outside [0, v_total).  Summing the shards' losses
 *   (exactly one term is nonzero) gives dce_finalize's loss over the whole vocabulary.
 *   DA_EINVAL unless 0 <= v_base and v_base + cols <= v_total.
 *   dce_backward_shard: the dLogits columns of this shard (as dce_backward; the one-hot is
 *   subtracted where the target falls in the shard). */
int dce_finalize_shard(const int64_t* den, const da_matrix* logits, int64_t v_base, int64_t v_total,
                       const int64_t* targets, const float* m, float* loss, double* denom, int32_t* dev_status,
                       da_stream_t stream);
int dce_backward_shard(const da_matrix* logits, int64_t v_base, const int64_t* targets, const float* m,
                       const double* denom, const float* grad, int reduction, void* dlogits, int32_t* dev_status,
                       da_stream_t stream);

/* det-cross-entropy "API", the loss reduction of cross_entropy: with S the exact sum of the
 * rows f32 losses (a Kulisch accumulator), reduction 1 ("sum") gives RN32(RN64(S)), 2
 * ("mean") RN32(RN64(RN64(S) / rows)); a NaN loss gives NaN, infinite losses their IEEE
 * sum; rows == 0 gives 0 ("sum") or NaN ("mean", 0 / 0), and loss may then be null.
 * loss: device f32 [rows]; out: device f32 [1].  Independent of the rows' order. */
int dce_reduce(const float* loss, int64_t rows, int reduction, float* out, da_stream_t stream);

/* Static-scratch variant of the cross-entropy forward, for callers that cannot allocate
 * device memory: code that runs where cudaMalloc is not allowed or not wanted, such as a
 * host framework whose device memory is owned by another allocator, an embedded runtime
 * with a fixed memory budget, or a call site that must not trigger allocation.  The pages
 * have no counterpart of this entry point; it computes what dce_rowmax over [0, cols),
 * dce_denom_digits over [0, cols) and dce_finalize compute, bit for bit, but keeps the
 * rowmax and the denominator digits in a file-scope device array of
 * DA_STATIC_MAX_ROWS rows (3.25 MiB) instead of caller memory.  It calls no cudaMalloc,
 * cudaFree or allocating library routine.
 *   - The caller still passes logits, targets (device int64 [rows]), loss (device f32
 *     [rows]) and denom (device f64 [rows]).
 *   - rows > DA_STATIC_MAX_ROWS returns DA_EWORKSPACE (the static scratch is too small).
 *   - Every GPU that loads the library holds the array until the process exits.  The
 *     first call on a device looks up the array's device address (once per device, with
 *     that device current); make that first call before any stream capture.
 *   - The looked-up address is kept for the life of the process: do not use the library
 *     across a cudaDeviceReset (or anything else that destroys and recreates the device's
 *     primary context), since the kept address would then be stale.
 *   - Every call shares the one array: calls whose work overlaps on the GPU (different
 *     streams, or several host threads) race on it.  Serialize them.  Each call overwrites
 *     every scratch entry it reads, so no clearing is needed between calls. */
#define DA_STATIC_MAX_ROWS 65536
int dce_forward_static(const da_matrix* logits, const int64_t* targets, float* loss, double* denom,
                       int32_t* dev_status, da_stream_t stream);

/* ---- Probes.  None computes anything of the method, and the pages have no counterpart
 * of them: one measures a hardware rate the benchmark reports against, one exercises the
 * bounded-wait path of the pipelined kernels, one checks the packed two-lane forms of the
 * cross-entropy arithmetic against the scalar forms. ---- */

/* Issue rate of exact 32 x 32 -> 64-bit integer multiply-adds (mad.wide.s32): nblocks CTAs of
 * 512 threads each run iters iterations of da_probe_int_mac_per_thread_iter() independent
 * multiply-adds per thread.  Time the launch on `stream` to get the GPU's rate; sink:
 * device int64 [1], written only in a practically unreachable case (it keeps the chain
 * live).  DA_EINVAL for iters < 0, nblocks outside [1, 2^20] or a null sink. */
int da_probe_int_mac(int64_t iters, int nblocks, int64_t* sink, da_stream_t stream);
int64_t da_probe_int_mac_per_thread_iter(void);

/* The cross-entropy kernels evaluate the exponentials of two adjacent logits (page
 * "det-cross-entropy", section "Method": the weight exp32_det(RN32(x - m))), and the backward
 * their quotients by the row's denominator, two at a time on the packed FP32 instructions.
 * This runs the packed and the scalar device forms on every binary32 bit pattern lo_bits,
 * lo_bits + 1, ..., lo_bits + count - 1 (mod 2^32) and adds to *mismatches (device int64 [1],
 * 8-byte aligned, not cleared here) the number of patterns whose results differ in any bit.
 * which 0: the reduction and polynomial of the exponential, the pattern read as x (NaN taken
 * as -inf, then clamped to [-104, 0] as the kernels clamp).  which 1: the quotient candidate
 * and its residual estimate, the pattern's low 24 bits giving p in [0.5, 2) and a hash of it
 * the divisor in [1, 2^21).  DA_EINVAL for which outside {0, 1}, count outside [0, 2^32] or a
 * null pointer. */
int da_probe_packed(int which, uint32_t lo_bits, int64_t count, int64_t* mismatches, da_stream_t stream);

/* One warp waits on an mbarrier phase that nothing completes, through the bounded wait the
 * pipelined kernels use (it gives up after about 2 s).  The kernel then ends normally and
 * ORs DA_STATUS_TIMEOUT into *dev_status (device int32, required): the caller reads the
 * status, and the context stays usable.  Exercises the timeout path without a fault. */
int da_probe_bounded_wait(int32_t* dev_status, da_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DETATTN_H */
