// Host side of the C ABI declared in include/detattn.h: argument checks, workspace
// layout, and the launch sequences of the fused and the KV-sharded paths (page
// "det-attn", section "API"; page "det-cross-entropy", section "API").
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/detattn.h"
#include "attn_kernels.h"

using namespace detattn;

namespace {

constexpr int64_t kMaxS = (int64_t)1 << 30;

int elem_size(int dtype) { return dtype == DA_F32 ? 4 : 2; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_tensor(const da_tensor& t) {
  if (t.dtype != DA_F32 && t.dtype != DA_BF16) return DA_EDTYPE;
  if (t.B < 0 || t.H < 1 || t.S < 0 || t.D < 1 || t.D > 256) return DA_ESHAPE;
  if (t.S > kMaxS || t.B > 65535 || t.H > 65535) return DA_ESHAPE;   // grid.z / grid.y limits
  if (t.stride[3] != 1) return DA_ESHAPE;
  if (t.B * t.S > 0 && t.ptr == nullptr) return DA_EINVAL;
  if (!aligned(t.ptr, elem_size(t.dtype))) return DA_EALIGN;
  return DA_OK;
}

int check_desc(const da_attn_desc* d) {
  if (!d) return DA_EINVAL;
  int e;
  if ((e = check_tensor(d->q)) || (e = check_tensor(d->k)) || (e = check_tensor(d->v))) return e;
  if (d->q.dtype != d->k.dtype || d->q.dtype != d->v.dtype) return DA_EDTYPE;
  if (d->k.B != d->q.B || d->v.B != d->q.B || d->k.D != d->q.D || d->v.D != d->q.D) return DA_ESHAPE;
  if (d->v.H != d->k.H || d->v.S != d->k.S) return DA_ESHAPE;
  if (d->q.H % d->k.H != 0) return DA_ESHAPE;
  if (d->causal && d->q.S != d->k.S) return DA_EINVAL;
  if (!std::isnan(d->scale) && !std::isfinite(d->scale)) return DA_EINVAL;
  return DA_OK;
}

AttnArgs make_args(const da_attn_desc* d) {
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = d->q.ptr; a.k = d->k.ptr; a.v = d->v.ptr;
  for (int t = 0; t < 4; t++) { a.qs[t] = d->q.stride[t]; a.ks[t] = d->k.stride[t]; a.vs[t] = d->v.stride[t]; }
  a.dtype = d->q.dtype;
  a.B = (int)d->q.B; a.Hq = (int)d->q.H; a.Hkv = (int)d->k.H;
  a.Sq = (int)d->q.S; a.Skv = (int)d->k.S; a.D = (int)d->q.D;
  a.causal = d->causal ? 1 : 0;
  a.scale32 = std::isnan(d->scale) ? (float)(1.0 / std::sqrt((double)d->q.D)) : d->scale;
  a.status = d->dev_status;
  return a;
}

int launched(cudaError_t e) { return e == cudaSuccess ? DA_OK : DA_ECUDA; }

size_t round_up(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t m, m2, num, den, kv, sc, sc_bytes, total;
};

size_t kv_bytes(const da_attn_desc* d) { return kv_prep_bytes((int)d->k.B, (int)d->k.H, (int)d->k.S, (int)d->k.D); }

// The score cache of the whole-range path (D <= 128, at most ACC_TP_MAX_TILES key tiles,
// causal only with Sq == Skv): bytes, or 0 when the path recomputes the scores instead (other
// head dimensions, or a cache above kScoreCacheCap).
constexpr size_t kScoreCacheCap = (size_t)16 << 30;
size_t sc_bytes(const da_attn_desc* d, int* nkt = nullptr, int64_t* per_bh = nullptr) {
  int n;
  int64_t pb;
  if (d->q.D > 128 || (d->k.S + KTILE - 1) / KTILE > ACC_TP_MAX_TILES) return 0;
  const size_t b = score_cache_bytes((int)d->q.B, (int)d->q.H, (int)d->q.S, (int)d->k.S, d->causal, &n, &pb);
  if (b > kScoreCacheCap) return 0;
  if (nkt) *nkt = n;
  if (per_bh) *per_bh = pb;
  return b;
}

WsLayout ws_layout(const da_attn_desc* d, int nsplits) {
  const size_t rows = (size_t)d->q.B * d->q.H * d->q.S;
  WsLayout w;
  w.m = 0;
  w.m2 = round_up(rows * 4);
  w.num = w.m2 + (nsplits > 1 ? round_up(rows * 4) : 0);
  w.den = w.num + round_up(rows * DA_NUM_NDIG * (size_t)d->q.D * 8);
  w.kv = w.den + round_up(rows * DA_DEN_NDIG * 8);
  w.sc = w.kv + round_up(kv_bytes(d));
  w.sc_bytes = nsplits == 1 ? sc_bytes(d) : 0;
  w.total = w.sc + round_up(w.sc_bytes);
  return w;
}

int check_kv_ws(const da_attn_desc* d, void* ws, size_t ws_bytes) {
  if (!ws || ws_bytes < kv_bytes(d)) return DA_EWORKSPACE;
  if (!aligned(ws, 256)) return DA_EALIGN;
  return DA_OK;
}

int check_matrix(const da_matrix* x) {
  if (!x) return DA_EINVAL;
  if (x->dtype != DA_F32 && x->dtype != DA_BF16) return DA_EDTYPE;
  if (x->rows < 0 || x->cols < 0 || x->row_stride < x->cols) return DA_ESHAPE;
  if (x->rows > ((int64_t)1 << 31) - 1) return DA_ESHAPE;
  if (x->rows * x->cols > 0 && !x->ptr) return DA_EINVAL;
  if (!aligned(x->ptr, elem_size(x->dtype))) return DA_EALIGN;
  return DA_OK;
}

DceArgs make_dce(const da_matrix* x) {
  DceArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = x->ptr; a.dtype = x->dtype; a.N = x->rows; a.V = x->cols; a.rs = x->row_stride;
  a.v_base = 0; a.v_total = x->cols;
  return a;
}

}  // namespace

// da_accumulate with the internal canon_in flag (the sharded composition's own digits)
int accumulate_range(const da_attn_desc* desc, const float* m, int64_t kv_lo, int64_t kv_hi, int64_t* num,
                     int64_t* den, int add_into, int canon_in, void* ws, size_t ws_bytes, da_stream_t stream);

#define DA_EXPORT __attribute__((visibility("default")))

extern "C" {

DA_EXPORT int da_abi_version(void) { return 3; }

DA_EXPORT const char* da_status_string(int code) {
  switch (code) {
    case DA_OK: return "ok";
    case DA_EINVAL: return "invalid argument";
    case DA_ESHAPE: return "inconsistent shape or stride";
    case DA_EDTYPE: return "unsupported or mismatched dtype";
    case DA_EALIGN: return "misaligned pointer";
    case DA_EWORKSPACE: return "workspace missing or too small";
    case DA_ECUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

DA_EXPORT size_t da_kv_workspace_bytes(const da_attn_desc* desc) {
  if (check_desc(desc)) return 0;
  return kv_bytes(desc);
}

DA_EXPORT int da_rowmax(const da_attn_desc* desc, int64_t kv_lo, int64_t kv_hi, float* m, void* ws, size_t ws_bytes,
                        da_stream_t stream) {
  int e = check_desc(desc);
  if (e) return e;
  if (kv_lo < 0 || kv_hi < kv_lo || kv_hi > desc->k.S) return DA_EINVAL;
  if (desc->q.B * desc->q.S == 0) return DA_OK;
  if (!m) return DA_EINVAL;
  if (!aligned(m, 4)) return DA_EALIGN;
  if ((e = check_kv_ws(desc, ws, ws_bytes))) return e;
  AttnArgs a = make_args(desc);
  a.kv_lo = (int)kv_lo; a.kv_hi = (int)kv_hi; a.m_out = m;
  KvPrep p = kv_prep_layout(ws, a.B, a.Hkv, a.Skv, a.D, 0);
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_kv_prep(a, p, st) != cudaSuccess) return DA_ECUDA;
  return launched(launch_rowmax(a, p, st));
}

DA_EXPORT int da_accumulate(const da_attn_desc* desc, const float* m, int64_t kv_lo, int64_t kv_hi, int64_t* num,
                            int64_t* den, int add_into, void* ws, size_t ws_bytes, da_stream_t stream) {
  return accumulate_range(desc, m, kv_lo, kv_hi, num, den, add_into, 0, ws, ws_bytes, stream);
}

}  // extern "C"

int accumulate_range(const da_attn_desc* desc, const float* m, int64_t kv_lo, int64_t kv_hi, int64_t* num,
                     int64_t* den, int add_into, int canon_in, void* ws, size_t ws_bytes, da_stream_t stream) {
  int e = check_desc(desc);
  if (e) return e;
  if (kv_lo < 0 || kv_hi < kv_lo || kv_hi > desc->k.S) return DA_EINVAL;
  if (desc->q.B * desc->q.S == 0) return DA_OK;
  if (!m || !num || !den) return DA_EINVAL;
  if (!aligned(m, 4) || !aligned(num, 8) || !aligned(den, 8)) return DA_EALIGN;
  if ((e = check_kv_ws(desc, ws, ws_bytes))) return e;
  AttnArgs a = make_args(desc);
  a.kv_lo = (int)kv_lo; a.kv_hi = (int)kv_hi;
  a.m_in = m; a.num = (long long*)num; a.den = (long long*)den; a.add_into = add_into ? 1 : 0;
  a.canon_in = canon_in;
  KvPrep p = kv_prep_layout(ws, a.B, a.Hkv, a.Skv, a.D, 1);
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_kv_prep(a, p, st) != cudaSuccess) return DA_ECUDA;
  return launched(launch_accumulate(a, p, st));
}

extern "C" {

DA_EXPORT int da_compose_max(float* dst, const float* src, int64_t n, da_stream_t stream) {
  if (n < 0) return DA_EINVAL;
  if (n == 0) return DA_OK;
  if (!dst || !src) return DA_EINVAL;
  if (!aligned(dst, 4) || !aligned(src, 4)) return DA_EALIGN;
  return launched(launch_compose_max(dst, src, n, (cudaStream_t)stream));
}

DA_EXPORT int da_compose_add(int64_t* dst, const int64_t* src, int64_t n, da_stream_t stream) {
  if (n < 0) return DA_EINVAL;
  if (n == 0) return DA_OK;
  if (!dst || !src) return DA_EINVAL;
  if (!aligned(dst, 16) || !aligned(src, 16)) return DA_EALIGN;
  return launched(launch_compose_add((long long*)dst, (const long long*)src, n, (cudaStream_t)stream));
}

DA_EXPORT int da_normalize(int64_t* digits, int64_t nrows, int ndig, int64_t inner, int32_t* dev_status, da_stream_t stream) {
  if (nrows < 0 || inner < 1 || (ndig != DA_NUM_NDIG && ndig != DA_DEN_NDIG)) return DA_EINVAL;
  if (nrows == 0) return DA_OK;
  if (!digits) return DA_EINVAL;
  if (!aligned(digits, 8)) return DA_EALIGN;
  return launched(launch_normalize((long long*)digits, nrows, ndig, inner, dev_status, (cudaStream_t)stream));
}

DA_EXPORT int da_finalize(const int64_t* num, const int64_t* den, int64_t B, int64_t Hq, int64_t Sq, int64_t D, float* out,
                int32_t* dev_status, da_stream_t stream) {
  if (B < 0 || Hq < 0 || Sq < 0 || D < 1 || D > 256) return DA_ESHAPE;
  const int64_t rows = B * Hq * Sq;
  if (rows == 0) return DA_OK;
  if (!num || !den || !out) return DA_EINVAL;
  if (!aligned(num, 8) || !aligned(den, 8) || !aligned(out, 4)) return DA_EALIGN;
  return launched(launch_finalize((const long long*)num, (const long long*)den, rows, (int)D, out, dev_status,
                                  (cudaStream_t)stream));
}

DA_EXPORT size_t da_workspace_bytes(const da_attn_desc* desc, int nsplits) {
  if (check_desc(desc)) return 0;
  return ws_layout(desc, nsplits).total;
}

DA_EXPORT int da_accumulate_finalize(const da_attn_desc* desc, const float* m, float* out, void* ws, size_t ws_bytes,
                                     da_stream_t stream) {
  int e = check_desc(desc);
  if (e) return e;
  if (desc->q.B * desc->q.S == 0) return DA_OK;
  if (!m || !out) return DA_EINVAL;
  if (!aligned(m, 4) || !aligned(out, 4)) return DA_EALIGN;
  WsLayout w = ws_layout(desc, 1);
  if (!ws || ws_bytes < w.total) return DA_EWORKSPACE;
  if (!aligned(ws, 256)) return DA_EALIGN;
  char* base = (char*)ws;
  int64_t* num = (int64_t*)(base + w.num);
  int64_t* den = (int64_t*)(base + w.den);
  void* kv = base + w.kv;
  const size_t kvb = ws_bytes - w.kv;
  if ((e = check_kv_ws(desc, kv, kvb))) return e;
  AttnArgs a = make_args(desc);
  a.kv_lo = 0; a.kv_hi = (int)desc->k.S;
  a.m_in = m; a.num = (long long*)num; a.den = (long long*)den; a.add_into = 0;
  KvPrep p = kv_prep_layout(kv, a.B, a.Hkv, a.Skv, a.D, 1);
  if (accumulate_is_tp(a, p)) {   // finalize in the epilogue: no NUM digits in device memory
    a.out = out;
    cudaStream_t st = (cudaStream_t)stream;
    if (launch_kv_prep(a, p, st) != cudaSuccess) return DA_ECUDA;
    return launched(launch_accumulate(a, p, st));
  }
  if ((e = da_accumulate(desc, m, 0, desc->k.S, num, den, 0, kv, kvb, stream))) return e;
  return da_finalize(num, den, desc->q.B, desc->q.H, desc->q.S, desc->q.D, out, desc->dev_status, stream);
}

DA_EXPORT size_t da_score_cache_bytes(const da_attn_desc* desc) {
  if (check_desc(desc)) return 0;
  return sc_bytes(desc);
}

DA_EXPORT int da_rowmax_cached(const da_attn_desc* desc, float* m, void* ws, size_t ws_bytes, da_stream_t stream) {
  int e = check_desc(desc);
  if (e) return e;
  if (desc->q.B * desc->q.S == 0) return DA_OK;
  if (!m) return DA_EINVAL;
  if (!aligned(m, 4)) return DA_EALIGN;
  WsLayout w = ws_layout(desc, 1);
  if (!ws || ws_bytes < w.total) return DA_EWORKSPACE;
  if (!aligned(ws, 256)) return DA_EALIGN;
  char* base = (char*)ws;
  if (!w.sc_bytes) return da_rowmax(desc, 0, desc->k.S, m, base + w.kv, ws_bytes - w.kv, stream);
  AttnArgs a = make_args(desc);
  a.kv_lo = 0; a.kv_hi = (int)desc->k.S; a.m_out = m;
  a.scores = (float*)(base + w.sc);
  sc_bytes(desc, &a.sc_nkt, &a.sc_per_bh);
  KvPrep p = kv_prep_layout(base + w.kv, a.B, a.Hkv, a.Skv, a.D, 1);   // keys and values, once for both passes
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_kv_prep(a, p, st) != cudaSuccess) return DA_ECUDA;
  return launched(launch_rowmax(a, p, st));
}

DA_EXPORT int da_accumulate_finalize_cached(const da_attn_desc* desc, const float* m, float* out, void* ws,
                                            size_t ws_bytes, da_stream_t stream) {
  int e = check_desc(desc);
  if (e) return e;
  if (desc->q.B * desc->q.S == 0) return DA_OK;
  if (!m || !out) return DA_EINVAL;
  if (!aligned(m, 4) || !aligned(out, 4)) return DA_EALIGN;
  WsLayout w = ws_layout(desc, 1);
  if (!ws || ws_bytes < w.total) return DA_EWORKSPACE;
  if (!aligned(ws, 256)) return DA_EALIGN;
  if (!w.sc_bytes) return da_accumulate_finalize(desc, m, out, ws, ws_bytes, stream);
  char* base = (char*)ws;
  AttnArgs a = make_args(desc);
  a.kv_lo = 0; a.kv_hi = (int)desc->k.S;
  a.m_in = m; a.out = out; a.add_into = 0;
  a.num = (long long*)(base + w.num); a.den = (long long*)(base + w.den);
  a.scores = (float*)(base + w.sc);
  sc_bytes(desc, &a.sc_nkt, &a.sc_per_bh);
  KvPrep p = kv_prep_layout(base + w.kv, a.B, a.Hkv, a.Skv, a.D, 1);   // prepared by da_rowmax_cached
  if (!accumulate_is_tp(a, p)) return DA_EINVAL;
  // the work order lives in the NUM digit room, which the fused finalize never writes
  if (tp_order_bytes(a) <= w.den - w.num && (e = launched(launch_tp_order(a, base + w.num, (cudaStream_t)stream))))
    return e;
  return launched(launch_accumulate(a, p, (cudaStream_t)stream));
}

DA_EXPORT int da_det_attn(const da_attn_desc* desc, float* out, void* ws, size_t ws_bytes, da_stream_t stream) {
  int e = check_desc(desc);
  if (e) return e;
  if (desc->q.B * desc->q.S == 0) return DA_OK;
  if (!out) return DA_EINVAL;
  WsLayout w = ws_layout(desc, 1);
  if (!ws || ws_bytes < w.total) return DA_EWORKSPACE;
  if (!aligned(ws, 256)) return DA_EALIGN;
  float* m = (float*)((char*)ws + w.m);
  if ((e = da_rowmax_cached(desc, m, ws, ws_bytes, stream))) return e;
  return da_accumulate_finalize_cached(desc, m, out, ws, ws_bytes, stream);
}

}  // extern "C"

namespace {

bool dense(const da_tensor& t) {   // [B, H, S, D] contiguous
  return t.stride[3] == 1 && t.stride[2] == t.D && t.stride[1] == t.S * t.D && t.stride[0] == t.H * t.S * t.D;
}

// det_attn with host buffers, split into groups of whole (batch, KV head) units: the flattened
// units [u0, u1) are contiguous in Q, K, V and the output, and each group is an independent
// det_attn problem (one batch of (u1 - u0) KV heads and their query heads).
// Streams for the host-buffer path's groups, created once per device and reused: creating
// them on every call costs host time while the first groups' work already runs.  A call takes
// what it needs and gives it back; calls from several host threads each get their own.
struct StreamPool {
  std::mutex mu;
  std::vector<std::pair<int, cudaStream_t>> free;   // (device, stream)
};
StreamPool& stream_pool() {
  static StreamPool* p = new StreamPool;   // never destroyed: streams outlive static destructors
  return *p;
}
int take_streams(int n, std::vector<cudaStream_t>& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DA_ECUDA;
  StreamPool& p = stream_pool();
  {
    std::lock_guard<std::mutex> lk(p.mu);
    for (size_t i = 0; i < p.free.size() && (int)out.size() < n;) {
      if (p.free[i].first == dev) {
        out.push_back(p.free[i].second);
        p.free.erase(p.free.begin() + (long)i);
      } else {
        i++;
      }
    }
  }
  while ((int)out.size() < n) {
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return DA_ECUDA;
    out.push_back(s);
  }
  return DA_OK;
}
void give_streams(const std::vector<cudaStream_t>& in) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  StreamPool& p = stream_pool();
  std::lock_guard<std::mutex> lk(p.mu);
  for (cudaStream_t s : in) p.free.emplace_back(dev, s);
}

struct HostPlan {
  int64_t units, per, ngroups;       // units = B * Hkv; per = units per group
  size_t qb, kb, ob;                 // bytes of one unit's query rows, key (= value) rows, output rows
  size_t q_off, k_off, v_off, o_off, w_off, w_bytes, total;
};

da_attn_desc group_desc(const da_attn_desc* d, const void* q, const void* k, const void* v, int64_t n) {
  da_attn_desc g = *d;
  const int64_t r = d->q.H / d->k.H;
  auto set = [](da_tensor& t, const void* ptr, int64_t h) {
    t.ptr = ptr;
    t.B = 1;
    t.H = h;
    t.stride[3] = 1;
    t.stride[2] = t.D;
    t.stride[1] = t.S * t.D;
    t.stride[0] = h * t.S * t.D;
  };
  set(g.q, q, n * r);
  set(g.k, k, n);
  set(g.v, v, n);
  return g;
}

int host_plan(const da_attn_desc* d, int ngroups, HostPlan& p) {
  int e = check_desc(d);
  if (e) return e;
  if (!dense(d->q) || !dense(d->k) || !dense(d->v)) return DA_ESHAPE;
  if (ngroups < 1) return DA_EINVAL;
  const int64_t r = d->q.H / d->k.H;
  const size_t es = (size_t)elem_size(d->q.dtype);
  p.units = d->q.B * d->k.H;
  p.ngroups = p.units == 0 ? 0 : std::min<int64_t>(ngroups, p.units);
  p.per = p.ngroups == 0 ? 0 : (p.units + p.ngroups - 1) / p.ngroups;
  p.ngroups = p.per == 0 ? 0 : (p.units + p.per - 1) / p.per;
  p.qb = (size_t)r * d->q.S * d->q.D * es;
  p.kb = (size_t)d->k.S * d->k.D * es;
  p.ob = (size_t)r * d->q.S * d->q.D * 4;
  p.q_off = 0;
  p.k_off = round_up(p.q_off + p.units * p.qb);
  p.v_off = round_up(p.k_off + p.units * p.kb);
  p.o_off = round_up(p.v_off + p.units * p.kb);
  p.w_off = round_up(p.o_off + p.units * p.ob);
  p.w_bytes = 0;
  if (p.per > 0) {
    const da_attn_desc g = group_desc(d, d->q.ptr, d->k.ptr, d->v.ptr, p.per);
    p.w_bytes = ws_layout(&g, 1).total;
  }
  p.total = p.w_off + p.ngroups * round_up(p.w_bytes);   // one det_attn workspace per group
  return DA_OK;
}

}  // namespace

extern "C" {

DA_EXPORT size_t da_det_attn_host_workspace_bytes(const da_attn_desc* desc, int ngroups) {
  HostPlan p;
  return host_plan(desc, ngroups, p) ? 0 : p.total;
}

DA_EXPORT int da_det_attn_host(const da_attn_desc* desc, float* out, int ngroups, void* ws, size_t ws_bytes,
                               da_stream_t stream) {
  HostPlan p;
  int e = host_plan(desc, ngroups, p);
  if (e) return e;
  if (desc->q.B * desc->q.S == 0) return DA_OK;
  if (!out) return DA_EINVAL;
  if (!ws || ws_bytes < p.total) return DA_EWORKSPACE;
  if (!aligned(ws, 256)) return DA_EALIGN;
  char* base = (char*)ws;
  cudaStream_t st = (cudaStream_t)stream;
  std::vector<cudaStream_t> gs;
  std::vector<cudaEvent_t> ev;
  auto event = [&]() {
    cudaEvent_t x = nullptr;
    if (cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess) return (cudaEvent_t) nullptr;
    ev.push_back(x);
    return x;
  };
  auto run = [&]() -> int {
    cudaEvent_t start = event();
    if (!start || cudaEventRecord(start, st) != cudaSuccess) return DA_ECUDA;
    if (int r = take_streams((int)p.ngroups, gs)) return r;
    const char* qh = (const char*)desc->q.ptr;
    const char* kh = (const char*)desc->k.ptr;
    const char* vh = (const char*)desc->v.ptr;
    // One stream per group: its inputs up, its det_attn (own workspace), its output down; the
    // groups' streams run side by side, so one group's copies overlap another's kernels and the
    // kernels of several groups fill each other's tails.  Every group's uploads are enqueued
    // before any kernel, so the copy engines have them all from the start (chaining them one
    // group after another measured slower).
    for (int64_t g = 0; g < p.ngroups; g++) {
      const int64_t u0 = g * p.per, n = std::min(p.per, p.units - u0);
      if (cudaStreamWaitEvent(gs[g], start, 0) != cudaSuccess ||
          cudaMemcpyAsync(base + p.q_off + u0 * p.qb, qh + u0 * p.qb, n * p.qb, cudaMemcpyHostToDevice, gs[g]) !=
              cudaSuccess ||
          cudaMemcpyAsync(base + p.k_off + u0 * p.kb, kh + u0 * p.kb, n * p.kb, cudaMemcpyHostToDevice, gs[g]) !=
              cudaSuccess ||
          cudaMemcpyAsync(base + p.v_off + u0 * p.kb, vh + u0 * p.kb, n * p.kb, cudaMemcpyHostToDevice, gs[g]) !=
              cudaSuccess)
        return DA_ECUDA;
    }
    for (int64_t g = 0; g < p.ngroups; g++) {
      const int64_t u0 = g * p.per, n = std::min(p.per, p.units - u0);
      float* od = (float*)(base + p.o_off + u0 * p.ob);
      const da_attn_desc gd = group_desc(desc, base + p.q_off + u0 * p.qb, base + p.k_off + u0 * p.kb,
                                         base + p.v_off + u0 * p.kb, n);
      const int r = da_det_attn(&gd, od, base + p.w_off + g * round_up(p.w_bytes), p.w_bytes, (da_stream_t)gs[g]);
      if (r) return r;
      if (cudaMemcpyAsync((char*)out + u0 * p.ob, od, n * p.ob, cudaMemcpyDeviceToHost, gs[g]) != cudaSuccess)
        return DA_ECUDA;
      cudaEvent_t done = event();
      if (!done || cudaEventRecord(done, gs[g]) != cudaSuccess || cudaStreamWaitEvent(st, done, 0) != cudaSuccess)
        return DA_ECUDA;
    }
    return DA_OK;
  };
  const int r = run();
  for (cudaEvent_t x : ev) cudaEventDestroy(x);   // released once the work that uses them has run
  if (r == DA_OK) give_streams(gs);               // their work is ordered before the caller's stream
  else
    for (cudaStream_t x : gs) cudaStreamDestroy(x);
  return r;
}

DA_EXPORT int da_det_attn_sharded(const da_attn_desc* desc, const int64_t* kv_splits, int nsplits, const int32_t* order,
                        float* out, void* ws, size_t ws_bytes, da_stream_t stream) {
  int e = check_desc(desc);
  if (e) return e;
  if (nsplits < 1 || !kv_splits) return DA_EINVAL;
  std::vector<int64_t> lo(nsplits), hi(nsplits);
  int64_t acc = 0;
  for (int k = 0; k < nsplits; k++) {
    if (kv_splits[k] < 0) return DA_EINVAL;
    lo[k] = acc;
    acc += kv_splits[k];
    hi[k] = acc;
  }
  if (acc != desc->k.S) return DA_EINVAL;
  std::vector<int32_t> ord(nsplits);
  std::vector<char> seen(nsplits, 0);
  for (int k = 0; k < nsplits; k++) {
    int32_t o = order ? order[k] : k;
    if (o < 0 || o >= nsplits || seen[o]) return DA_EINVAL;
    seen[o] = 1;
    ord[k] = o;
  }
  if (desc->q.B * desc->q.S == 0) return DA_OK;
  if (!out) return DA_EINVAL;
  WsLayout w = ws_layout(desc, nsplits);
  if (!ws || ws_bytes < w.total) return DA_EWORKSPACE;
  if (!aligned(ws, 256)) return DA_EALIGN;
  char* base = (char*)ws;
  float* m = (float*)(base + w.m);
  float* m2 = (float*)(base + w.m2);
  int64_t* num = (int64_t*)(base + w.num);
  int64_t* den = (int64_t*)(base + w.den);
  void* kv = base + w.kv;
  const size_t kvb = ws_bytes - w.kv;
  const int64_t rows = desc->q.B * desc->q.H * desc->q.S;
  // pass 1: shard rowmaxes composed by max (a max all-reduce across context-parallel ranks)
  for (int k = 0; k < nsplits; k++) {
    const int s = ord[k];
    if ((e = da_rowmax(desc, lo[s], hi[s], k == 0 ? m : m2, kv, kvb, stream))) return e;
    if (k > 0 && (e = da_compose_max(m, m2, rows, stream))) return e;
  }
  // pass 2: shard digits with the global rowmax, composed by integer add (a sum reduce); the
  // digits already there are this call's own canonical digits, so a row with no key in a shard
  // (causal masking) is left as it is
  for (int k = 0; k < nsplits; k++) {
    const int s = ord[k];
    if ((e = accumulate_range(desc, m, lo[s], hi[s], num, den, k == 0 ? 0 : 1, 1, kv, kvb, stream))) return e;
  }
  return da_finalize(num, den, desc->q.B, desc->q.H, desc->q.S, desc->q.D, out, desc->dev_status, stream);
}

DA_EXPORT int dce_rowmax(const da_matrix* logits, int64_t v_lo, int64_t v_hi, float* m, int32_t* dev_status,
               da_stream_t stream) {
  int e = check_matrix(logits);
  if (e) return e;
  if (v_lo < 0 || v_hi < v_lo || v_hi > logits->cols) return DA_EINVAL;
  if (logits->rows == 0) return DA_OK;
  if (!m) return DA_EINVAL;
  if (!aligned(m, 4)) return DA_EALIGN;
  DceArgs a = make_dce(logits);
  a.v_lo = v_lo; a.v_hi = v_hi; a.m_out = m; a.status = dev_status;
  return launched(launch_dce_rowmax(a, (cudaStream_t)stream));
}

DA_EXPORT int dce_denom_digits(const da_matrix* logits, const float* m, int64_t v_lo, int64_t v_hi, int64_t* den,
                     int add_into, int32_t* dev_status, da_stream_t stream) {
  int e = check_matrix(logits);
  if (e) return e;
  if (v_lo < 0 || v_hi < v_lo || v_hi > logits->cols) return DA_EINVAL;
  if (v_hi - v_lo > ((int64_t)1 << 31)) return DA_EINVAL;
  if (logits->rows == 0) return DA_OK;
  if (!m || !den) return DA_EINVAL;
  if (!aligned(m, 4) || !aligned(den, 8)) return DA_EALIGN;
  DceArgs a = make_dce(logits);
  a.v_lo = v_lo; a.v_hi = v_hi; a.m_in = m; a.den = (long long*)den; a.add_into = add_into ? 1 : 0;
  a.status = dev_status;
  return launched(launch_dce_denom(a, (cudaStream_t)stream));
}

DA_EXPORT int dce_finalize(const int64_t* den, const da_matrix* logits, const int64_t* targets, const float* m, float* loss,
                 double* denom, int32_t* dev_status, da_stream_t stream) {
  int e = check_matrix(logits);
  if (e) return e;
  if (logits->rows == 0) return DA_OK;
  if (!den || !targets || !m || !loss || !denom) return DA_EINVAL;
  if (!aligned(den, 8) || !aligned(targets, 8) || !aligned(m, 4) || !aligned(loss, 4) || !aligned(denom, 8))
    return DA_EALIGN;
  DceArgs a = make_dce(logits);
  a.den = (long long*)den; a.targets = targets; a.m_in = m; a.loss = loss; a.denom = denom; a.status = dev_status;
  return launched(launch_dce_finalize(a, (cudaStream_t)stream));
}

DA_EXPORT int dce_backward(const da_matrix* logits, const int64_t* targets, const float* m, const double* denom,
                           const float* grad, int reduction, void* dlogits, int32_t* dev_status, da_stream_t stream) {
  int e = check_matrix(logits);
  if (e) return e;
  if (reduction < 0 || reduction > 2) return DA_EINVAL;
  if (logits->rows == 0 || logits->cols == 0) return DA_OK;
  if (!targets || !m || !denom || !grad || !dlogits) return DA_EINVAL;
  if (!aligned(targets, 8) || !aligned(m, 4) || !aligned(denom, 8) || !aligned(grad, 4) ||
      !aligned(dlogits, logits->dtype == 0 ? 4 : 2))
    return DA_EALIGN;
  DceArgs a = make_dce(logits);
  a.targets = targets; a.m_in = m; a.denom = (double*)denom; a.status = dev_status;
  return launched(launch_dce_backward(a, grad, reduction, dlogits, (cudaStream_t)stream));
}

DA_EXPORT int dce_finalize_shard(const int64_t* den, const da_matrix* logits, int64_t v_base, int64_t v_total,
                                 const int64_t* targets, const float* m, float* loss, double* denom,
                                 int32_t* dev_status, da_stream_t stream) {
  int e = check_matrix(logits);
  if (e) return e;
  if (v_base < 0 || v_total < 1 || v_base > v_total || logits->cols > v_total - v_base) return DA_EINVAL;
  if (logits->rows == 0) return DA_OK;
  if (!den || !targets || !m || !loss || !denom) return DA_EINVAL;
  if (!aligned(den, 8) || !aligned(targets, 8) || !aligned(m, 4) || !aligned(loss, 4) || !aligned(denom, 8))
    return DA_EALIGN;
  DceArgs a = make_dce(logits);
  a.den = (long long*)den; a.targets = targets; a.m_in = m; a.loss = loss; a.denom = denom; a.status = dev_status;
  a.v_base = v_base; a.v_total = v_total;
  return launched(launch_dce_finalize(a, (cudaStream_t)stream));
}

DA_EXPORT int dce_backward_shard(const da_matrix* logits, int64_t v_base, const int64_t* targets, const float* m,
                                 const double* denom, const float* grad, int reduction, void* dlogits,
                                 int32_t* dev_status, da_stream_t stream) {
  int e = check_matrix(logits);
  if (e) return e;
  if (v_base < 0 || reduction < 0 || reduction > 2) return DA_EINVAL;
  if (logits->rows == 0 || logits->cols == 0) return DA_OK;
  if (!targets || !m || !denom || !grad || !dlogits) return DA_EINVAL;
  if (!aligned(targets, 8) || !aligned(m, 4) || !aligned(denom, 8) || !aligned(grad, 4) ||
      !aligned(dlogits, logits->dtype == 0 ? 4 : 2))
    return DA_EALIGN;
  DceArgs a = make_dce(logits);
  a.targets = targets; a.m_in = m; a.denom = (double*)denom; a.status = dev_status; a.v_base = v_base;
  return launched(launch_dce_backward(a, grad, reduction, dlogits, (cudaStream_t)stream));
}

DA_EXPORT int dce_reduce(const float* loss, int64_t rows, int reduction, float* out, da_stream_t stream) {
  if (rows < 0 || (reduction != 1 && reduction != 2)) return DA_EINVAL;
  if ((!loss && rows > 0) || !out) return DA_EINVAL;
  if (!aligned(loss, 4) || !aligned(out, 4)) return DA_EALIGN;
  return launched(launch_dce_reduce(loss, rows, reduction, out, (cudaStream_t)stream));
}

}  // extern "C"
