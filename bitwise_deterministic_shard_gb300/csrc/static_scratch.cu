// dce_forward_static: the cross-entropy forward for callers that cannot allocate device
// memory (see include/detattn.h).  Its intermediates (the per-token rowmax and the six
// denominator digits) live in one file-scope device array instead of caller memory.
#include <mutex>

#include "../../include/detattn.h"
#include "attn_kernels.h"

namespace {

constexpr int64_t kRows = DA_STATIC_MAX_ROWS;
constexpr size_t kDenBytes = sizeof(long long) * DA_DEN_NDIG * kRows;   // digits first: 8-byte aligned
constexpr size_t kBytes = kDenBytes + sizeof(float) * kRows;

// One copy per device that loads the library, held until the process exits.  In host code
// this name is only a host-side stand-in: kernels get the device address from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_dce_scratch[kBytes];

constexpr int kMaxDevices = 64;
void* g_addr[kMaxDevices] = {};
std::mutex g_lock;

// Device address of the scratch on the current device, looked up once per device.
void* scratch_address(int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = DA_ECUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(g_lock);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dce_scratch) != cudaSuccess || !p) {
      *err = DA_ECUDA;
      return nullptr;
    }
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int dce_forward_static(const da_matrix* logits,
                                                                         const int64_t* targets, float* loss,
                                                                         double* denom, int32_t* dev_status,
                                                                         da_stream_t stream) {
  if (!logits) return DA_EINVAL;
  if (logits->dtype != DA_F32 && logits->dtype != DA_BF16) return DA_EDTYPE;
  if (logits->rows < 0 || logits->cols < 1 || logits->row_stride < logits->cols) return DA_ESHAPE;
  if (logits->rows > kRows) return DA_EWORKSPACE;   // beyond the static scratch
  if (logits->cols > ((int64_t)1 << 31)) return DA_EINVAL;
  if (logits->rows == 0) return DA_OK;
  if (!logits->ptr || !targets || !loss || !denom) return DA_EINVAL;
  const size_t es = logits->dtype == DA_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(logits->ptr) % es || reinterpret_cast<uintptr_t>(targets) % 8 ||
      reinterpret_cast<uintptr_t>(loss) % 4 || reinterpret_cast<uintptr_t>(denom) % 8)
    return DA_EALIGN;
  int err = DA_OK;
  unsigned char* base = static_cast<unsigned char*>(scratch_address(&err));
  if (!base) return err;
  long long* den = reinterpret_cast<long long*>(base);
  float* m = reinterpret_cast<float*>(base + kDenBytes);

  detattn::DceArgs a;
  a.x = logits->ptr;
  a.dtype = logits->dtype;
  a.N = logits->rows;
  a.V = logits->cols;
  a.rs = logits->row_stride;
  a.v_lo = 0;
  a.v_hi = logits->cols;
  a.v_base = 0;
  a.v_total = logits->cols;
  a.m_in = m;
  a.m_out = m;
  a.den = den;
  a.add_into = 0;   // the digit kernel overwrites every digit it later reads: nothing to clear
  a.targets = targets;
  a.loss = loss;
  a.denom = denom;
  a.status = dev_status;
  cudaStream_t st = (cudaStream_t)stream;
  if (detattn::launch_dce_rowmax(a, st) != cudaSuccess) return DA_ECUDA;
  if (detattn::launch_dce_denom(a, st) != cudaSuccess) return DA_ECUDA;
  if (detattn::launch_dce_finalize(a, st) != cudaSuccess) return DA_ECUDA;
  return DA_OK;
}
