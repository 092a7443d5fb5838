// cpattn_ring_bwd_noalloc: the ring backward for callers that cannot allocate
// device memory.  Some callers own no allocator at the point where they run the
// backward: plugins of an inference or training engine that may only enqueue
// work into buffers the engine handed them, programs that reserve all device
// memory up front and forbid allocation during a step, and code with a fixed
// memory budget.  cpattn_ring_bwd needs a workspace from its caller; this entry
// point instead uses a scratch array compiled into the library.
//
// The scratch is a file-scope __device__ array: every GPU that loads the library
// holds it (kNoAllocScratchBytes) until the process exits.  In host code its name
// is only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the first
// call made there; that first call should therefore come before any stream
// capture.  All calls on a device share the array and it keeps the last call's
// contents; the backward overwrites every word it reads before reading it, so
// nothing needs clearing, but two calls that overlap on the GPU (different
// streams without ordering between them) race on it.
#include <mutex>

#include "../../include/cpattn.h"
#include "kernels.h"

// Scratch size: the float32 per-query-row statistics of the backward for up to
// 2,097,152 query rows (B * H_q * T), two 8 MiB sections, and the 256 bytes of the
// dQ kernel's item counter.
static constexpr size_t kNoAllocScratchBytes = (size_t(16) << 20) + 256;

static __device__ __align__(256) float g_bwd_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_addr[128];

// Device address of g_bwd_scratch on the current device (set up on first use).
cpattn_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return CPATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
      return CPATTN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CPATTN_OK;
}

}  // namespace

extern "C" cpattn_status cpattn_ring_bwd_noalloc(const cpattn_desc* desc, const void* q,
                                                 const void* k, const void* v, const void* o,
                                                 const float* lse, const void* dO, void* dq,
                                                 void* dk, void* dv, void* stream) {
  const size_t need = cpattn_ring_bwd_workspace(desc);
  if (need == 0)  // the descriptor is not valid: report exactly what the backward reports
    return cpattn_ring_bwd(desc, q, k, v, o, lse, dO, dq, dk, dv, nullptr, 0, stream);
  if (need > kNoAllocScratchBytes) return CPATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const cpattn_status s = scratch_address(&scratch);
  if (s != CPATTN_OK) return s;
  return cpattn_ring_bwd(desc, q, k, v, o, lse, dO, dq, dk, dv, scratch, kNoAllocScratchBytes,
                         stream);
}
