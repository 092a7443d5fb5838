// Entry points shared by the C ABI's translation units (internal to libcpattn).
#pragma once

#include <cuda_runtime.h>

#include "../../include/cpattn.h"
#include "kernels.h"

namespace cpattn {

// cpattn_ring_bwd with optional work queued on its stream once dk and dv are final
// (between the dK/dV and the dQ kernel on the tensor-core path, after both on the
// exact path, which runs dQ first), and optionally the dQ kernel run in parts with
// work queued after each (see AfterDqPart; on the exact path all parts' work comes
// after both kernels).
cpattn_status ring_bwd_after_dkdv(const cpattn_desc* desc, const void* q, const void* k,
                                  const void* v, const void* o, const float* lse, const void* dO,
                                  void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                  void* stream, const AfterDkdv* after,
                                  const AfterDqPart* dq_parts);

}  // namespace cpattn
