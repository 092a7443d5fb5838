// The C ABI of libcpattn: argument validation, dispatch to the kernels, the
// per-device status word, tensor-map encoding and kernel timing.
#include <math.h>
#include <stdio.h>

#include <mutex>
#include <string>
#include <vector>

#include "../../include/cpattn.h"
#include "api_internal.h"
#include "kernels.h"

// Device status word (one per device that loads the library): the first error a
// kernel detects (a bounded wait that ran out) is latched here; cpattn_check
// reads and clears it.
static __device__ int g_cpattn_status;

namespace cpattn {

// ---------------------------------------------------------------------------
// status word address per device
// ---------------------------------------------------------------------------
static std::mutex g_mu;
static int* g_status_ptr[128];

static int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_cpattn_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

// ---------------------------------------------------------------------------
// tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry point)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor [rows][inner], box [box_rows][box_inner], 128-byte swizzle.
CUresult encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                             uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                            uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// ---------------------------------------------------------------------------
// kernel timing
// ---------------------------------------------------------------------------
struct TimingEntry {
  std::string name;
  double total_ms = 0;
  int64_t launches = 0;
};
struct PendingTiming {
  int idx;
  cudaEvent_t a, b;
};
static bool g_timing = false;
static std::vector<TimingEntry> g_entries;
static std::vector<PendingTiming> g_pending;
static thread_local int t_open = -1;

void timing_begin(const char* name, cudaStream_t st) {
  if (!g_timing) return;
  std::lock_guard<std::mutex> lk(g_mu);
  int idx = -1;
  for (size_t i = 0; i < g_entries.size(); ++i)
    if (g_entries[i].name == name) idx = (int)i;
  if (idx < 0) {
    g_entries.push_back(TimingEntry{name, 0.0, 0});
    idx = (int)g_entries.size() - 1;
  }
  PendingTiming p{idx, nullptr, nullptr};
  if (cudaEventCreate(&p.a) != cudaSuccess || cudaEventCreate(&p.b) != cudaSuccess) return;
  cudaEventRecord(p.a, st);
  g_pending.push_back(p);
  t_open = (int)g_pending.size() - 1;
}

void timing_end(cudaStream_t st) {
  if (!g_timing || t_open < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (t_open < (int)g_pending.size()) cudaEventRecord(g_pending[t_open].b, st);
  t_open = -1;
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
static bool aligned16(const void* p) { return p && ((uintptr_t)p % 16 == 0); }

static cpattn_status validate(const cpattn_desc* d, Ring* R) {
  if (!d) return CPATTN_ERR_INVALID_ARG;
  if (d->B <= 0 || d->H_q <= 0 || d->H_kv <= 0 || d->T <= 0 || d->D <= 0 || d->cp <= 0 ||
      d->a2a <= 0)
    return CPATTN_ERR_INVALID_ARG;
  if (d->H_q % d->H_kv || d->cp % d->a2a || d->H_q % d->a2a || d->H_kv % d->a2a)
    return CPATTN_ERR_INVALID_ARG;
  if (d->layout != CPATTN_CONTIGUOUS && d->layout != CPATTN_ZIGZAG) return CPATTN_ERR_INVALID_ARG;
  if (d->dtype != CPATTN_F32 && d->dtype != CPATTN_BF16) return CPATTN_ERR_INVALID_ARG;
  if (!(d->scale > 0.f) || !isfinite(d->scale)) return CPATTN_ERR_INVALID_ARG;
  if (d->causal != 1) return CPATTN_ERR_UNSUPPORTED;
  if (d->D > 128) return CPATTN_ERR_UNSUPPORTED;
  const int p2p = d->cp / d->a2a;
  if (d->T % p2p) return CPATTN_ERR_INVALID_ARG;
  if (d->layout == CPATTN_ZIGZAG && d->T % (2 * p2p)) return CPATTN_ERR_INVALID_ARG;
  const double elems = (double)d->B * d->H_q * d->T * d->D;
  if (elems > 4.0e18 || d->T > (1 << 30)) return CPATTN_ERR_UNSUPPORTED;
  if (R) {
    R->B = d->B * d->a2a;
    R->Hq = d->H_q / d->a2a;
    R->Hkv = d->H_kv / d->a2a;
    R->T = d->T;
    R->D = d->D;
    R->cp = p2p;
    R->zz = d->layout == CPATTN_ZIGZAG;
    R->scale = d->scale;
    R->bf16 = d->dtype == CPATTN_BF16;
    R->debug_fault = d->debug_fault;
  }
  return CPATTN_OK;
}

static cpattn_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

}  // namespace cpattn

using namespace cpattn;

extern "C" {

cpattn_status cpattn_partial_fwd(const cpattn_desc* desc, int q_rank, int kv_rank,
                                 const void* q, const void* k, const void* v, float* o_part,
                                 float* lse_part, void* stream) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if (q_rank < 0 || q_rank >= R.cp || kv_rank < 0 || kv_rank >= R.cp)
    return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part) || !aligned16(lse_part))
    return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  if (R.bf16 && tc_supported(R))
    return from_cuda(launch_tc_fwd(R, q_rank, kv_rank, q, k, v, o_part, lse_part, status_ptr(), st));
  return from_cuda(launch_simt_fwd(R, q_rank, kv_rank, q, k, v, o_part, lse_part, st));
}

cpattn_status cpattn_merge(int64_t rows, int D, const float* o_a, const float* lse_a,
                           const float* o_b, const float* lse_b, float* o_out, float* lse_out,
                           void* stream) {
  if (rows < 0 || D <= 0) return CPATTN_ERR_INVALID_ARG;
  if (rows == 0) return CPATTN_OK;
  if (!aligned16(o_a) || !aligned16(lse_a) || !aligned16(o_b) || !aligned16(lse_b) ||
      !aligned16(o_out) || !aligned16(lse_out))
    return CPATTN_ERR_INVALID_ARG;
  cudaGetLastError();
  return from_cuda(launch_merge(rows, D, o_a, lse_a, o_b, lse_b, o_out, lse_out,
                                (cudaStream_t)stream));
}

cpattn_status cpattn_ring_fwd(const cpattn_desc* desc, const void* q, const void* k,
                              const void* v, void* o, float* lse, void* stream) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  if (R.bf16 && tc_supported(R))
    return from_cuda(launch_tc_fwd(R, -1, -1, q, k, v, o, lse, status_ptr(), st));
  return from_cuda(launch_simt_fwd(R, -1, -1, q, k, v, o, lse, st));
}

// Workspace: Delta (float32 per query row), then the LSE in base 2 (float32 per
// query row), then the dQ kernel's item counter (kClaimBytes), each section
// 256-byte aligned.
static size_t ws_section(const cpattn_desc* desc) {
  const size_t rows = (size_t)desc->B * desc->H_q * desc->T;
  return (rows * sizeof(float) + 255) / 256 * 256;
}
static constexpr size_t kClaimBytes = 256;

size_t cpattn_ring_bwd_workspace(const cpattn_desc* desc) {
  if (validate(desc, nullptr) != CPATTN_OK) return 0;
  return 2 * ws_section(desc) + kClaimBytes;
}

cpattn_status cpattn_ring_bwd(const cpattn_desc* desc, const void* q, const void* k,
                              const void* v, const void* o, const float* lse, const void* dO,
                              void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                              void* stream) {
  return cpattn::ring_bwd_after_dkdv(desc, q, k, v, o, lse, dO, dq, dk, dv, workspace, ws_bytes,
                                     stream, nullptr, nullptr);
}

}  // extern "C"

cpattn_status cpattn::ring_bwd_after_dkdv(const cpattn_desc* desc, const void* q, const void* k,
                                          const void* v, const void* o, const float* lse,
                                          const void* dO, void* dq, void* dk, void* dv,
                                          void* workspace, size_t ws_bytes, void* stream,
                                          const AfterDkdv* after, const AfterDqPart* dq_parts) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(workspace))
    return CPATTN_ERR_INVALID_ARG;
  if (ws_bytes < cpattn_ring_bwd_workspace(desc)) return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  float* delta = static_cast<float*>(workspace);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws_section(desc));
  int* claim = reinterpret_cast<int*>(static_cast<char*>(workspace) + 2 * ws_section(desc));
  const int64_t rows = (int64_t)R.B * R.Hq * R.T;
  const bool tc = R.bf16 && tc_supported(R);
  cudaError_t e = launch_delta(rows, R.D, R.bf16, o, dO, lse, delta, tc ? lse2 : nullptr, st);
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  if (tc)
    return from_cuda(launch_tc_bwd(R, q, k, v, lse2, delta, dO, dq, dk, dv, status_ptr(), st,
                                   nullptr, nullptr, nullptr, nullptr, after, dq_parts, claim));
  e = launch_simt_bwd_dq(R, q, k, v, lse, delta, dO, dq, st);
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  e = launch_simt_bwd_dkdv(R, q, k, v, lse, delta, dO, dk, dv, st);
  if (e == cudaSuccess && after != nullptr && after->fn != nullptr) e = after->fn(after->ctx, st);
  if (dq_parts != nullptr && dq_parts->fn != nullptr)
    for (int j = 0; j < dq_parts->parts && e == cudaSuccess; ++j)
      e = dq_parts->fn(dq_parts->ctx, st, j);
  return from_cuda(e);
}

extern "C" {

// ---------------------------------------------------------------------------
// packed sequences
// ---------------------------------------------------------------------------
// Workspace: lo, hi (int32 per batch row and position), the work orders of the
// query and key tiles (int32 per batch row and 128-token tile), then the
// backward's statistics as for cpattn_ring_bwd; each section 256-byte aligned.
static size_t doc_section(const cpattn_desc* desc) {
  return ((size_t)desc->B * desc->T * sizeof(int) + 255) / 256 * 256;
}
static size_t order_section(const cpattn_desc* desc) {
  return ((size_t)desc->B * (desc->T / 128) * sizeof(int) + 255) / 256 * 256;
}
static size_t packed_stats_offset(const cpattn_desc* desc) {
  return 2 * doc_section(desc) + 2 * order_section(desc);
}

size_t cpattn_packed_workspace(const cpattn_desc* desc) {
  if (validate(desc, nullptr) != CPATTN_OK || desc->a2a != 1) return 0;
  return packed_stats_offset(desc) + cpattn_ring_bwd_workspace(desc);
}

// lo, hi and (tensor-core path only) the tile work orders of a packed call
struct PackedTables {
  int *lo, *hi, *ord_q, *ord_k;
};
static cudaError_t packed_tables(const cpattn_desc* desc, const Ring& R, const int32_t* starts,
                                 int n_docs, void* workspace, bool tc, cudaStream_t st,
                                 PackedTables* t) {
  char* w = static_cast<char*>(workspace);
  t->lo = reinterpret_cast<int*>(w);
  t->hi = reinterpret_cast<int*>(w + doc_section(desc));
  t->ord_q = reinterpret_cast<int*>(w + 2 * doc_section(desc));
  t->ord_k = reinterpret_cast<int*>(w + 2 * doc_section(desc) + order_section(desc));
  cudaError_t e = launch_doc_bounds(R.B, R.T, n_docs, starts, t->lo, t->hi, st);
  if (e != cudaSuccess || !tc) return e;
  return launch_doc_order(R.B, R.T, t->lo, t->hi, t->ord_q, t->ord_k, st);
}

static cpattn_status packed_args(const cpattn_desc* desc, const int32_t* starts, int n_docs,
                                 void* workspace, size_t ws_bytes) {
  if (desc->a2a != 1) return CPATTN_ERR_UNSUPPORTED;
  if (n_docs < 1 || !starts || ((uintptr_t)starts & 3u)) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(workspace) || ws_bytes < cpattn_packed_workspace(desc))
    return CPATTN_ERR_INVALID_ARG;
  return CPATTN_OK;
}

cpattn_status cpattn_ring_fwd_packed(const cpattn_desc* desc, const int32_t* starts, int n_docs,
                                     const void* q, const void* k, const void* v, void* o,
                                     float* lse, void* workspace, size_t ws_bytes, void* stream) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if ((s = packed_args(desc, starts, n_docs, workspace, ws_bytes)) != CPATTN_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  const bool tc = R.bf16 && tc_supported(R);
  PackedTables t;
  if (packed_tables(desc, R, starts, n_docs, workspace, tc, st, &t) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  if (tc)
    return from_cuda(
        launch_tc_fwd(R, -1, -1, q, k, v, o, lse, status_ptr(), st, t.lo, t.ord_q));
  return from_cuda(launch_simt_fwd(R, -1, -1, q, k, v, o, lse, st, t.lo));
}

cpattn_status cpattn_ring_bwd_packed(const cpattn_desc* desc, const int32_t* starts, int n_docs,
                                     const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dO, void* dq, void* dk,
                                     void* dv, void* workspace, size_t ws_bytes, void* stream) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if ((s = packed_args(desc, starts, n_docs, workspace, ws_bytes)) != CPATTN_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  char* stats = static_cast<char*>(workspace) + packed_stats_offset(desc);
  float* delta = reinterpret_cast<float*>(stats);
  float* lse2 = reinterpret_cast<float*>(stats + ws_section(desc));
  int* claim = reinterpret_cast<int*>(stats + 2 * ws_section(desc));
  const bool tc = R.bf16 && tc_supported(R);
  PackedTables t;
  if (packed_tables(desc, R, starts, n_docs, workspace, tc, st, &t) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  const int* lo = t.lo;
  const int* hi = t.hi;
  const int64_t rows = (int64_t)R.B * R.Hq * R.T;
  cudaError_t e = launch_delta(rows, R.D, R.bf16, o, dO, lse, delta, tc ? lse2 : nullptr, st);
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  if (tc)
    return from_cuda(
        launch_tc_bwd(R, q, k, v, lse2, delta, dO, dq, dk, dv, status_ptr(), st, lo, hi, t.ord_q,
                      t.ord_k, nullptr, nullptr, claim));
  e = launch_simt_bwd_dq(R, q, k, v, lse, delta, dO, dq, st, lo);
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  return from_cuda(launch_simt_bwd_dkdv(R, q, k, v, lse, delta, dO, dk, dv, st, hi));
}

// ---------------------------------------------------------------------------
// all-gather mode
// ---------------------------------------------------------------------------
cpattn_status cpattn_allgather_fwd(const cpattn_desc* desc, int q_rank, const void* q,
                                   const void* k, const void* v, void* o, float* lse,
                                   void* stream) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if (q_rank < 0 || q_rank >= R.cp) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  if (R.bf16 && tc_supported(R))
    return from_cuda(launch_tc_fwd(R, q_rank, -1, q, k, v, o, lse, status_ptr(), st));
  return from_cuda(launch_simt_fwd(R, q_rank, -1, q, k, v, o, lse, st));
}

// Workspace: Delta, then the LSE in base 2, of the rank's rows (float32 each),
// each section 256-byte aligned.
static size_t ag_section(const Ring& R) {
  const size_t rows = (size_t)R.B * R.Hq * (R.T / R.cp);
  return (rows * sizeof(float) + 255) / 256 * 256;
}

size_t cpattn_allgather_bwd_workspace(const cpattn_desc* desc) {
  Ring R;
  if (validate(desc, &R) != CPATTN_OK) return 0;
  return 2 * ag_section(R) + kClaimBytes;  // Delta, LSE in base 2, the dQ item counter
}

cpattn_status cpattn_allgather_bwd(const cpattn_desc* desc, int q_rank, const void* q,
                                   const void* k, const void* v, const void* o,
                                   const float* lse, const void* dO, void* dq, float* dk_sum,
                                   float* dv_sum, int accumulate, void* workspace,
                                   size_t ws_bytes, void* stream) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if (q_rank < 0 || q_rank >= R.cp || (accumulate != 0 && accumulate != 1))
    return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk_sum) || !aligned16(dv_sum) ||
      !aligned16(workspace))
    return CPATTN_ERR_INVALID_ARG;
  if (ws_bytes < cpattn_allgather_bwd_workspace(desc)) return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  float* delta = static_cast<float*>(workspace);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + ag_section(R));
  int* claim = reinterpret_cast<int*>(static_cast<char*>(workspace) + 2 * ag_section(R));
  const int64_t rows = (int64_t)R.B * R.Hq * (R.T / R.cp);
  const bool tc = R.bf16 && tc_supported(R);
  cudaError_t e = launch_delta(rows, R.D, R.bf16, o, dO, lse, delta, tc ? lse2 : nullptr, st);
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  if (tc)
    return from_cuda(launch_tc_allgather_bwd(R, q_rank, q, k, v, lse2, delta, dO, dq, dk_sum,
                                             dv_sum, accumulate, status_ptr(), st, claim));
  return from_cuda(launch_simt_allgather_bwd(R, q_rank, q, k, v, lse, delta, dO, dq, dk_sum,
                                             dv_sum, accumulate, st));
}

// ---------------------------------------------------------------------------
// one ring step of the backward
// ---------------------------------------------------------------------------
// Workspace: two float32 sections of the rank's rows, each 256-byte aligned.  The
// tensor-core path keeps -Delta and -LSE log2(e) there, the SIMT path Delta and
// the LSE (natural log).
size_t cpattn_partial_bwd_workspace(const cpattn_desc* desc) {
  return cpattn_allgather_bwd_workspace(desc);
}

cpattn_status cpattn_partial_bwd_stats(const cpattn_desc* desc, const void* o, const float* lse,
                                       const void* dO, void* workspace, size_t ws_bytes,
                                       void* stream) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if (!aligned16(o) || !aligned16(lse) || !aligned16(dO) || !aligned16(workspace))
    return CPATTN_ERR_INVALID_ARG;
  if (ws_bytes < cpattn_partial_bwd_workspace(desc)) return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  float* delta = static_cast<float*>(workspace);
  float* sec1 = reinterpret_cast<float*>(static_cast<char*>(workspace) + ag_section(R));
  const int64_t rows = (int64_t)R.B * R.Hq * (R.T / R.cp);
  const bool tc = R.bf16 && tc_supported(R);
  cudaError_t e = launch_delta(rows, R.D, R.bf16, o, dO, lse, delta, tc ? sec1 : nullptr, st);
  if (e == cudaSuccess && !tc)
    e = cudaMemcpyAsync(sec1, lse, rows * sizeof(float), cudaMemcpyDeviceToDevice, st);
  return from_cuda(e);
}

cpattn_status cpattn_partial_bwd(const cpattn_desc* desc, int q_rank, int kv_rank,
                                 const void* q, const void* k, const void* v, const void* dO,
                                 float* dq_part, float* dk_part, float* dv_part, int accumulate,
                                 void* workspace, size_t ws_bytes, void* stream) {
  Ring R;
  cpattn_status s = validate(desc, &R);
  if (s != CPATTN_OK) return s;
  if (q_rank < 0 || q_rank >= R.cp || kv_rank < 0 || kv_rank >= R.cp ||
      (accumulate != 0 && accumulate != 1))
    return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq_part) ||
      !aligned16(dk_part) || !aligned16(dv_part) || !aligned16(workspace))
    return CPATTN_ERR_INVALID_ARG;
  if (ws_bytes < cpattn_partial_bwd_workspace(desc)) return CPATTN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  const float* delta = static_cast<const float*>(workspace);
  const float* sec1 =
      reinterpret_cast<const float*>(static_cast<const char*>(workspace) + ag_section(R));
  int* claim = reinterpret_cast<int*>(static_cast<char*>(workspace) + 2 * ag_section(R));
  if (R.bf16 && tc_supported(R))
    return from_cuda(launch_tc_partial_bwd(R, q_rank, kv_rank, q, k, v, sec1, delta, dO, dq_part,
                                           dk_part, dv_part, accumulate, status_ptr(), st, claim));
  return from_cuda(launch_simt_partial_bwd(R, q_rank, kv_rank, q, k, v, sec1, delta, dO, dq_part,
                                           dk_part, dv_part, accumulate, st));
}

// Checks of one tensor of a permute; fills the arguments shared by every tensor.
static cpattn_status permute_args(int permute, const cpattn_desc* desc, const void* src,
                                  const void* dst, int n_heads, PermuteArgs* out) {
  cpattn_status s = validate(desc, nullptr);
  if (s != CPATTN_OK) return s;
  if (permute < CPATTN_ZIGZAG_FWD || permute > CPATTN_A2A_INV || n_heads <= 0)
    return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst) || src == dst) return CPATTN_ERR_INVALID_ARG;
  if (permute >= CPATTN_A2A_FWD) {
    if (n_heads % desc->a2a || desc->T % desc->cp) return CPATTN_ERR_INVALID_ARG;
    if (desc->layout == CPATTN_ZIGZAG && desc->T % (2 * desc->cp)) return CPATTN_ERR_INVALID_ARG;
  }
  PermuteArgs& a = *out;
  a.kind = permute;
  a.B = desc->B;
  a.H = n_heads;
  a.T = desc->T;
  a.D = desc->D;
  a.elt = desc->dtype == CPATTN_BF16 ? 2 : 4;
  a.cp = desc->cp;
  a.a2a = desc->a2a;
  a.zz = desc->layout == CPATTN_ZIGZAG;
  return CPATTN_OK;
}

cpattn_status cpattn_layout_batch(int permute, const cpattn_desc* desc, int n,
                                  const void* const* src, void* const* dst, const int* n_heads,
                                  void* stream) {
  if (n < 1 || n > kMaxBatch || !src || !dst || !n_heads) return CPATTN_ERR_INVALID_ARG;
  PermuteArgs a;
  for (int i = 0; i < n; ++i) {
    cpattn_status s = permute_args(permute, desc, src[i], dst[i], n_heads[i], &a);
    if (s != CPATTN_OK) return s;
  }
  cudaGetLastError();
  return from_cuda(launch_permute_batch(a, n, src, dst, n_heads, (cudaStream_t)stream));
}

cpattn_status cpattn_layout(int permute, const cpattn_desc* desc, const void* src, void* dst,
                            int n_heads, void* stream) {
  PermuteArgs a;
  cpattn_status s = permute_args(permute, desc, src, dst, n_heads, &a);
  if (s != CPATTN_OK) return s;
  cudaGetLastError();
  return from_cuda(launch_permute(a, src, dst, (cudaStream_t)stream));
}

cpattn_status cpattn_check(void* stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CPATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_cpattn_status, sizeof(int)) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  if (v != 0) {
    int zero = 0;
    if (cudaMemcpyToSymbol(g_cpattn_status, &zero, sizeof(int)) != cudaSuccess)
      return CPATTN_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return CPATTN_ERR_CUDA;
  return v == 0 ? CPATTN_OK : (cpattn_status)v;
}

const char* cpattn_status_string(cpattn_status status) {
  switch (status) {
    case CPATTN_OK: return "ok";
    case CPATTN_ERR_INVALID_ARG: return "invalid argument";
    case CPATTN_ERR_UNSUPPORTED: return "unsupported shape or option";
    case CPATTN_ERR_CUDA: return "CUDA error";
    case CPATTN_ERR_TIMEOUT: return "device wait timed out";
    case CPATTN_ERR_BOUNDS: return "device bounds check failed (debug build)";
    default: return "unknown status";
  }
}

cpattn_status cpattn_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timing = on != 0;
  return CPATTN_OK;
}

cpattn_status cpattn_timing_collect(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  cpattn_status s = CPATTN_OK;
  for (auto& p : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.b) == cudaSuccess && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      g_entries[p.idx].total_ms += ms;
      g_entries[p.idx].launches += 1;
    } else {
      s = CPATTN_ERR_CUDA;
    }
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  g_pending.clear();
  return s;
}

int cpattn_timing_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return (int)g_entries.size();
}

cpattn_status cpattn_timing_get(int index, const char** name, double* total_ms,
                                int64_t* launches) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (index < 0 || index >= (int)g_entries.size()) return CPATTN_ERR_INVALID_ARG;
  if (name) *name = g_entries[index].name.c_str();
  if (total_ms) *total_ms = g_entries[index].total_ms;
  if (launches) *launches = g_entries[index].launches;
  return CPATTN_OK;
}

cpattn_status cpattn_timing_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& p : g_pending) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  g_pending.clear();
  g_entries.clear();
  return CPATTN_OK;
}

}  // extern "C"
