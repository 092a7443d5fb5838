// Host-side launchers of the library's kernels (internal to libcpattn).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace cpattn {

// The ring problem one launch solves, after the a2a split of the hierarchical
// mode has been folded into the batch (B = a2a * B_user, heads / a2a, cp / a2a).
struct Ring {
  int B, Hq, Hkv, T, D, cp, zz;
  float scale;
  int bf16;          // 1: bf16 tensors, 0: f32
  int debug_fault;
};

// ---- layout.cu -------------------------------------------------------------
enum PermuteKind { kZigzagFwd = 0, kZigzagInv = 1, kA2AFwd = 2, kA2AInv = 3 };
struct PermuteArgs {
  int kind;
  int B, H, T, D, elt;     // elt = element bytes
  int cp, a2a, zz;         // cp = ranks of the token shards; ring ranks = cp / a2a
};
cudaError_t launch_permute(const PermuteArgs& a, const void* src, void* dst, cudaStream_t st);
// n permutes of one kind over tensors of one descriptor, n_heads[i] heads each
// (a.H is ignored); zigzag permutes of 16-byte rows go out as a single launch.
constexpr int kMaxBatch = 8;
cudaError_t launch_permute_batch(const PermuteArgs& a, int n, const void* const* src,
                                 void* const* dst, const int* n_heads, cudaStream_t st);

// ---- merge.cu --------------------------------------------------------------
// Packed sequences: from the document starts [B][n_docs + 1] (natural positions,
// starts[b][0] = 0, non-decreasing, starts[b][n_docs] = T) the first and last
// position of every position's document, lo/hi [B][T] int32.  Positions are
// clamped into their own document so that every query sees at least itself.
cudaError_t launch_doc_bounds(int B, int T, int n_docs, const int* starts, int* lo, int* hi,
                              cudaStream_t st);
// Packed sequences: (batch row, 128-token tile) entries b * (T/128) + tile in order
// of decreasing work, for query tiles (ord_q) and key tiles (ord_k), B * T/128 each.
cudaError_t launch_doc_order(int B, int T, const int* lo, const int* hi, int* ord_q, int* ord_k,
                             cudaStream_t st);
cudaError_t launch_merge(int64_t rows, int D, const float* oa, const float* la, const float* ob,
                         const float* lb, float* oo, float* lo, cudaStream_t st);
// delta[row] = sum_d dO[row, d] * O[row, d] (float32 accumulation).  When lse2 is
// not null (the tensor-core backward's form) the statistics are stored negated:
// delta[row] = -Delta and lse2[row] = -lse[row] * log2(e).
cudaError_t launch_delta(int64_t rows, int D, int bf16, const void* o, const void* dO,
                         const float* lse, float* delta, float* lse2, cudaStream_t st);

// ---- simt_attn.cu (exact float32 / any-D path) ------------------------------
// partial: q_rank >= 0 selects one rank's queries against kv_rank's chunk and
// writes float32 o/lse of c rows per (b, h); q_rank >= 0 with kv_rank < 0 is the
// all-gather mode (that rank's c rows per (b, h) over every chunk, o in the tensor
// dtype); q_rank < 0 runs the whole ring and writes o in the tensor dtype.
cudaError_t launch_simt_fwd(const Ring& R, int q_rank, int kv_rank, const void* q, const void* k,
                            const void* v, void* o, float* lse, cudaStream_t st,
                            const int* doc_lo = nullptr);
cudaError_t launch_simt_bwd_dq(const Ring& R, const void* q, const void* k, const void* v,
                               const float* lse, const float* delta, const void* dO, void* dq,
                               cudaStream_t st, const int* doc_lo = nullptr);
cudaError_t launch_simt_bwd_dkdv(const Ring& R, const void* q, const void* k, const void* v,
                                 const float* lse, const float* delta, const void* dO, void* dk,
                                 void* dv, cudaStream_t st, const int* doc_hi = nullptr);
// All-gather mode backward of rank q_rank: lse/delta/dO/dq hold the rank's c rows
// per (b, h), q the whole sequence; dk_sum/dv_sum (float32, all T rows) receive
// the rank's share (added when `accumulate`).
cudaError_t launch_simt_allgather_bwd(const Ring& R, int q_rank, const void* q, const void* k,
                                      const void* v, const float* lse, const float* delta,
                                      const void* dO, void* dq, float* dk_sum, float* dv_sum,
                                      int accumulate, cudaStream_t st);

// One ring step of the backward: rank q_rank's rows (lse/delta/dO hold its c rows
// per (b, h)) against the keys of chunk kv_rank; float32 contributions to the
// rank's dQ rows (dq_part, c rows per (b, h)) and to the chunk's dK/dV rows
// (dk_part/dv_part, c rows per (b, g)), overwritten or added when `accumulate`.
cudaError_t launch_simt_partial_bwd(const Ring& R, int q_rank, int kv_rank, const void* q,
                                    const void* k, const void* v, const float* lse,
                                    const float* delta, const void* dO, float* dq_part,
                                    float* dk_part, float* dv_part, int accumulate,
                                    cudaStream_t st);

// ---- tc_fwd.cu / tc_bwd.cu (bf16 tcgen05 path, D in {64, 128}) --------------
bool tc_supported(const Ring& R);
// doc_lo (packed sequences, ring mode only): per batch row and natural position
// the first position of its document, [B][T] int32; nullptr for plain causal.
cudaError_t launch_tc_fwd(const Ring& R, int q_rank, int kv_rank, const void* q, const void* k,
                          const void* v, void* o, float* lse, int* status, cudaStream_t st,
                          const int* doc_lo = nullptr, const int* ord_q = nullptr);
// Work a caller queues on the backward's stream between the dK/dV and the dQ
// kernel (dk and dv are final there): fn(ctx, st).
struct AfterDkdv {
  cudaError_t (*fn)(void* ctx, cudaStream_t st);
  void* ctx;
};
// The dQ kernel run as `parts` launches, part j over the j-th contiguous parts-th of
// every tensor (an independent problem of the same kind), with fn(ctx, st, j)
// queued after launch j, so another stream can take part j's dq while the next
// part computes.  Plain ring problems only; where the problem does not split so,
// one launch is followed by fn for every part in order.
struct AfterDqPart {
  cudaError_t (*fn)(void* ctx, cudaStream_t st, int part);
  void* ctx;
  int parts;
};
// doc_lo / doc_hi (packed sequences): first and last position of each position's
// document, [B][T] int32 each; nullptr for plain causal.  after (optional): see
// AfterDkdv; dq_parts (optional): see AfterDqPart.  dq_claim (optional): one int of
// device memory that the dQ kernel's CTAs claim their items from; given (and with
// neither after nor dq_parts), the dQ kernel is launched on st as a programmatic
// dependent of the dK/dV kernel and overlaps its last CTAs.
cudaError_t launch_tc_bwd(const Ring& R, const void* q, const void* k, const void* v,
                          const float* lse2, const float* delta, const void* dO, void* dq,
                          void* dk, void* dv, int* status, cudaStream_t st,
                          const int* doc_lo = nullptr, const int* doc_hi = nullptr,
                          const int* ord_q = nullptr, const int* ord_k = nullptr,
                          const AfterDkdv* after = nullptr, const AfterDqPart* dq_parts = nullptr,
                          int* dq_claim = nullptr);
// All-gather mode backward of rank q_rank (see launch_simt_allgather_bwd); lse2 /
// delta are the pre-pass statistics of the rank's rows; dq_claim (optional) as for
// launch_tc_bwd.
cudaError_t launch_tc_allgather_bwd(const Ring& R, int q_rank, const void* q, const void* k,
                                    const void* v, const float* lse2, const float* delta,
                                    const void* dO, void* dq, float* dk_sum, float* dv_sum,
                                    int accumulate, int* status, cudaStream_t st,
                                    int* dq_claim = nullptr);

// One ring step of the backward (see launch_simt_partial_bwd); lse2 / delta are the
// pre-pass statistics of the rank's rows.
cudaError_t launch_tc_partial_bwd(const Ring& R, int q_rank, int kv_rank, const void* q,
                                  const void* k, const void* v, const float* lse2,
                                  const float* delta, const void* dO, float* dq_part,
                                  float* dk_part, float* dv_part, int accumulate, int* status,
                                  cudaStream_t st, int* dq_claim = nullptr);

// The register split of the tensor-core kernels (3 warpgroups: one control, two
// math) must fit in what a launch of `kern` allocates; a split that does not fit
// would make setmaxnreg.inc wait forever, so such a launch is refused.
template <typename K>
inline cudaError_t check_register_split(K kern, int threads) {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, kern);
  if (e != cudaSuccess) return e;
  const long need = 128L * kRegsCtl + (long)(threads - 128) * kRegsMath;
  return (long)a.numRegs * threads >= need ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// ---- api.cu: kernel timing hooks -------------------------------------------
void timing_begin(const char* name, cudaStream_t st);
void timing_end(cudaStream_t st);

// Tensor-map encoder (driver entry point fetched through the runtime).
CUresult encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                             uint32_t box_inner, uint32_t box_rows);
// The same for a float32 [rows][inner] tensor.
CUresult encode_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                             uint32_t box_inner, uint32_t box_rows);

}  // namespace cpattn
