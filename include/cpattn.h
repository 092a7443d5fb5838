/*
 * cpattn — causal blockwise ring attention for one GB300 (sm_103a), C ABI.
 *
 * The operation (tutorial "上下文并行", section "朴素 Ring Attention"; pull request
 * "Feat: Context Parallel" #181, mode table row "p2p"): the sequence of T tokens
 * is split over cp context-parallel ranks; each rank's query chunk attends to one
 * key/value chunk per ring step (rank r holds the K/V of rank (r - i) mod cp at
 * step i) with the causal mask taken from GLOBAL token positions, and the
 * per-step partial results are merged by the single-pass online softmax
 * (running max and sum, carried as (O, LSE)).  The backward pass recomputes the
 * probabilities and returns dQ and, for every K/V chunk, the dK/dV its owner
 * receives.  On one GPU the ranks are chunk indices inside one kernel launch;
 * nothing is exchanged between GPUs.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Tensors are row-major and contiguous, D fastest:
 *   q, o, dq, dO : [B, H_q, T, D]        k, v, dk, dv : [B, H_kv, T, D]
 *   lse          : [B, H_q, T] float32, natural logarithm
 * The token axis T is in LAYOUT ORDER: rank r holds slots [r*c, (r+1)*c),
 * c = T / cp.  With CPATTN_CONTIGUOUS, slot t is natural position t.  With
 * CPATTN_ZIGZAG (tutorial, section "Zig-Zag Ring Attention") the sequence is cut
 * into 2*cp chunks of c/2 tokens and rank r holds chunk r followed by chunk
 * 2cp-1-r.  cpattn_layout converts between natural and layout order.
 * Query head h uses key/value head h / (H_q / H_kv): the H_q heads form H_kv
 * groups of n_rep = H_q / H_kv consecutive heads (the grouped-query view of the
 * pull request's review thread on RepeatKVHeads, resolved here as an index map;
 * no repeated K/V copy is made).  dK, dV sum over the heads of a group.
 * With a2a > 1 (the hierarchical "a2a+p2p" mode) q/k/v/o/lse and the gradients
 * are the head-sharded tensors that cpattn_layout(CPATTN_A2A_FWD) produces,
 * [a2a][B][H/a2a][T][D], and the ring runs over p2p = cp / a2a ranks inside each
 * of the a2a slices.
 *
 * dtype CPATTN_BF16: q/k/v/o/dO/dq/dk/dv are bfloat16, all accumulation is
 * float32, probabilities are rounded to bf16 only as an MMA operand and O is
 * rounded only after the division by the softmax sum.  dtype CPATTN_F32: every
 * tensor is float32 and every step runs in float32.
 *
 * Ownership: the caller allocates and owns every buffer; the library allocates
 * no device memory in any call.  Every call is asynchronous on `stream` (a
 * cudaStream_t passed as void*; NULL is the legacy default stream) and returns
 * after enqueueing.  Pointers are device pointers unless stated otherwise and
 * must be 16-byte aligned.
 *
 * Errors: invalid arguments are reported synchronously, before anything is
 * enqueued (CPATTN_ERR_INVALID_ARG; CPATTN_ERR_UNSUPPORTED for shapes outside the
 * implemented set).  Launch failures return CPATTN_ERR_CUDA.  Errors detected on
 * the device (a bounded wait that ran out; in a CPATTN_DEBUG build also a failed
 * bounds check) are latched in a per-device status word and reported by
 * cpattn_check.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cpattn_status {
  CPATTN_OK = 0,
  CPATTN_ERR_INVALID_ARG = 1,
  CPATTN_ERR_UNSUPPORTED = 2,
  CPATTN_ERR_CUDA = 3,
  CPATTN_ERR_TIMEOUT = 4,
  CPATTN_ERR_BOUNDS = 5  /* only from a library built with CPATTN_DEBUG: a kernel's
                            bounds check on a computed tensor row failed, and the
                            access was skipped */
} cpattn_status;

typedef enum cpattn_dtype { CPATTN_F32 = 0, CPATTN_BF16 = 1 } cpattn_dtype;

typedef enum cpattn_seq_layout { CPATTN_CONTIGUOUS = 0, CPATTN_ZIGZAG = 1 } cpattn_seq_layout;

typedef enum cpattn_permute {
  CPATTN_ZIGZAG_FWD = 0, /* natural order -> layout order (desc.layout over the ring's ranks) */
  CPATTN_ZIGZAG_INV = 1, /* layout order -> natural order */
  CPATTN_A2A_FWD = 2,    /* token-sharded [cp][B][T/cp][H][D] -> head-sharded [a2a][B][H/a2a][T][D] */
  CPATTN_A2A_INV = 3     /* head-sharded -> token-sharded */
} cpattn_permute;

/* Problem descriptor.  Integers are int32; layout and dtype hold the enum values. */
typedef struct cpattn_desc {
  int32_t B;           /* batch */
  int32_t H_q;         /* query heads (a multiple of H_kv) */
  int32_t H_kv;        /* key/value heads */
  int32_t T;           /* tokens per sequence */
  int32_t D;           /* head dimension (<= 128; the bf16 tensor-core path takes 64 or 128) */
  int32_t cp;          /* context-parallel ranks emulated in the launch */
  int32_t a2a;         /* all-to-all group size of the hierarchical mode; 1 = plain ring */
  int32_t layout;      /* cpattn_seq_layout */
  int32_t dtype;       /* cpattn_dtype */
  float scale;         /* softmax scale, > 0 (1/sqrt(D) for standard attention) */
  int32_t causal;      /* must be 1: the pages define causal self-attention only */
  int32_t debug_fault; /* 0.  Test hook of the bounded waits: 1 makes the tensor-core
                          forward, 2 the backward's dK/dV kernel and 3 its dQ kernel
                          withhold one load, so that the waits on it run out
                          (CPATTN_ERR_TIMEOUT via cpattn_check, within about 50 ms;
                          any non-zero value shortens every bounded wait of the
                          tensor-core kernels to 50 ms). */
} cpattn_desc;

/*
 * One ring step's partial result: the queries of rank q_rank against the K/V
 * chunk of rank kv_rank, causal mask from global positions (tutorial, section
 * "朴素 Ring Attention": partial = Softmax(Q_i K^T / sqrt(d)) V for the block
 * held at that step).
 *   q, k, v   : full layout-order tensors (see above), dtype desc->dtype
 *   o_part    : [B', H_q', c, D] float32, normalised within the chunk
 *   lse_part  : [B', H_q', c] float32; a row that sees no key of the chunk gets
 *               o = 0 and lse = -inf (the identity of cpattn_merge)
 * (B' = a2a*B, H_q' = H_q/a2a, c = T/(cp/a2a); ranks index the p2p ring.)
 * Errors: rank outside [0, cp/a2a) -> CPATTN_ERR_INVALID_ARG.
 */
cpattn_status cpattn_partial_fwd(const cpattn_desc* desc, int q_rank, int kv_rank,
                                 const void* q, const void* k, const void* v,
                                 float* o_part, float* lse_part, void* stream);

/* Bytes of device workspace that holds one rank's row statistics for
 * cpattn_partial_bwd (float32, two values per query row of the rank) and its
 * 256-byte work counter: the size of cpattn_allgather_bwd's workspace. */
size_t cpattn_partial_bwd_workspace(const cpattn_desc* desc);

/*
 * The row statistics of a rank's backward ring steps, computed once per rank and
 * backward pass (the backward's pre-pass, Delta = rowsum(dO * O), with the LSE in
 * the form the kernels read), into `workspace`; every cpattn_partial_bwd of that
 * rank reads them, so the pre-pass is not repeated at each of its cp steps.
 *   o, lse, dO : the rank's rows of the forward's output, of its LSE (the whole
 *                forward's, every step merged) and of the upstream gradient:
 *                [B', H_q', c, D] dtype, [B', H_q', c] float32, [B', H_q', c, D]
 *   workspace  : at least cpattn_partial_bwd_workspace(desc) bytes (smaller ->
 *                CPATTN_ERR_INVALID_ARG)
 * Errors as cpattn_ring_bwd.
 */
cpattn_status cpattn_partial_bwd_stats(const cpattn_desc* desc, const void* o, const float* lse,
                                       const void* dO, void* workspace, size_t ws_bytes,
                                       void* stream);

/*
 * One ring step of the backward pass (tutorial "上下文并行", section "朴素 Ring
 * Attention": at step i rank r holds the K/V chunk of rank s = (r - i) mod cp and
 * recomputes that step's probabilities from the saved statistics; pull request
 * #181, mode table row "p2p": each chunk's K/V gradient travels the ring with the
 * chunk and arrives back at its owner).  The gradient contributions of rank
 * q_rank's queries against the K/V chunk of rank kv_rank:
 *   q, k, v     : full layout-order tensors (as cpattn_partial_fwd: only q_rank's
 *                 query slots and kv_rank's key slots are read)
 *   dO          : rank q_rank's rows of the upstream gradient, [B', H_q', c, D]
 *   workspace   : the rank's statistics, as cpattn_partial_bwd_stats left them for
 *                 the same rank's o, lse and dO (read only), and after them a
 *                 256-byte work counter that the call writes: the step's dQ kernel
 *                 overlaps the end of its dK/dV kernel, as in cpattn_ring_bwd.
 *                 Calls that share a workspace must be ordered (one stream).
 *   dq_part     : [B', H_q', c, D] float32, the step's dQ contribution to the
 *                 rank's rows
 *   dk_part, dv_part : [B', H_kv', c, D] float32, the step's dK / dV contribution
 *                 to chunk kv_rank's rows (slot order within the chunk)
 *   accumulate  : 0 overwrites dq_part, dk_part and dv_part; 1 adds to them
 *   ws_bytes    : at least cpattn_partial_bwd_workspace(desc) (smaller ->
 *                 CPATTN_ERR_INVALID_ARG)
 * Summed over the steps -- dq_part of rank r over every kv_rank, dk_part/dv_part
 * of chunk s over every q_rank -- the contributions give cpattn_ring_bwd's dq
 * (rank r's rows) and dk/dv (chunk s's rows), in float32.  A pair with no
 * visible (query, key) pair contributes zeros.  (B', H_q', H_kv' = H_kv/a2a, c
 * as for cpattn_partial_fwd.)
 * Errors: a rank outside [0, cp/a2a) or accumulate not 0/1 ->
 * CPATTN_ERR_INVALID_ARG; others as cpattn_ring_bwd.
 */
cpattn_status cpattn_partial_bwd(const cpattn_desc* desc, int q_rank, int kv_rank,
                                 const void* q, const void* k, const void* v, const void* dO,
                                 float* dq_part, float* dk_part, float* dv_part, int accumulate,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * Online-softmax merge of two partial results over disjoint key sets (tutorial,
 * section "朴素 Ring Attention": the block order does not matter as long as the
 * current O, max and sum are carried; section "Zig-Zag Ring Attention": the
 * softmax_lse update).  For each of `rows` rows of D floats:
 *   lse = ln(e^lse_a + e^lse_b),  o = e^(lse_a-lse) o_a + e^(lse_b-lse) o_b,
 * evaluated max-shifted; an empty operand (lse = -inf) is the identity and two
 * empty operands give (0, -inf), never NaN.  All buffers are float32;
 * o_out/lse_out may alias o_a/lse_a (or o_b/lse_b) exactly.
 */
cpattn_status cpattn_merge(int64_t rows, int D, const float* o_a, const float* lse_a,
                           const float* o_b, const float* lse_b, float* o_out,
                           float* lse_out, void* stream);

/*
 * All cp ring steps of the forward pass, merged in ring order inside one launch:
 * o = causal attention output (dtype desc->dtype), lse = its log-sum-exp.
 * (Pull request #181, mode "p2p": the K/V travel the ring and the chunk results
 * are merged with a single-pass online softmax.)
 */
cpattn_status cpattn_ring_fwd(const cpattn_desc* desc, const void* q, const void* k,
                              const void* v, void* o, float* lse, void* stream);

/* Bytes of device workspace cpattn_ring_bwd needs (float32 row statistics and a
 * 256-byte work counter). */
size_t cpattn_ring_bwd_workspace(const cpattn_desc* desc);

/*
 * Backward pass of cpattn_ring_fwd (pull request #181, mode "p2p": recompute the
 * probabilities; the K/V gradients go back to their owner).  Inputs are the
 * forward's q, k, v, o, lse and the upstream gradient dO (same dtype as q);
 * outputs dq [B,H_q,T,D], dk and dv [B,H_kv,T,D] in layout order, so each rank's
 * slice of dk/dv is what its owner receives.  `workspace` is device scratch of at
 * least cpattn_ring_bwd_workspace(desc) bytes (ws_bytes smaller ->
 * CPATTN_ERR_INVALID_ARG); its contents on entry do not matter.
 * On the tensor-core path the dQ kernel is launched as a programmatic dependent
 * of the dK/dV kernel on `stream` (it starts on the SMs that the dK/dV kernel's
 * last CTAs leave idle), and completes only after the dK/dV kernel has: work
 * queued on `stream` afterwards sees every result.
 */
cpattn_status cpattn_ring_bwd(const cpattn_desc* desc, const void* q, const void* k,
                              const void* v, const void* o, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * The backward pass for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is an interface addition of this library.  Callers
 * such as engine plugins that may only enqueue work into buffers handed to them,
 * or programs that reserve all device memory up front and forbid allocation
 * while a step runs, cannot provide the workspace cpattn_ring_bwd asks for.
 * This call computes exactly what cpattn_ring_bwd computes (same arguments
 * minus the workspace) and uses instead a scratch array compiled into the
 * library: 16 MiB and 256 bytes of device memory that every GPU loading the
 * library holds until the process exits.  It allocates nothing, on the device or
 * through any allocating library routine.
 *   Limit: cpattn_ring_bwd_workspace(desc) <= 16 MiB + 256 bytes, i.e. B * H_q * T <=
 *   2,097,152 query rows; larger problems return CPATTN_ERR_UNSUPPORTED before
 *   anything is enqueued.
 *   Set-up: the first call on a device looks up the scratch's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 *   Sharing: every call on a device uses the same scratch, which keeps the last
 *   call's contents (nothing needs clearing: each call writes what it reads).
 *   Two calls that overlap on the GPU race on it; order them on one stream.
 *   Device reset: the scratch's address is cached per device for the life of
 *   the process; after cudaDeviceReset it is stale, so do not call this entry
 *   point again in a process that has reset the device.
 * Other errors as cpattn_ring_bwd.
 */
cpattn_status cpattn_ring_bwd_noalloc(const cpattn_desc* desc, const void* q, const void* k,
                                      const void* v, const void* o, const float* lse,
                                      const void* dO, void* dq, void* dk, void* dv,
                                      void* stream);

/*
 * One forward + backward step over tensors in HOST memory, with the transfers
 * overlapping the compute.  The pages put no host transfer on the path; this call
 * is the library's own form of what a caller whose tensors live on the host does
 * each step (upload, permute to layout order, cpattn_ring_fwd, cpattn_ring_bwd,
 * permute back, download), so that the copies hide behind the kernels instead of
 * adding to them.  The problem is cut into two independent halves when it splits
 * evenly (batch rows when B is even, else the K/V heads with their query heads when
 * B = 1 and H_kv is even): one half's uploads run while the other computes, and its
 * results download while the next work runs, on two copy streams the library
 * creates once per device; calls on one device share them.
 *   q, k, v, dO       : HOST, natural token order, [B, H, T, D] in desc->dtype
 *   o, dq, dk, dv     : HOST, natural token order, same shapes
 *   lse               : HOST, [B, H_q, T] float32, natural order
 *   workspace         : device memory, 256-byte aligned, at least
 *                       cpattn_ring_step_host_workspace(desc) bytes (staging, the
 *                       layout-order tensors and the backward's statistics)
 * Host buffers should be page-locked (cudaHostAlloc); pageable memory works but its
 * copies do not overlap.  The call returns after enqueueing; the host outputs are
 * complete when `stream`'s work is (for example after cpattn_check(stream)).
 * Errors: desc->a2a != 1 -> CPATTN_ERR_UNSUPPORTED; a null pointer, a misaligned or
 * too small workspace -> CPATTN_ERR_INVALID_ARG, before anything is enqueued;
 * others as cpattn_ring_fwd / cpattn_ring_bwd.
 */
size_t cpattn_ring_step_host_workspace(const cpattn_desc* desc);
cpattn_status cpattn_ring_step_host(const cpattn_desc* desc, const void* q, const void* k,
                                    const void* v, const void* dO, void* o, float* lse, void* dq,
                                    void* dk, void* dv, void* workspace, size_t ws_bytes,
                                    void* stream);

/*
 * Packed sequences (transformers pull request #50497: the packed variant restarts
 * the position ids mid-sequence and the mask is rebuilt for the documents; the
 * InfiniTrain pull request #181 leaves packed / variable-length sequences out).
 * Every batch row holds n_docs documents back to back: document d of row b is
 * natural positions [starts[b][d], starts[b][d+1]), and a token attends to the
 * keys of its own document at or before it (causal attention with the position
 * restarting at every document).  Otherwise as cpattn_ring_fwd / cpattn_ring_bwd.
 *   starts    : device int32 [B][n_docs + 1], natural positions, starts[b][0] = 0,
 *               non-decreasing (empty documents allowed), starts[b][n_docs] = T;
 *               4-byte aligned.  Starts that break this contract give unspecified
 *               (but finite, in-bounds) results.
 *   workspace : at least cpattn_packed_workspace(desc) bytes (the documents of
 *               every position, the 128-token tiles in order of decreasing work,
 *               and for the backward the row statistics and a work counter)
 * Errors: n_docs < 1, null or misaligned starts, workspace too small ->
 * CPATTN_ERR_INVALID_ARG; desc->a2a != 1 -> CPATTN_ERR_UNSUPPORTED; others as
 * cpattn_ring_fwd / cpattn_ring_bwd.
 */
size_t cpattn_packed_workspace(const cpattn_desc* desc);
cpattn_status cpattn_ring_fwd_packed(const cpattn_desc* desc, const int32_t* starts, int n_docs,
                                     const void* q, const void* k, const void* v, void* o,
                                     float* lse, void* workspace, size_t ws_bytes, void* stream);
cpattn_status cpattn_ring_bwd_packed(const cpattn_desc* desc, const int32_t* starts, int n_docs,
                                     const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dO, void* dq, void* dk,
                                     void* dv, void* workspace, size_t ws_bytes, void* stream);

/*
 * All-gather mode, forward (pull request #181, mode table row "all_gather": the
 * K/V of every rank is gathered and the rank's own queries attend to it; tutorial
 * "上下文并行", section "Zig-Zag Ring Attention 的通信与计算重叠", bullet
 * "all-gather": each GPU receives the complete K/V in one collective).  Rank
 * q_rank's query rows attend to every key at or before their global position in
 * one pass: no ring steps and no merge.
 *   q, k, v : full layout-order tensors (the rank's rows are q's slots
 *             [q_rank*c, (q_rank+1)*c); k and v are the gathered sequence)
 *   o       : [B', H_q', c, D], dtype desc->dtype (the rank's rows, slot order)
 *   lse     : [B', H_q', c] float32, natural logarithm
 * (B', H_q', c as for cpattn_partial_fwd.)
 * Errors: q_rank outside [0, cp/a2a) -> CPATTN_ERR_INVALID_ARG.
 */
cpattn_status cpattn_allgather_fwd(const cpattn_desc* desc, int q_rank, const void* q,
                                   const void* k, const void* v, void* o, float* lse,
                                   void* stream);

/* Bytes of device workspace cpattn_allgather_bwd needs (float32 row statistics of
 * one rank's rows and a 256-byte work counter; on the tensor-core path the call's
 * dQ kernel overlaps the end of its dK/dV kernel, as in cpattn_ring_bwd). */
size_t cpattn_allgather_bwd_workspace(const cpattn_desc* desc);

/*
 * All-gather mode, backward (pull request #181, mode table row "all_gather": the
 * K/V gradients of all ranks are summed by a ReduceScatter).  Computes rank
 * q_rank's dQ and its share of the K/V gradient of the whole sequence, and adds
 * that share into float32 sums, which is the ReduceScatter's addition:
 *   q, k, v          : full layout-order tensors
 *   o, lse, dO       : the rank's rows, as cpattn_allgather_fwd returns them
 *                      ([B', H_q', c, D], [B', H_q', c] float32, [B', H_q', c, D])
 *   dq               : [B', H_q', c, D], dtype desc->dtype
 *   dk_sum, dv_sum   : [B', H_kv', T, D] float32, layout order.  accumulate = 0
 *                      overwrites them with the rank's share, 1 adds the share to
 *                      what they hold.  Calling q_rank = 0 (accumulate 0), then
 *                      1, ..., cp/a2a - 1 (accumulate 1) in order on one stream
 *                      leaves the full dK, dV: rank s's slice [s*c, (s+1)*c) is
 *                      what s receives from the ReduceScatter.
 *   workspace        : at least cpattn_allgather_bwd_workspace(desc) bytes
 *                      (smaller -> CPATTN_ERR_INVALID_ARG); contents on entry do
 *                      not matter.
 * Errors: q_rank outside [0, cp/a2a) or accumulate not 0/1 -> CPATTN_ERR_INVALID_ARG;
 * others as cpattn_ring_bwd.
 */
cpattn_status cpattn_allgather_bwd(const cpattn_desc* desc, int q_rank, const void* q,
                                   const void* k, const void* v, const void* o,
                                   const float* lse, const void* dO, void* dq, float* dk_sum,
                                   float* dv_sum, int accumulate, void* workspace,
                                   size_t ws_bytes, void* stream);

/*
 * Permutes one tensor of n_heads heads (H_q or H_kv) between orders:
 *  CPATTN_ZIGZAG_FWD / _INV : [B][n_heads][T][D] natural <-> layout order of
 *      desc->layout over the ring's cp/a2a ranks (tutorial, section "Zig-Zag Ring
 *      Attention": rank r holds chunks r and 2cp-1-r).
 *  CPATTN_A2A_FWD / _INV : the all-to-all of the hierarchical mode (pull request
 *      #181, mode "a2a+p2p"; tutorial, section "Ulysses CP").  Token-sharded
 *      [cp][B][T/cp][n_heads][D] (rank r's tokens in desc->layout order over cp)
 *      <-> head-sharded [a2a][B][n_heads/a2a][T][D]: the cp ranks form a2a groups
 *      of consecutive ranks; slice j holds heads [j*n_heads/a2a, ...) of every
 *      token, and its token axis is the layout order of the p2p = cp/a2a ring
 *      whose rank k is a2a group k.
 * Element size from desc->dtype.  A pure copy: bit-exact.  src and dst must not
 * overlap.
 */
cpattn_status cpattn_layout(int permute, const cpattn_desc* desc, const void* src, void* dst,
                            int n_heads, void* stream);

/*
 * The permutes of several tensors of one descriptor in one call, e.g. a step's q,
 * k, v and dO before the ring, or o, dq, dk and dv after it: tensor i goes from
 * src[i] to dst[i] and has n_heads[i] heads.  The result is that of n calls of
 * cpattn_layout; zigzag permutes whose rows are whole 16-byte vectors run as a
 * single launch of chunk moves (the K/V-sized tensors alone would be launch-bound).
 *   n        : 1 <= n <= 8
 *   src, dst, n_heads : HOST arrays of n entries (device pointers in src and dst)
 * Errors: n out of range or a null array -> CPATTN_ERR_INVALID_ARG; each tensor is
 * checked as by cpattn_layout, before anything is enqueued.
 */
cpattn_status cpattn_layout_batch(int permute, const cpattn_desc* desc, int n,
                                  const void* const* src, void* const* dst, const int* n_heads,
                                  void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns the first device error since the last check
 * (CPATTN_ERR_TIMEOUT: a kernel's bounded wait ran out; CPATTN_ERR_BOUNDS: a
 * bounds check of a CPATTN_DEBUG build failed), CPATTN_ERR_CUDA on a CUDA error,
 * else CPATTN_OK.
 */
cpattn_status cpattn_check(void* stream);

/* Static English text for a status code. */
const char* cpattn_status_string(cpattn_status status);

/*
 * Kernel timing (instrumentation for measurement).  While enabled, every kernel
 * the library enqueues is bracketed by CUDA events recorded on its stream.
 * cpattn_timing_collect synchronises those events and adds their durations to
 * per-kernel totals; cpattn_timing_get reads total milliseconds and launch count
 * of entry `index` (0 <= index < cpattn_timing_count()).  Host-side only.
 */
cpattn_status cpattn_timing_enable(int on);
cpattn_status cpattn_timing_collect(void);
int cpattn_timing_count(void);
cpattn_status cpattn_timing_get(int index, const char** name, double* total_ms,
                                int64_t* launches);
cpattn_status cpattn_timing_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
