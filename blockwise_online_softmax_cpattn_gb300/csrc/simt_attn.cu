// SIMT ring attention: the exact float32 path (and the path for shapes the
// tensor-core kernels do not take: D not in {64, 128} or chunk halves that are
// not multiples of 128 tokens).
//
// One warp owns one output row; lane l holds elements d = l + 32*j (j < 4) of
// the q/dO/o rows, so D <= 128.  The forward follows the ring literally: for
// each step i the rank's query row attends to the K/V chunk of rank
// (r - i) mod cp, producing a chunk-local (max, sum, output) by the online
// softmax, which is then merged into the running state (tutorial "上下文并行",
// section "朴素 Ring Attention"; pull request "Feat: Context Parallel" #181, mode
// "p2p").  Keys are visible when their global position is <= the query's.
#include <math.h>

#include "kernels.h"

namespace cpattn {

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

template <typename T>
__device__ __forceinline__ void load_row(const T* p, int D, int lane, float (&x)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int d = lane + 32 * j;
    x[j] = d < D ? to_f(p[d]) : 0.f;
  }
}

template <typename T>
__device__ __forceinline__ float dot_row(const float (&a)[4], const T* p, int D, int lane) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int d = lane + 32 * j;
    if (d < D) s += a[j] * to_f(p[d]);
  }
  return warp_sum(s);
}

struct SimtFwd {
  int B, Hq, Hkv, T, D, n_rep;
  SeqMap m;
  float scale;
  int q_slot0, n_q_slots;  // queries: slots [q_slot0, q_slot0 + n_q_slots)
  int kv_fixed;            // < 0: whole ring; else only this rank's chunk
  int local_rows;          // o/lse hold n_q_slots rows per (b, h) instead of T
  const int* doc_lo;       // packed: first position of each position's document, [B][T]
};

template <typename TI, typename TO>
__global__ void __launch_bounds__(256) simt_fwd_kernel(SimtFwd p, const TI* __restrict__ q,
                                                       const TI* __restrict__ k,
                                                       const TI* __restrict__ v,
                                                       TO* __restrict__ o,
                                                       float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t n_rows = (int64_t)p.B * p.Hq * p.n_q_slots;
  if (w >= n_rows) return;
  const int64_t bh = w / p.n_q_slots;
  const int i_loc = (int)(w - bh * p.n_q_slots);
  const int slot = p.q_slot0 + i_loc;
  const int b = (int)(bh / p.Hq), h = (int)(bh % p.Hq), g = h / p.n_rep;
  const int D = p.D;
  float qv[4];
  load_row(q + ((int64_t)bh * p.T + slot) * D, D, lane, qv);
  const int qpos = p.m.pos(slot);
  const int r = slot / p.m.c;
  const TI* kb = k + ((int64_t)b * p.Hkv + g) * p.T * D;
  const TI* vb = v + ((int64_t)b * p.Hkv + g) * p.T * D;

  float mrun = -INFINITY, lrun = 0.f, orun[4] = {0.f, 0.f, 0.f, 0.f};
  const int steps = p.kv_fixed >= 0 ? 1 : p.m.cp;
  const int lo_q = p.doc_lo ? p.doc_lo[(int64_t)b * p.T + qpos] : 0;
  for (int i = 0; i < steps; ++i) {
    const int s = p.kv_fixed >= 0 ? p.kv_fixed : (r - i + p.m.cp) % p.m.cp;
    // chunk-local online softmax over the K/V held at this step
    float mc = -INFINITY, lc = 0.f, oc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int t = s * p.m.c; t < (s + 1) * p.m.c; ++t) {
      const int kp = p.m.pos(t);
      if (kp > qpos || kp < lo_q) continue;
      const float sc = dot_row(qv, kb + (int64_t)t * D, D, lane) * p.scale;
      const float mn = fmaxf(mc, sc);
      const float corr = expf(mc - mn);
      const float pr = expf(sc - mn);
      lc = lc * corr + pr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int d = lane + 32 * j;
        float vv = d < D ? to_f(vb[(int64_t)t * D + d]) : 0.f;
        oc[j] = oc[j] * corr + pr * vv;
      }
      mc = mn;
    }
    // merge the step's partial into the running state
    if (lc > 0.f) {
      const float mn = fmaxf(mrun, mc);
      const float a = expf(mrun - mn), c = expf(mc - mn);
      lrun = lrun * a + lc * c;
#pragma unroll
      for (int j = 0; j < 4; ++j) orun[j] = orun[j] * a + oc[j] * c;
      mrun = mn;
    }
  }
  const int64_t orow = p.local_rows ? bh * (int64_t)p.n_q_slots + i_loc : bh * (int64_t)p.T + slot;
  const float inv = lrun > 0.f ? 1.f / lrun : 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int d = lane + 32 * j;
    if (d < D) o[orow * D + d] = from_f<TO>(orun[j] * inv);
  }
  if (lane == 0) lse[orow] = lrun > 0.f ? mrun + logf(lrun) : -INFINITY;
}

// dQ_i = scale * sum_j P_ij (dP_ij - Delta_i) k_j, P recomputed from the LSE.
struct SimtBwd {
  int B, Hq, Hkv, T, D, n_rep;
  SeqMap m;
  float scale;
  // All-gather mode (ag_rank >= 0): only rank ag_rank's query rows take part; its
  // o/lse/dO/Delta/dQ hold c = T/cp rows per (b, h) (local rows) while q holds
  // the whole sequence, and dK/dV (float32) receive the rank's share, added to
  // what they hold when `accumulate` is set.
  int ag_rank;
  int accumulate;
  // One ring step (kv_rank >= 0, with ag_rank the query rank): only the keys of
  // chunk kv_rank take part; dQ is float32 and dK/dV hold the chunk's c rows per
  // (b, g), all overwritten or added to like dK/dV above.
  int kv_rank;
  // packed sequences: first / last position of each position's document, [B][T]
  const int* doc_lo;
  const int* doc_hi;
};

template <typename T, typename TO>
__global__ void __launch_bounds__(256) simt_bwd_dq_kernel(SimtBwd p, const T* __restrict__ q,
                                                          const T* __restrict__ k,
                                                          const T* __restrict__ v,
                                                          const float* __restrict__ lse,
                                                          const float* __restrict__ delta,
                                                          const T* __restrict__ dO,
                                                          TO* __restrict__ dq) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  // w indexes the rows of dO / lse / Delta / dQ: all T slots, or the rank's c
  const int n_slots = p.ag_rank >= 0 ? p.m.c : p.T;
  if (w >= (int64_t)p.B * p.Hq * n_slots) return;
  const int64_t bh = w / n_slots;
  const int slot = (int)(w - bh * n_slots) + (p.ag_rank >= 0 ? p.ag_rank * p.m.c : 0);
  const int b = (int)(bh / p.Hq), h = (int)(bh % p.Hq), g = h / p.n_rep;
  const int D = p.D;
  float qv[4], dov[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
  load_row(q + (bh * p.T + slot) * D, D, lane, qv);
  load_row(dO + w * D, D, lane, dov);
  const float L = lse[w], Dl = delta[w];
  const int qpos = p.m.pos(slot);
  const int r = slot / p.m.c;
  const T* kb = k + ((int64_t)b * p.Hkv + g) * p.T * D;
  const T* vb = v + ((int64_t)b * p.Hkv + g) * p.T * D;
  const int lo_q = p.doc_lo ? p.doc_lo[(int64_t)b * p.T + qpos] : 0;
  const bool step = p.kv_rank >= 0;
  for (int i = 0; i < (step ? 1 : p.m.cp); ++i) {
    const int s = step ? p.kv_rank : (r - i + p.m.cp) % p.m.cp;
    for (int t = s * p.m.c; t < (s + 1) * p.m.c; ++t) {
      const int kp = p.m.pos(t);
      if (kp > qpos || kp < lo_q) continue;
      const float pr = expf(dot_row(qv, kb + (int64_t)t * D, D, lane) * p.scale - L);
      const float ds = pr * (dot_row(dov, vb + (int64_t)t * D, D, lane) - Dl);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int d = lane + 32 * j;
        if (d < D) acc[j] += ds * to_f(kb[(int64_t)t * D + d]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int d = lane + 32 * j;
    if (d < D) {
      float x = acc[j] * p.scale;
      if (step && p.accumulate) x += to_f(dq[w * D + d]);
      dq[w * D + d] = from_f<TO>(x);
    }
  }
}

// dK_j = scale * sum_{group heads, i} dS_ij q_i,  dV_j = sum P_ij dO_i, one warp
// per key row; the query ranks are visited in the order the chunk's gradient
// travels the ring back to its owner s: ranks s, s+1, ..., s-1.
template <typename T, typename TO>
__global__ void __launch_bounds__(256) simt_bwd_dkdv_kernel(
    SimtBwd p, const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ lse, const float* __restrict__ delta, const T* __restrict__ dO,
    TO* __restrict__ dk, TO* __restrict__ dv) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  // w indexes the rows of dK / dV: all T slots, or (one ring step) chunk kv_rank's c
  const bool step = p.kv_rank >= 0;
  const int n_slots = step ? p.m.c : p.T;
  if (w >= (int64_t)p.B * p.Hkv * n_slots) return;
  const int64_t bg = w / n_slots;
  const int slot = (int)(w - bg * n_slots) + (step ? p.kv_rank * p.m.c : 0);
  const int b = (int)(bg / p.Hkv), g = (int)(bg % p.Hkv);
  const int D = p.D;
  float kv_[4], vv[4], ak[4] = {0.f, 0.f, 0.f, 0.f}, av[4] = {0.f, 0.f, 0.f, 0.f};
  load_row(k + (bg * p.T + slot) * D, D, lane, kv_);
  load_row(v + (bg * p.T + slot) * D, D, lane, vv);
  const int kpos = p.m.pos(slot);
  const int s = slot / p.m.c;
  const int hi_k = p.doc_hi ? p.doc_hi[(int64_t)b * p.T + kpos] : p.T;
  const bool ag = p.ag_rank >= 0;
  for (int i = 0; i < (ag ? 1 : p.m.cp); ++i) {
    const int r = ag ? p.ag_rank : (s + i) % p.m.cp;
    for (int hh = 0; hh < p.n_rep; ++hh) {
      const int64_t qbh = (int64_t)b * p.Hq + g * p.n_rep + hh;
      for (int t = r * p.m.c; t < (r + 1) * p.m.c; ++t) {
        const int qp = p.m.pos(t);
        if (qp < kpos || qp > hi_k) continue;
        const int64_t qrow = qbh * p.T + t;
        const int64_t srow = ag ? qbh * p.m.c + (t - r * p.m.c) : qrow;  // dO / statistics
        const T* qr = q + qrow * D;
        const T* dor = dO + srow * D;
        const float pr = expf(dot_row(kv_, qr, D, lane) * p.scale - lse[srow]);
        const float ds = pr * (dot_row(vv, dor, D, lane) - delta[srow]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int d = lane + 32 * j;
          if (d < D) {
            av[j] += pr * to_f(dor[d]);
            ak[j] += ds * to_f(qr[d]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int d = lane + 32 * j;
    if (d < D) {
      float ok = ak[j] * p.scale, ov = av[j];
      if (p.accumulate) {
        ok += to_f(dk[w * D + d]);
        ov += to_f(dv[w * D + d]);
      }
      dk[w * D + d] = from_f<TO>(ok);
      dv[w * D + d] = from_f<TO>(ov);
    }
  }
}

static unsigned blocks_for(int64_t warps) { return (unsigned)((warps + 7) / 8); }

cudaError_t launch_simt_fwd(const Ring& R, int q_rank, int kv_rank, const void* q, const void* k,
                            const void* v, void* o, float* lse, cudaStream_t st,
                            const int* doc_lo) {
  SimtFwd p;
  p.B = R.B;
  p.Hq = R.Hq;
  p.Hkv = R.Hkv;
  p.T = R.T;
  p.D = R.D;
  p.n_rep = R.Hq / R.Hkv;
  p.m = SeqMap::make(R.T, R.cp, R.zz);
  p.scale = R.scale;
  // q_rank >= 0 with kv_rank >= 0: one ring step (float32 out); with kv_rank < 0:
  // the all-gather mode (that rank's rows over every chunk, output dtype)
  const bool local = q_rank >= 0;
  const bool partial = local && kv_rank >= 0;
  p.q_slot0 = local ? q_rank * p.m.c : 0;
  p.n_q_slots = local ? p.m.c : R.T;
  p.kv_fixed = partial ? kv_rank : -1;
  p.local_rows = local ? 1 : 0;
  p.doc_lo = doc_lo;
  const int64_t warps = (int64_t)p.B * p.Hq * p.n_q_slots;
  if (warps == 0) return cudaSuccess;
  timing_begin(partial ? "simt_partial_fwd" : local ? "simt_allgather_fwd" : "simt_ring_fwd", st);
  if (R.bf16) {
    if (partial)
      simt_fwd_kernel<__nv_bfloat16, float><<<blocks_for(warps), 256, 0, st>>>(
          p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
          (float*)o, lse);
    else
      simt_fwd_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks_for(warps), 256, 0, st>>>(
          p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
          (__nv_bfloat16*)o, lse);
  } else {
    simt_fwd_kernel<float, float><<<blocks_for(warps), 256, 0, st>>>(
        p, (const float*)q, (const float*)k, (const float*)v, (float*)o, lse);
  }
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

static SimtBwd make_bwd(const Ring& R) {
  SimtBwd p;
  p.B = R.B;
  p.Hq = R.Hq;
  p.Hkv = R.Hkv;
  p.T = R.T;
  p.D = R.D;
  p.n_rep = R.Hq / R.Hkv;
  p.m = SeqMap::make(R.T, R.cp, R.zz);
  p.scale = R.scale;
  p.ag_rank = -1;
  p.accumulate = 0;
  p.kv_rank = -1;
  p.doc_lo = nullptr;
  p.doc_hi = nullptr;
  return p;
}

cudaError_t launch_simt_bwd_dq(const Ring& R, const void* q, const void* k, const void* v,
                               const float* lse, const float* delta, const void* dO, void* dq,
                               cudaStream_t st, const int* doc_lo) {
  SimtBwd p = make_bwd(R);
  p.doc_lo = doc_lo;
  const int64_t warps = (int64_t)p.B * p.Hq * p.T;
  timing_begin("simt_bwd_dq", st);
  if (R.bf16)
    simt_bwd_dq_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks_for(warps), 256, 0, st>>>(
        p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, lse, delta,
        (const __nv_bfloat16*)dO, (__nv_bfloat16*)dq);
  else
    simt_bwd_dq_kernel<float, float><<<blocks_for(warps), 256, 0, st>>>(
        p, (const float*)q, (const float*)k, (const float*)v, lse, delta, (const float*)dO,
        (float*)dq);
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

cudaError_t launch_simt_bwd_dkdv(const Ring& R, const void* q, const void* k, const void* v,
                                 const float* lse, const float* delta, const void* dO, void* dk,
                                 void* dv, cudaStream_t st, const int* doc_hi) {
  SimtBwd p = make_bwd(R);
  p.doc_hi = doc_hi;
  const int64_t warps = (int64_t)p.B * p.Hkv * p.T;
  timing_begin("simt_bwd_dkdv", st);
  if (R.bf16)
    simt_bwd_dkdv_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks_for(warps), 256, 0, st>>>(
        p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, lse, delta,
        (const __nv_bfloat16*)dO, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv);
  else
    simt_bwd_dkdv_kernel<float, float><<<blocks_for(warps), 256, 0, st>>>(
        p, (const float*)q, (const float*)k, (const float*)v, lse, delta, (const float*)dO,
        (float*)dk, (float*)dv);
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

cudaError_t launch_simt_allgather_bwd(const Ring& R, int q_rank, const void* q, const void* k,
                                      const void* v, const float* lse, const float* delta,
                                      const void* dO, void* dq, float* dk_sum, float* dv_sum,
                                      int accumulate, cudaStream_t st) {
  SimtBwd p = make_bwd(R);
  p.ag_rank = q_rank;
  p.accumulate = accumulate ? 1 : 0;
  const int64_t q_warps = (int64_t)p.B * p.Hq * p.m.c;
  const int64_t kv_warps = (int64_t)p.B * p.Hkv * p.T;
  timing_begin("simt_allgather_bwd", st);
  if (R.bf16) {
    simt_bwd_dq_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks_for(q_warps), 256, 0, st>>>(
        p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, lse, delta,
        (const __nv_bfloat16*)dO, (__nv_bfloat16*)dq);
    simt_bwd_dkdv_kernel<__nv_bfloat16, float><<<blocks_for(kv_warps), 256, 0, st>>>(
        p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, lse, delta,
        (const __nv_bfloat16*)dO, dk_sum, dv_sum);
  } else {
    simt_bwd_dq_kernel<float, float><<<blocks_for(q_warps), 256, 0, st>>>(
        p, (const float*)q, (const float*)k, (const float*)v, lse, delta, (const float*)dO,
        (float*)dq);
    simt_bwd_dkdv_kernel<float, float><<<blocks_for(kv_warps), 256, 0, st>>>(
        p, (const float*)q, (const float*)k, (const float*)v, lse, delta, (const float*)dO,
        dk_sum, dv_sum);
  }
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

// One ring step of the backward: rank q_rank's queries against chunk kv_rank's
// keys; float32 contributions to the rank's dQ rows and to the chunk's dK/dV rows.
cudaError_t launch_simt_partial_bwd(const Ring& R, int q_rank, int kv_rank, const void* q,
                                    const void* k, const void* v, const float* lse,
                                    const float* delta, const void* dO, float* dq_part,
                                    float* dk_part, float* dv_part, int accumulate,
                                    cudaStream_t st) {
  SimtBwd p = make_bwd(R);
  p.ag_rank = q_rank;
  p.kv_rank = kv_rank;
  p.accumulate = accumulate ? 1 : 0;
  const int64_t warps = (int64_t)p.B * p.Hq * p.m.c;
  const int64_t kv_warps = (int64_t)p.B * p.Hkv * p.m.c;
  timing_begin("simt_partial_bwd", st);
  if (R.bf16) {
    simt_bwd_dq_kernel<__nv_bfloat16, float><<<blocks_for(warps), 256, 0, st>>>(
        p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, lse, delta,
        (const __nv_bfloat16*)dO, dq_part);
    simt_bwd_dkdv_kernel<__nv_bfloat16, float><<<blocks_for(kv_warps), 256, 0, st>>>(
        p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, lse, delta,
        (const __nv_bfloat16*)dO, dk_part, dv_part);
  } else {
    simt_bwd_dq_kernel<float, float><<<blocks_for(warps), 256, 0, st>>>(
        p, (const float*)q, (const float*)k, (const float*)v, lse, delta, (const float*)dO,
        dq_part);
    simt_bwd_dkdv_kernel<float, float><<<blocks_for(kv_warps), 256, 0, st>>>(
        p, (const float*)q, (const float*)k, (const float*)v, lse, delta, (const float*)dO,
        dk_part, dv_part);
  }
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

}  // namespace cpattn
