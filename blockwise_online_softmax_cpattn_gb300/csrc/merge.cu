// (O, LSE) merge of two partial results, and the backward pre-pass
// Delta = rowsum(dO * O) (plus the LSE rescaled to base 2 for the tensor-core
// backward).  Both are HBM-bound row kernels: one warp per row, 16-byte vector
// accesses, float32 arithmetic.
#include <math.h>

#include "kernels.h"

namespace cpattn {

// Online-softmax merge (tutorial "上下文并行", section "朴素 Ring Attention": the
// block order is free as long as the current output, max and sum are carried).
// lse = m + ln(e^(la-m) + e^(lb-m)) with m = max(la, lb); an operand with
// lse = -inf contributes nothing; two empty operands give (0, -inf).
// All lanes read both LSEs before lane 0 overwrites lse_out (which may alias
// lse_a or lse_b); o_out[i] depends only on o_a[i], o_b[i].
template <bool VEC4>
__global__ void __launch_bounds__(256) merge_kernel(int64_t rows, int D,
                                                    const float* oa, const float* la,
                                                    const float* ob, const float* lb,
                                                    float* oo, float* lo) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    float4 xa, xb;
    if (VEC4 && D == 128) {  // the row's operands in flight before its weights are known
      xa = reinterpret_cast<const float4*>(oa + row * 128)[lane];
      xb = reinterpret_cast<const float4*>(ob + row * 128)[lane];
    }
    const float a = la[row], b = lb[row];
    const float m = fmaxf(a, b);
    float wa = 0.f, wb = 0.f, lse = -INFINITY;
    if (m != -INFINITY) {
      const float ea = expf(a - m), eb = expf(b - m);
      const float s = ea + eb;
      wa = ea / s;
      wb = eb / s;
      lse = m + logf(s);
    }
    const int64_t base = row * (int64_t)D;
    if (VEC4 && D == 128) {
      float4 z;
      z.x = wa * xa.x + wb * xb.x;
      z.y = wa * xa.y + wb * xb.y;
      z.z = wa * xa.z + wb * xb.z;
      z.w = wa * xa.w + wb * xb.w;
      reinterpret_cast<float4*>(oo + base)[lane] = z;
    } else if (VEC4) {
      const float4* pa = reinterpret_cast<const float4*>(oa + base);
      const float4* pb = reinterpret_cast<const float4*>(ob + base);
      float4* po = reinterpret_cast<float4*>(oo + base);
      for (int i = lane; i < D / 4; i += 32) {
        float4 x = pa[i], y = pb[i], z;
        z.x = wa * x.x + wb * y.x;
        z.y = wa * x.y + wb * y.y;
        z.z = wa * x.z + wb * y.z;
        z.w = wa * x.w + wb * y.w;
        po[i] = z;
      }
    } else {
      for (int i = lane; i < D; i += 32) oo[base + i] = wa * oa[base + i] + wb * ob[base + i];
    }
    __syncwarp();
    if (lane == 0) lo[row] = lse;
  }
}

cudaError_t launch_merge(int64_t rows, int D, const float* oa, const float* la, const float* ob,
                         const float* lb, float* oo, float* lo, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (rows + 7) / 8;
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  timing_begin("merge", st);
  if (D % 4 == 0)
    merge_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(rows, D, oa, la, ob, lb, oo, lo);
  else
    merge_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(rows, D, oa, la, ob, lb, oo, lo);
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

// ---------------------------------------------------------------------------
__device__ __forceinline__ float ld_f(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__global__ void __launch_bounds__(256) delta_kernel(int64_t rows, int D, const T* __restrict__ o,
                                                    const T* __restrict__ dO,
                                                    const float* __restrict__ lse,
                                                    float* __restrict__ delta,
                                                    float* __restrict__ lse2) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const int64_t base = row * (int64_t)D;
    float acc = 0.f;
    constexpr int kVec = 16 / sizeof(T);
    if (D % kVec == 0) {
      for (int i = lane * kVec; i < D; i += 32 * kVec) {
        int4 a = *reinterpret_cast<const int4*>(o + base + i);
        int4 b = *reinterpret_cast<const int4*>(dO + base + i);
        const T* pa = reinterpret_cast<const T*>(&a);
        const T* pb = reinterpret_cast<const T*>(&b);
#pragma unroll
        for (int k = 0; k < kVec; ++k) acc += ld_f(pa, k) * ld_f(pb, k);
      }
    } else {
      for (int i = lane; i < D; i += 32) acc += ld_f(o, base + i) * ld_f(dO, base + i);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      if (lse2) {  // tensor-core form: both statistics negated, LSE in base 2
        delta[row] = -acc;
        lse2[row] = -lse[row] * 1.44269504088896340736f;
      } else {
        delta[row] = acc;
      }
    }
  }
}

// bf16 rows of V int4 vectors (D = 8V): four lanes per row, each holding its V/4
// vector loads of o and dO in flight at once, so a warp covers 8 rows per pass
// and the loads of many rows overlap (the one-warp-per-row form above keeps only
// two loads of one row in flight and is latency-bound at these sizes).
template <int V>
__global__ void __launch_bounds__(256) delta_rows4_kernel(int64_t rows,
                                                          const __nv_bfloat16* __restrict__ o,
                                                          const __nv_bfloat16* __restrict__ dO,
                                                          const float* __restrict__ lse,
                                                          float* __restrict__ delta,
                                                          float* __restrict__ lse2) {
  constexpr int kPer = V / 4;  // vectors per lane
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;
  const int64_t groups = (int64_t)gridDim.x * (blockDim.x >> 2);
  for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 2; row < rows;
       row += groups) {
    const int4* a4 = reinterpret_cast<const int4*>(o) + row * V + sub * kPer;
    const int4* b4 = reinterpret_cast<const int4*>(dO) + row * V + sub * kPer;
    int4 a[kPer], b[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      a[k] = __ldcs(a4 + k);
      b[k] = __ldcs(b4 + k);
    }
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a[k]);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(pa[e]), fb = __bfloat1622float2(pb[e]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
    // the four lanes of a row are consecutive; the loop bound is uniform per group
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (sub == 0) {
      delta[row] = -acc;
      lse2[row] = -lse[row] * 1.44269504088896340736f;
    }
  }
}

cudaError_t launch_delta(int64_t rows, int D, int bf16, const void* o, const void* dO,
                         const float* lse, float* delta, float* lse2, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (rows + 7) / 8;
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  if (blocks < 1) blocks = 1;
  timing_begin("bwd_prepass", st);
  const bool aligned = (((uintptr_t)o | (uintptr_t)dO) & 15) == 0;
  if (bf16 && lse2 && aligned && (D == 128 || D == 64) && rows % 8 == 0) {
    // 64 rows per block and pass, at most four blocks per SM, each striding over
    // several passes (measured at the LLaMA shape: 27 us with four blocks per SM, 32 us
    // with eight, 43 us with one)
    int64_t g = rows / 64;
    if (g > (int64_t)sms * 4) g = (int64_t)sms * 4;
    if (g < 1) g = 1;
    if (D == 128)
      delta_rows4_kernel<16><<<(unsigned)g, 256, 0, st>>>(rows, (const __nv_bfloat16*)o,
                                                          (const __nv_bfloat16*)dO, lse, delta, lse2);
    else
      delta_rows4_kernel<8><<<(unsigned)g, 256, 0, st>>>(rows, (const __nv_bfloat16*)o,
                                                         (const __nv_bfloat16*)dO, lse, delta, lse2);
  } else if (bf16)
    delta_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        rows, D, (const __nv_bfloat16*)o, (const __nv_bfloat16*)dO, lse, delta, lse2);
  else
    delta_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(rows, D, (const float*)o,
                                                          (const float*)dO, lse, delta, lse2);
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

// ---------------------------------------------------------------------------
// Packed sequences: the document of every position (transformers pull request
// #50497: position ids restart at every packed document, and the mask is rebuilt
// from them).  One thread per (batch row, position): the last document whose start
// is <= the position, found by binary search over the row's starts.
// ---------------------------------------------------------------------------
__global__ void doc_bounds_kernel(int B, int T, int n_docs, const int* __restrict__ starts,
                                  int* __restrict__ lo, int* __restrict__ hi) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)B * T) return;
  const int b = (int)(i / T), pos = (int)(i - (int64_t)b * T);
  const int* st = starts + (int64_t)b * (n_docs + 1);
  int a = 0, z = n_docs - 1;  // the document index lies in [a, z]
  while (a < z) {
    const int mid = (a + z + 1) >> 1;
    if (st[mid] <= pos) a = mid;
    else z = mid - 1;
  }
  int l = st[a], h = st[a + 1] - 1;
  // starts that break the contract still leave every position inside its own
  // document (each query sees at least itself)
  l = l > pos ? pos : (l < 0 ? 0 : l);
  h = h < pos ? pos : (h > T - 1 ? T - 1 : h);
  lo[i] = l;
  hi[i] = h;
}

cudaError_t launch_doc_bounds(int B, int T, int n_docs, const int* starts, int* lo, int* hi,
                              cudaStream_t st) {
  const int64_t n = (int64_t)B * T;
  if (n == 0) return cudaSuccess;
  timing_begin("doc_bounds", st);
  doc_bounds_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(B, T, n_docs, starts, lo, hi);
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

// Packed sequences: the (batch row, 128-token tile) entries in order of decreasing
// work, for the query tiles (keys from the tile holding the document start up to
// the diagonal) and for the key tiles (queries from the diagonal up to the tile
// holding the document end), so that the kernels hand out the heaviest work first.
// One block, a counting sort over work (capped at kOrderBuckets - 1 tiles); the
// order inside a bucket is whatever the atomics give, which changes the
// scheduling only, never a result.  Entry value: b * n_tiles + tile.
constexpr int kOrderBuckets = 1024;

__global__ void __launch_bounds__(1024) doc_order_kernel(int B, int T, const int* __restrict__ lo,
                                                         const int* __restrict__ hi,
                                                         int* __restrict__ ord_q,
                                                         int* __restrict__ ord_k) {
  __shared__ int count[2][kOrderBuckets];
  const int nt = T >> 7, n = B * nt;
  // a tile visits at most nt tiles: buckets 0..top
  const int top = nt < kOrderBuckets - 1 ? nt : kOrderBuckets - 1;
  for (int i = threadIdx.x; i < 2 * kOrderBuckets; i += blockDim.x) (&count[0][0])[i] = 0;
  __syncthreads();
  auto work = [&](int e, int which) {
    const int b = e / nt, t = e - b * nt;
    const int wk = which == 0 ? t - (lo[(int64_t)b * T + (t << 7)] >> 7) + 1
                              : (hi[(int64_t)b * T + (t << 7) + 127] >> 7) - t + 1;
    return wk < 1 ? 1 : (wk > top ? top : wk);
  };
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    atomicAdd(&count[0][work(e, 0)], 1);
    atomicAdd(&count[1][work(e, 1)], 1);
  }
  __syncthreads();
  if (threadIdx.x < 2) {  // start of each bucket, heaviest bucket first
    int run = 0;
    for (int v = top; v >= 0; --v) {
      const int c = count[threadIdx.x][v];
      count[threadIdx.x][v] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    ord_q[atomicAdd(&count[0][work(e, 0)], 1)] = e;
    ord_k[atomicAdd(&count[1][work(e, 1)], 1)] = e;
  }
}

cudaError_t launch_doc_order(int B, int T, const int* lo, const int* hi, int* ord_q, int* ord_k,
                             cudaStream_t st) {
  if (B <= 0 || T < 128) return cudaSuccess;
  timing_begin("doc_order", st);
  doc_order_kernel<<<1, 1024, 0, st>>>(B, T, lo, hi, ord_q, ord_k);
  cudaError_t e = cudaGetLastError();
  timing_end(st);
  return e;
}

}  // namespace cpattn
