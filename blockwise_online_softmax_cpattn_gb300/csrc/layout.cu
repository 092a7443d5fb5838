// Layout permutes: the zigzag token map and the all-to-all head<->sequence
// re-layout of the hierarchical mode, as chunk moves (zigzag) or row gathers with
// 16-byte vectors.
//
// Every destination row (D elements) is copied from one source row; threads
// walk the destination in order, so stores are fully coalesced and each source
// row is read as one contiguous run.  Pure copies: bit-exact by construction.
#include "kernels.h"

namespace cpattn {

struct PermuteDev {
  int kind, B, H, T, a2a, Hs, c_src;
  SeqMap ring;   // layout map over the ring's ranks (zigzag permutes; a2a destination)
  SeqMap shard;  // layout map over all cp ranks (a2a source shards)
};

// Source row of destination row `row`.
__device__ __forceinline__ int64_t permute_src_row(const PermuteDev& p, int64_t row) {
  switch (p.kind) {
    case kZigzagFwd: {  // dst [b][h][slot] <- src [b][h][pos(slot)]
      int64_t bh = row / p.T;
      int t = (int)(row - bh * p.T);
      return bh * p.T + p.ring.pos(t);
    }
    case kZigzagInv: {  // dst [b][h][pos] <- src [b][h][slot(pos)]
      int64_t bh = row / p.T;
      int t = (int)(row - bh * p.T);
      return bh * p.T + p.ring.slot(t);
    }
    case kA2AFwd: {  // dst [j][b][hh][t] <- src [r][b][w][h]
      int t = (int)(row % p.T);
      int64_t rest = row / p.T;
      int hh = (int)(rest % p.Hs);
      rest /= p.Hs;
      int b = (int)(rest % p.B);
      int j = (int)(rest / p.B);
      int pos = p.ring.pos(t);
      int s = p.shard.slot(pos);
      int r = s / p.c_src, w = s - r * p.c_src;
      return (((int64_t)r * p.B + b) * p.c_src + w) * p.H + (j * p.Hs + hh);
    }
    default: {  // kA2AInv: dst [r][b][w][h] <- src [j][b][hh][t]
      int h = (int)(row % p.H);
      int64_t rest = row / p.H;
      int w = (int)(rest % p.c_src);
      rest /= p.c_src;
      int b = (int)(rest % p.B);
      int r = (int)(rest / p.B);
      int pos = p.shard.pos(r * p.c_src + w);
      int t = p.ring.slot(pos);
      int j = h / p.Hs, hh = h - j * p.Hs;
      return (((int64_t)j * p.B + b) * p.Hs + hh) * p.T + t;
    }
  }
}

template <typename V>
__global__ void __launch_bounds__(256) permute_kernel(PermuteDev p, const V* __restrict__ src,
                                                      V* __restrict__ dst, int64_t rows,
                                                      int vpr) {
  const int64_t total = rows * (int64_t)vpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t row = i / vpr;
    int v = (int)(i - row * vpr);
    int64_t s = permute_src_row(p, row);
    dst[i] = __ldcs(src + s * vpr + v);
  }
}

// Row gathers for rows of 8, 16 or 32 16-byte vectors: G = 8 threads share a row,
// each copying VPT = vpr / 8 of its vectors (so a group reads and writes 128
// contiguous bytes per instruction), and every thread keeps kRowsInFlight rows in
// flight; the source row is worked out once per row and thread rather than once
// per vector.
constexpr int kRowGroup = 8;
constexpr int kRowsInFlight = 4;

template <int VPT>
__global__ void __launch_bounds__(256) gather_rows_kernel(PermuteDev p, const int4* __restrict__ src,
                                                          int4* __restrict__ dst, int64_t rows) {
  constexpr int vpr = kRowGroup * VPT;
  const int lg = threadIdx.x % kRowGroup;
  const int64_t grp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kRowGroup;
  const int64_t ngrp = (int64_t)gridDim.x * blockDim.x / kRowGroup;
  for (int64_t r0 = grp; r0 < rows; r0 += ngrp * kRowsInFlight) {
    int4 v[kRowsInFlight][VPT];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int64_t row = r0 + u * ngrp;
      if (row < rows) {
        const int4* s = src + permute_src_row(p, row) * vpr + lg;
#pragma unroll
        for (int i = 0; i < VPT; ++i) v[u][i] = __ldcs(s + i * kRowGroup);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int64_t row = r0 + u * ngrp;
      if (row < rows) {
        int4* d = dst + row * vpr + lg;
#pragma unroll
        for (int i = 0; i < VPT; ++i) __stcs(d + i * kRowGroup, v[u][i]);
      }
    }
  }
}

// Row gathers of several tensors (same kind, row size and token count; head
// counts of their own) in one launch: rows [first[i], first[i + 1]) of the launch
// are tensor i's.
struct RowBatch {
  const int4* src[kMaxBatch];
  int4* dst[kMaxBatch];
  int64_t first[kMaxBatch + 1];
  int H[kMaxBatch];
  int n;
};

template <int VPT>
__global__ void __launch_bounds__(256) gather_rows_batch_kernel(PermuteDev p, RowBatch jobs) {
  constexpr int vpr = kRowGroup * VPT;
  const int lg = threadIdx.x % kRowGroup;
  const int64_t rows = jobs.first[jobs.n];
  const int64_t grp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kRowGroup;
  const int64_t ngrp = (int64_t)gridDim.x * blockDim.x / kRowGroup;
  for (int64_t r0 = grp; r0 < rows; r0 += ngrp * kRowsInFlight) {
    int4 v[kRowsInFlight][VPT];
    int4* d[kRowsInFlight];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int64_t row = r0 + u * ngrp;
      d[u] = nullptr;
      if (row < rows) {
        int ti = 0;  // the tensor this row belongs to
        while (ti + 1 < jobs.n && row >= jobs.first[ti + 1]) ++ti;
        const int64_t local = row - jobs.first[ti];
        PermuteDev q = p;
        q.H = jobs.H[ti];
        q.Hs = q.H / p.a2a;
        const int4* s = jobs.src[ti] + permute_src_row(q, local) * vpr + lg;
#pragma unroll
        for (int i = 0; i < VPT; ++i) v[u][i] = __ldcs(s + i * kRowGroup);
        d[u] = jobs.dst[ti] + local * vpr + lg;
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      if (d[u] != nullptr) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) __stcs(d[u] + i * kRowGroup, v[u][i]);
      }
    }
  }
}

template <int VPT>
static cudaError_t run_rows_batch(const PermuteDev& p, const RowBatch& jobs, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = jobs.first[jobs.n];
  int64_t blocks = (rows * kRowGroup + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  gather_rows_batch_kernel<VPT><<<(unsigned)blocks, 256, 0, st>>>(p, jobs);
  return cudaGetLastError();
}

template <int VPT>
static cudaError_t run_rows(const PermuteDev& p, const void* src, void* dst, int64_t rows,
                            cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (rows * kRowGroup + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  gather_rows_kernel<VPT><<<(unsigned)blocks, 256, 0, st>>>(p, (const int4*)src, (int4*)dst, rows);
  return cudaGetLastError();
}

// Zigzag permutes as chunk moves.  Each (batch, head) sequence is 2*cp chunks of
// h = T/(2cp) rows (cp chunks of T/cp rows for the contiguous layout, where the
// map is the identity); slot-chunk k holds natural chunk k/2 for even k and
// 2cp-1-k/2 for odd k (tutorial "上下文并行", section "Zig-Zag Ring
// Attention").  A block copies one part of one destination chunk with streaming
// 16-byte loads, kUnroll of them in flight per thread; no per-element index math.
constexpr int kChunkThreads = 256;
constexpr int kUnroll = 8;

// The tensors one chunk-copy launch moves: up to kMaxBatch of them, all with the
// same chunk size; tensor i's chunks are units [first[i], first[i + 1]) of the
// launch (B * heads sequences of nchunk chunks each).
struct ChunkBatch {
  const int4* src[kMaxBatch];
  int4* dst[kMaxBatch];
  int64_t first[kMaxBatch + 1];
  int n;
};

__global__ void __launch_bounds__(kChunkThreads) chunk_copy_kernel(
    ChunkBatch jobs, int64_t chunk_vecs, int nchunk, int cp, int zz, int inverse, int splits) {
  const int64_t blk = blockIdx.x;
  const int part = (int)(blk % splits);
  int64_t unit = blk / splits;
  int ti = 0;  // the tensor this unit belongs to
  while (ti + 1 < jobs.n && unit >= jobs.first[ti + 1]) ++ti;
  unit -= jobs.first[ti];
  const int4* __restrict__ src = jobs.src[ti];
  int4* __restrict__ dst = jobs.dst[ti];
  const int k = (int)(unit % nchunk);  // destination chunk
  const int64_t bh = unit / nchunk;
  int c = k;                            // source chunk
  if (zz) {
    if (!inverse) c = (k & 1) ? 2 * cp - 1 - (k >> 1) : (k >> 1);
    else c = k < cp ? 2 * k : 2 * (2 * cp - 1 - k) + 1;
  }
  const int64_t per = chunk_vecs / splits;
  const int4* s = src + (bh * nchunk + c) * chunk_vecs + part * per;
  int4* d = dst + (bh * nchunk + k) * chunk_vecs + part * per;
  for (int64_t i0 = threadIdx.x; i0 < per; i0 += (int64_t)kChunkThreads * kUnroll) {
    int4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + (int64_t)u * kChunkThreads;
      if (i < per) v[u] = __ldcs(s + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + (int64_t)u * kChunkThreads;
      if (i < per) __stcs(d + i, v[u]);
    }
  }
}

// n zigzag permutes of tensors with the same T, D and element size (heads[i] heads
// each) as one launch of chunk moves.
static cudaError_t run_chunks(const PermuteArgs& a, int n, const void* const* src,
                              void* const* dst, const int* heads, int row_bytes,
                              cudaStream_t st) {
  const int cpr = a.cp / a.a2a;  // ranks of the ring the permute serves
  const int nchunk = a.zz ? 2 * cpr : cpr;
  const int64_t chunk_vecs = (int64_t)(a.T / nchunk) * row_bytes / 16;
  ChunkBatch jobs;
  jobs.n = n;
  jobs.first[0] = 0;
  for (int i = 0; i < n; ++i) {
    jobs.src[i] = static_cast<const int4*>(src[i]);
    jobs.dst[i] = static_cast<int4*>(dst[i]);
    jobs.first[i + 1] = jobs.first[i] + (int64_t)a.B * heads[i] * nchunk;
  }
  const int64_t units = jobs.first[n];
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // enough blocks to cover every SM several times over
  int splits = 1;
  while (splits < 64 && units * splits < 4LL * sms && chunk_vecs % (2 * splits) == 0 &&
         chunk_vecs / (2 * splits) >= kChunkThreads)
    splits *= 2;
  const int64_t blocks = units * splits;
  if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  chunk_copy_kernel<<<(unsigned)blocks, kChunkThreads, 0, st>>>(
      jobs, chunk_vecs, nchunk, cpr, a.zz, a.kind == kZigzagInv, splits);
  return cudaGetLastError();
}

template <typename V>
static cudaError_t run(const PermuteDev& p, const void* src, void* dst, int64_t rows, int vpr,
                       cudaStream_t st) {
  int64_t total = rows * vpr;
  int64_t blocks = (total + 255) / 256;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  permute_kernel<V><<<(unsigned)blocks, 256, 0, st>>>(p, (const V*)src, (V*)dst, rows, vpr);
  return cudaGetLastError();
}

cudaError_t launch_permute(const PermuteArgs& a, const void* src, void* dst, cudaStream_t st) {
  PermuteDev p;
  p.kind = a.kind;
  p.B = a.B;
  p.H = a.H;
  p.T = a.T;
  p.a2a = a.a2a;
  p.Hs = a.H / a.a2a;
  p.c_src = a.T / a.cp;
  p.ring = SeqMap::make(a.T, a.cp / a.a2a, a.zz);
  p.shard = SeqMap::make(a.T, a.cp, a.zz);
  const int64_t rows = (int64_t)a.B * a.H * a.T;
  const int row_bytes = a.D * a.elt;
  const uintptr_t al = (uintptr_t)src | (uintptr_t)dst;
  timing_begin(a.kind <= kZigzagInv ? "layout_zigzag" : "layout_a2a", st);
  cudaError_t e;
  const int nchunk = a.zz ? 2 * (a.cp / a.a2a) : a.cp / a.a2a;
  if (a.kind <= kZigzagInv && row_bytes % 16 == 0 && al % 16 == 0 && a.T % nchunk == 0)
    e = run_chunks(a, 1, &src, &dst, &a.H, row_bytes, st);
  else if (row_bytes % 16 == 0 && al % 16 == 0 && row_bytes / 16 == 16)
    e = run_rows<2>(p, src, dst, rows, st);
  else if (row_bytes % 16 == 0 && al % 16 == 0 && row_bytes / 16 == 8)
    e = run_rows<1>(p, src, dst, rows, st);
  else if (row_bytes % 16 == 0 && al % 16 == 0 && row_bytes / 16 == 32)
    e = run_rows<4>(p, src, dst, rows, st);
  else if (row_bytes % 16 == 0 && al % 16 == 0)
    e = run<int4>(p, src, dst, rows, row_bytes / 16, st);
  else if (row_bytes % 8 == 0 && al % 8 == 0)
    e = run<int2>(p, src, dst, rows, row_bytes / 8, st);
  else if (row_bytes % 4 == 0 && al % 4 == 0)
    e = run<int>(p, src, dst, rows, row_bytes / 4, st);
  else
    e = run<short>(p, src, dst, rows, row_bytes / 2, st);
  timing_end(st);
  return e;
}

// Several permutes of one kind over tensors of one descriptor (n_heads[i] heads
// each): zigzag permutes whose rows are whole 16-byte vectors go out as one launch
// of chunk moves; anything else as one launch per tensor.
cudaError_t launch_permute_batch(const PermuteArgs& a, int n, const void* const* src,
                                 void* const* dst, const int* n_heads, cudaStream_t st) {
  const int row_bytes = a.D * a.elt;
  const int nchunk = a.zz ? 2 * (a.cp / a.a2a) : a.cp / a.a2a;
  bool aligned = n <= kMaxBatch;
  for (int i = 0; i < n && aligned; ++i)
    aligned = (((uintptr_t)src[i] | (uintptr_t)dst[i]) % 16) == 0;
  const bool chunks = aligned && a.kind <= kZigzagInv && row_bytes % 16 == 0 && a.T % nchunk == 0;
  const int vpr = row_bytes / 16;
  const bool gathers = aligned && a.kind >= kA2AFwd && row_bytes % 16 == 0 &&
                       (vpr == 8 || vpr == 16 || vpr == 32);
  if (gathers) {
    // the a2a re-layouts of all the tensors as one launch of row gathers
    PermuteDev p;
    p.kind = a.kind;
    p.B = a.B;
    p.T = a.T;
    p.a2a = a.a2a;
    p.c_src = a.T / a.cp;
    p.ring = SeqMap::make(a.T, a.cp / a.a2a, a.zz);
    p.shard = SeqMap::make(a.T, a.cp, a.zz);
    p.H = n_heads[0];
    p.Hs = p.H / a.a2a;
    RowBatch jobs;
    jobs.n = n;
    jobs.first[0] = 0;
    for (int i = 0; i < n; ++i) {
      jobs.src[i] = static_cast<const int4*>(src[i]);
      jobs.dst[i] = static_cast<int4*>(dst[i]);
      jobs.H[i] = n_heads[i];
      jobs.first[i + 1] = jobs.first[i] + (int64_t)a.B * n_heads[i] * a.T;
    }
    timing_begin("layout_a2a_batch", st);
    cudaError_t e = vpr == 16 ? run_rows_batch<2>(p, jobs, st)
                    : vpr == 8 ? run_rows_batch<1>(p, jobs, st)
                               : run_rows_batch<4>(p, jobs, st);
    timing_end(st);
    return e;
  }
  if (!chunks) {
    for (int i = 0; i < n; ++i) {
      PermuteArgs ai = a;
      ai.H = n_heads[i];
      cudaError_t e = launch_permute(ai, src[i], dst[i], st);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  timing_begin("layout_zigzag_batch", st);
  cudaError_t e = run_chunks(a, n, src, dst, n_heads, row_bytes, st);
  timing_end(st);
  return e;
}

}  // namespace cpattn
