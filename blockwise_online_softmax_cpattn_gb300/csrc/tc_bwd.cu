// Ring-attention backward on the 5th-generation tensor cores (sm_103a).
//
// The pull request "Feat: Context Parallel" #181 (mode "p2p") computes the ring
// backward by recomputing the probabilities from the saved statistics and
// sending each K/V chunk's gradient around the ring back to its owner.  On one
// GPU the same sums are formed by two kernels, neither of which adds its results
// with atomics (each output tile is summed by one CTA, in a fixed order):
//
//  dkdv_kernel  one CTA per 128-row K/V tile (K/V stationary in shared memory).
//               Its producer walks the query tiles that can see it (the other
//               roles count them), in the order the
//               chunk's gradient travels the ring (ranks s, s+1, ..., s-1), for
//               every query head of its group, so the grouped-query sum over the
//               n_rep heads (the reverse of RepeatKVHeads) happens in the TMEM
//               accumulators:
//                 S^T = K Q^T, dP^T = V dO^T          (SS MMAs, M = keys)
//                 P^T = 2^(S^T scale log2e - LSE log2e), masked from positions
//                 dS^T = P^T (dP^T - Delta)
//                 dV += P^T dO, dK += dS^T Q          (TS MMAs, P^T/dS^T in TMEM)
//               TMEM: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D, 256+2D).
//  dq_kernel    persistent CTAs over 128-row query tiles (Q, dO stationary),
//               walking the K/V tiles in ring order like the forward:
//                 S = Q K^T, dP = dO V^T, dS = P (dP - Delta), dQ += dS K.
//               TMEM: S [0,128), dP double-buffered [128,384), dQ [384, 384+D).
//               Launched after the dK/dV kernel; when nothing is queued between
//               them, as its programmatic dependent, so it overlaps that kernel's
//               last CTAs, its CTAs claiming their query tiles from a counter.
//
// Delta = rowsum(dO * O) comes from the pre-pass kernel (merge.cu).  Compute
// warps: 8, warp w handles TMEM lane quadrant w%4 and column half (w-4)/4.
// Warp 0 loads through TMA.  The MMA issuers are whole warps: every lane runs
// the issue loop (warp-uniform descriptor arithmetic and waits) and one lane,
// chosen by elect.sync, issues each tcgen05 instruction and commit.  dK/dV:
// warp 1 issues S^T, warp 2 dP^T, dV and dK.  dQ: warp 1 issues S, warp 3 dP,
// warp 2 dQ.
// Every mbarrier wait is bounded (see tc_fwd.cu for the abort protocol).
#include <math.h>

#include "kernels.h"

namespace cpattn {
namespace tcbwd {

constexpr int kTile = 128;
constexpr int kThreads = 384;
constexpr uint64_t kTimeoutNs = 2000000000ull;     // 2 s
constexpr uint64_t kDebugTimeoutNs = 50000000ull;  // 50 ms under the fault hook
constexpr uint64_t kDrainTimeoutNs = 200000000ull;
// Values of the descriptor's test hook that make one of these kernels withhold a
// load (1 is the forward's)
constexpr int kFaultDkdv = 2;
constexpr int kFaultDq = 3;
constexpr float kLog2e = 1.44269504088896340736f;

enum : int { kEmpty = 0, kFull = 1, kDiag = 2 };

struct Params {
  int B, Hq, Hkv, T, n_rep;
  SeqMap m;
  float scale, scale_log2;
  const float* lse2;   // -LSE * log2(e) per query row, from the pre-pass
  const float* delta;  // -Delta per query row, from the pre-pass
  void* out0;  // dkdv: dK ; dq: dQ
  void* out1;  // dkdv: dV
  int* status;
  // All-gather mode (ag_rank >= 0): only rank ag_rank's query rows take part.  q
  // holds the whole sequence; dO, the statistics and dQ hold the rank's c rows per
  // (b, h); dK/dV are float32 and receive the rank's share, added to what they
  // hold when `accumulate` is set.
  int ag_rank;
  int accumulate;
  // One ring step (kv_chunk >= 0, with ag_rank the query rank): only the K/V tiles
  // of chunk kv_chunk take part.  dK/dV hold that chunk's c rows per (b, g), and dQ
  // is float32 (the rank's rows), overwritten or added to like dK/dV.
  int kv_chunk;
  // packed sequences (ring mode): first / last natural position of each position's
  // document per batch row, [B][T]; nullptr for plain causal attention
  const int* doc_lo;
  const int* doc_hi;
  // packed: (batch row, tile) entries b * (T/128) + tile in decreasing work, for the
  // dQ kernel's query tiles and the dK/dV kernel's key tiles
  const int* ord_q;
  const int* ord_k;
  // test hook: kFaultDkdv / kFaultDq make that kernel's producer withhold its first
  // query-side load, so the bounded waits on it run out (50 ms under any hook value)
  int debug_fault;
  // dQ kernel: an item counter, zero at launch, from which the CTAs claim their
  // items in the heaviest-first order (nullptr: each CTA takes a fixed share)
  int* claim;
};

// Query tiles of rank r at positions >= kpos0 (chunk bounds and kpos0 lie on the
// 128-token grid).
__device__ __forceinline__ int rank_tiles_from(const SeqMap& m, int r, int kpos0) {
  auto part = [&](int p0, int len) {
    const int lo = p0 > kpos0 ? p0 : kpos0;
    return lo < p0 + len ? (p0 + len - lo) >> 7 : 0;
  };
  if (!m.zz) return part(r * m.c, m.c);
  return part(r * m.h, m.h) + part((2 * m.cp - 1 - r) * m.h, m.h);
}

// Tile pairs on the same 128-position grid (see the forward kernel): plain causal
// without documents (lo_row nullptr); with packed documents also empty when every
// key lies before the first query's document and full only when every key lies in
// the last query's document.
__device__ __forceinline__ int classify(int qpos0, int kpos0, const int* lo_row) {
  if (kpos0 > qpos0 + kTile - 1) return kEmpty;
  if (lo_row == nullptr) return kpos0 + kTile - 1 <= qpos0 ? kFull : kDiag;
  if (kpos0 + kTile - 1 < lo_row[qpos0]) return kEmpty;
  return kpos0 + kTile - 1 <= qpos0 && kpos0 >= lo_row[qpos0 + kTile - 1] ? kFull : kDiag;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t par, volatile int* abort,
                                          int* status, uint64_t tmo) {
  bool ok = mbar_wait(bar, par, abort, status, tmo);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t par) {
  int never = 0;
  return mbar_wait(bar, par, &never, nullptr, kDrainTimeoutNs);
}

// Store 32 consecutive fp32 values (times `mul`) of one row as bf16.
__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32],
                                                 float mul) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 w;
    w.x = pack_bf16(__uint_as_float(v[8 * j + 0]) * mul, __uint_as_float(v[8 * j + 1]) * mul);
    w.y = pack_bf16(__uint_as_float(v[8 * j + 2]) * mul, __uint_as_float(v[8 * j + 3]) * mul);
    w.z = pack_bf16(__uint_as_float(v[8 * j + 4]) * mul, __uint_as_float(v[8 * j + 5]) * mul);
    w.w = pack_bf16(__uint_as_float(v[8 * j + 6]) * mul, __uint_as_float(v[8 * j + 7]) * mul);
    d4[j] = w;
  }
}

// The same with two 32-byte stores (dst 32-byte aligned).
__device__ __forceinline__ void store_row32_bf16_v8(__nv_bfloat16* dst, const uint32_t (&v)[32],
                                                    float mul) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      w[j] = pack_bf16(__uint_as_float(v[16 * h + 2 * j]) * mul,
                       __uint_as_float(v[16 * h + 2 * j + 1]) * mul);
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * h),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7])
                 : "memory");
  }
}

// ===========================================================================
// dK / dV
// ===========================================================================
template <int D>
struct DkdvSmem {
  // K and V stationary.  Q and dO in rings of their own, each stage with its
  // per-query statistics (-LSE log2e with Q, -Delta with dO): Q has the extra stage
  // because S^T, its first reader, runs a tile ahead of everything else.  No
  // alignment slack: the kernel declares its dynamic shared memory 1024-byte
  // aligned and checks it.
  static constexpr int kQStages = 3;
  static constexpr int kDOStages = 2;
  static constexpr int kTB = kTile * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kTB;
  static constexpr int kQ = 2 * kTB;
  static constexpr int kDO = kQ + kQStages * kTB;
  static constexpr int kLse = kDO + kDOStages * kTB;
  static constexpr int kDelta = kLse + kQStages * 512;
  static constexpr int kBar = kDelta + kDOStages * 512;
  // kv_full, q_full[QS], q_empty[QS], do_full[DS], do_empty[DS], s_full, s_free,
  // dp_full, p_full, ds_full, final (gradient issuer), final_s (S^T issuer),
  // s_issued, dp_issued
  static constexpr int kNumBars = 1 + 2 * kQStages + 2 * kDOStages + 9;
  static constexpr int kMisc = kBar + kNumBars * 8;
  // TMEM address, abort flag, then the first query position of each Q stage's tile
  static constexpr int kQPos = kMisc + 8;
  static constexpr int kBytes = kQPos + 4 * kQStages + 4;
};

template <int D, bool AG, bool PK>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                const Params p) {
  using L = DkdvSmem<D>;
  constexpr int QS = L::kQStages, DS = L::kDOStages;
  // a dQ kernel launched as this grid's programmatic dependent may start once every
  // CTA of this grid has started (it reads nothing that this kernel writes)
  griddep_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the layout has no alignment slack
    if (threadIdx.x == 0) latch_status(p.status, kStatusLaunch);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBar;
  const uint32_t kv_full = bars;
  auto q_full = [&](int s) { return bars + 8 * (1 + s); };
  auto q_empty = [&](int s) { return bars + 8 * (1 + QS + s); };
  auto do_full = [&](int s) { return bars + 8 * (1 + 2 * QS + s); };
  auto do_empty = [&](int s) { return bars + 8 * (1 + 2 * QS + DS + s); };
  const uint32_t s_full = bars + 8 * (1 + 2 * QS + 2 * DS);
  const uint32_t s_free = s_full + 8;
  const uint32_t dp_full = s_full + 16;
  const uint32_t p_full = s_full + 24;
  const uint32_t ds_full = s_full + 32;
  const uint32_t final_bar = s_full + 40;  // every MMA of the gradient issuer done
  const uint32_t final_s = s_full + 48;
  // issue order (plain arrivals once a product's MMAs are queued): S^T(t+1) goes in
  // behind dP^T(t), dP^T(t+1) behind S^T(t+1)
  const uint32_t s_issued = s_full + 56;
  const uint32_t dp_issued = s_full + 64;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  volatile int* stage_qpos = reinterpret_cast<volatile int*>(smem + L::kQPos);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = p.debug_fault ? kDebugTimeoutNs : kTimeoutNs;
  // row extents of the tensors (for the bounds checks of a CPATTN_DEBUG build): q,
  // k/v, and dO / the statistics / dQ (the rank's rows only in all-gather mode)
  const int64_t q_rows = (int64_t)p.B * p.Hq * p.T, kv_rows = (int64_t)p.B * p.Hkv * p.T;
  const int64_t s_rows = p.ag_rank >= 0 ? (int64_t)p.B * p.Hq * p.m.c : q_rows;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) {
      const uint32_t b = bars + 8 * i;
      mbar_init(b, (b == s_free || b == p_full || b == ds_full) ? 256 : 1);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // work item: kv tiles with the earliest positions (the most queries) first
  int ti, b, g;
  if constexpr (PK) {
    // packed: key tiles in decreasing work, every K/V head of a (batch row, tile) together
    const int nt = p.T >> 7;
    const int ent = p.ord_k[blockIdx.x / p.Hkv];
    g = blockIdx.x - (blockIdx.x / p.Hkv) * p.Hkv;
    b = ent / nt;
    ti = ent - b * nt;
  } else {
    const int units = p.B * p.Hkv;
    ti = blockIdx.x / units;
    const int rem = blockIdx.x - ti * units;
    b = rem / p.Hkv;
    g = rem - (rem / p.Hkv) * p.Hkv;
  }
  // one ring step: tile ti of chunk kv_chunk in slot order (its earliest positions
  // first); otherwise the tile at natural position ti * 128
  const bool step = AG && p.kv_chunk >= 0;
  const int kslot0 = step ? p.kv_chunk * p.m.c + ti * kTile : p.m.slot(ti * kTile);
  const int kpos0 = step ? p.m.pos(kslot0) : ti * kTile;
  const int s_own = kslot0 / p.m.c;
  // query tiles in the order the chunk's gradient travels the ring back to its
  // owner: ranks s, s+1, ..., s-1; every query head of the group per rank; tiles
  // that cannot see this K/V tile are skipped (by the producer's walk, which the
  // other roles follow)
  // packed sequences only in the PK instantiation, so the plain path keeps its code
  const int* lo_row = PK ? p.doc_lo + (int64_t)b * p.T : nullptr;
  // packed: the query tiles from this one up to the tile holding the end of its last
  // key's document, in natural order (every head of the group in turn)
  using Walk = std::conditional_t<PK, NatWalk, TileWalk>;
  const int pk_last = PK ? p.doc_hi[(int64_t)b * p.T + kpos0 + kTile - 1] >> 7 : 0;
  // Only the producer walks; it jumps over the hidden query tiles (see
  // TileWalk::settle_queries) and writes each tile's first query position next to its
  // Q stage.  The other roles count: every query tile at or after this K/V tile's
  // position sees it, once per query head of the group.
  auto walk_start = [&](Walk& w) {
    if constexpr (PK) {
      w.start(p.m, kpos0 >> 7, pk_last, p.n_rep);
    } else {
      if (AG) w.start(p.m, p.ag_rank, 1, +1, p.n_rep);  // all-gather: one rank's queries
      else w.start(p.m, s_own, p.m.cp, +1, p.n_rep);
      w.settle_queries(kpos0);
    }
  };
  auto walk_next = [&](Walk& w) {
    w.next();
    if constexpr (!PK) w.settle_queries(kpos0);
  };
  const int n_tiles =
      PK ? p.n_rep * (pk_last - (kpos0 >> 7) + 1)
         : p.n_rep * (AG ? rank_tiles_from(p.m, p.ag_rank, kpos0) : (p.T - kpos0) >> 7);

  if (warp < 4) {
  regs_ctl();  // warpgroup 0: TMA producer (warp 0) and MMA issuers (warps 1, 2, 3)
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const int krow = (b * p.Hkv + g) * p.T + kslot0;
      mbar_expect_tx(kv_full, 2 * L::kTB);
      if (in_bounds(krow, kTile, kv_rows, p.status))
        for (int kb = 0; kb < D / 64; ++kb) {
          tma_load_2d(sbase + L::kK + kb * (kTile * 128), &tm_k, kb * 64, krow, kv_full);
          tma_load_2d(sbase + L::kV + kb * (kTile * 128), &tm_v, kb * 64, krow, kv_full);
        }
      StageRing<QS> qr;
      StageRing<DS> dr;
      bool first = true;
      Walk wk;
      for (walk_start(wk); !wk.done(); walk_next(wk)) {
        const int qbh = b * p.Hq + g * p.n_rep + wk.rep;
        const int qrow = qbh * p.T + wk.slot();
        // rows of dO and of the statistics (the rank's own rows in all-gather mode)
        const int srow = AG ? qbh * p.m.c + (wk.slot() - p.ag_rank * p.m.c) : qrow;
        if (!mbar_wait(q_empty(qr.stage), qr.par ^ 1, abort, p.status, tmo)) break;
        stage_qpos[qr.stage] = wk.pos();  // published by the arrival below
        // fault hook: the first Q tile never arrives, so the waits on it run out
        if (!(p.debug_fault == kFaultDkdv && first)) {
          mbar_expect_tx(q_full(qr.stage), L::kTB + 512);
          if (in_bounds(qrow, kTile, q_rows, p.status) && in_bounds(srow, kTile, s_rows, p.status)) {
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_2d(sbase + L::kQ + qr.stage * L::kTB + kb * (kTile * 128), &tm_q, kb * 64,
                          qrow, q_full(qr.stage));
            bulk_load(sbase + L::kLse + qr.stage * 512, p.lse2 + srow, 512, q_full(qr.stage));
          }
          qr.mark_issued();
        }
        first = false;
        if (!mbar_wait(do_empty(dr.stage), dr.par ^ 1, abort, p.status, tmo)) break;
        mbar_expect_tx(do_full(dr.stage), L::kTB + 512);
        if (in_bounds(srow, kTile, s_rows, p.status)) {
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_2d(sbase + L::kDO + dr.stage * L::kTB + kb * (kTile * 128), &tm_do, kb * 64,
                        srow, do_full(dr.stage));
          bulk_load(sbase + L::kDelta + dr.stage * 512, p.delta + srow, 512, do_full(dr.stage));
        }
        dr.mark_issued();
        qr.advance();
        dr.advance();
      }
      drain_wait(kv_full, 0);
      for (int s = 0; s < QS; ++s)
        if (qr.was_issued(s)) drain_wait(q_full(s), qr.issued_parity(s));
      for (int s = 0; s < DS; ++s)
        if (dr.was_issued(s)) drain_wait(do_full(s), dr.issued_parity(s));
    }
  } else if (warp == 1) {
    {
      // S^T = K Q^T issuer (SS, K-major).  Issuing a tcgen05.mma that runs 64
      // cycles at N = 128 takes its thread tens of cycles, and the thread's next
      // memory access after a tcgen05.commit waits for the committed MMAs, so S^T
      // has a warp of its own and the gradient warp (warp 2) issues dP^T, dV and dK.
      // The whole warp runs the loop (warp-uniform descriptors); one elected lane
      // issues.
      const bool leader = elect_one();
      constexpr uint32_t kIdSS = idesc_bf16(128, 128, false, false);
      bool ok = warp_wait(kv_full, 0, abort, p.status, tmo);
      tc_fence_after();
      constexpr uint32_t kTD = L::kTB >> 4;
      const uint64_t kd = sdesc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t qd0 = sdesc_sw128(sbase + L::kQ, 16, 1024);
      StageRing<QS> qr;
      int cnt = 0;
      for (int t = 0; t < n_tiles && ok; ++t) {
        // The tensor pipe runs MMAs in the order they are queued.  The gradient warp
        // queues ... dV(t-1), dK(t-1), dP^T(t) back to back; S^T(t+1) goes in behind
        // dP^T(t), where it runs while the compute warps turn dP^T(t) into P^T(t).
        // The two warps wait for each other's previous product to be queued
        // (S^T(t+1) after dP^T(t), dP^T(t+1) after S^T(t+1)), which keeps the two
        // arrival barriers in lockstep.
        if (cnt > 0 && !(ok = warp_wait(dp_issued, (cnt - 1) & 1, abort, p.status, tmo))) break;
        if (!(ok = warp_wait(q_full(qr.stage), qr.par, abort, p.status, tmo))) break;
        // the S region is free once the compute warps have loaded the previous S^T
        if (cnt > 0 && !(ok = warp_wait(s_free, (cnt - 1) & 1, abort, p.status, tmo))) break;
        tc_fence_after();
        const uint64_t qd = qd0 + (uint64_t)(qr.stage * kTD);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;
          if (leader) mma_ss(tmem, kd + off, qd + off, kIdSS, kk > 0);
        }
        if (leader) {
          mbar_arrive(s_issued);  // before the commit, so it does not wait
          mma_commit(s_full);
        }
        __syncwarp();
        ++cnt;
        qr.advance();
      }
      if (leader) mma_commit(final_s);
      __syncwarp();
      drain_wait(final_s, 0);
    }
  } else if (warp == 2) {
    {
      // Gradient warp: dP^T = V dO^T (SS, K-major) into the dP region, then
      // dV += P^T dO and dK += dS^T Q (TS: P^T and dS^T stored over dP^T, Q / dO
      // MN-major), queued per tile as dV(t), dK(t), dP^T(t+1).  dP^T(t+1)
      // overwrites what dV(t) and dK(t) read, which is safe because one thread's
      // MMAs run in issue order, so it follows dK(t) without a round trip through
      // an mbarrier.  The operands of dK(t) and dP^T(t+1) are waited for before the
      // commits of tile t: a thread's first mbarrier access after a commit waits for
      // the committed MMAs.
      const bool leader = elect_one();
      constexpr uint32_t kIdSS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdTS = idesc_bf16(128, D, false, true);
      constexpr uint32_t kTD = L::kTB >> 4;
      const uint64_t vd = sdesc_sw128(sbase + L::kV, 16, 1024);
      const uint64_t dod_k0 = sdesc_sw128(sbase + L::kDO, 16, 1024);
      const uint64_t qd_mn0 = sdesc_sw128(sbase + L::kQ, kTile * 128, 1024);
      const uint64_t dod_mn0 = sdesc_sw128(sbase + L::kDO, kTile * 128, 1024);
      bool ok = warp_wait(kv_full, 0, abort, p.status, tmo);
      tc_fence_after();
      StageRing<QS> qr;   // Q stage of tile t
      StageRing<DS> dr;   // dO stage of tile t
      StageRing<DS> dpr;  // dO stage of the next dP^T
      auto issue_dp = [&]() {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;
          if (leader)
            mma_ss(tmem + 128, vd + off, dod_k0 + (uint64_t)(dpr.stage * kTD) + off, kIdSS,
                   kk > 0);
        }
        if (leader) {
          mbar_arrive(dp_issued);
          mma_commit(dp_full);
        }
        __syncwarp();
        dpr.advance();
      };
      // dP^T(0), behind S^T(0)
      if (ok && n_tiles > 0 && (ok = warp_wait(do_full(dpr.stage), dpr.par, abort, p.status, tmo)) &&
          (ok = warp_wait(s_issued, 0, abort, p.status, tmo))) {
        tc_fence_after();
        issue_dp();
      }
      for (int t = 0; ok && t < n_tiles; ++t) {
        // dV(t) += P^T(t) dO(t)  (dO landed before dP^T(t) was issued)
        if (!(ok = warp_wait(p_full, t & 1, abort, p.status, tmo))) break;
        tc_fence_after();
        const uint64_t dod = dod_mn0 + (uint64_t)(dr.stage * kTD);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t acol = 128 + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
          if (leader)
            mma_ts(tmem + 256, tmem + acol, dod + kk * 128, kIdTS, (t > 0 || kk > 0) ? 1u : 0u);
        }
        // dK(t) += dS^T(t) Q(t) (Q landed before S^T(t)); dO(t+1) landed and S^T(t+1)
        // queued for dP^T(t+1)
        const bool more = t + 1 < n_tiles;
        if (!(ok = warp_wait(ds_full, t & 1, abort, p.status, tmo))) break;
        if (more && !(ok = warp_wait(do_full(dpr.stage), dpr.par, abort, p.status, tmo))) break;
        if (more && !(ok = warp_wait(s_issued, (t + 1) & 1, abort, p.status, tmo))) break;
        tc_fence_after();
        const uint64_t qd = qd_mn0 + (uint64_t)(qr.stage * kTD);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t acol = 128 + 32 + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
          if (leader)
            mma_ts(tmem + 256 + D, tmem + acol, qd + kk * 128, kIdTS,
                   (t > 0 || kk > 0) ? 1u : 0u);
        }
        if (leader) {
          // every read of tile t's Q and dO stages is issued: S^T(t) and dP^T(t)
          // completed before the compute warps released p_full / ds_full, by which
          // they also hold the stages' statistics
          mma_commit(do_empty(dr.stage));
          mma_commit(q_empty(qr.stage));
        }
        __syncwarp();
        if (more) issue_dp();
        qr.advance();
        dr.advance();
      }
      if (leader) mma_commit(final_bar);
      __syncwarp();
      drain_wait(final_bar, 0);
    }
  }
  } else {
    regs_math();  // warpgroups 1 and 2: softmax / gradient math
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int row = quad * 32 + lane;  // key row of the tile
    // packed: this key is seen by the queries up to its document's last position
    const int hi_k = PK ? p.doc_hi[(int64_t)b * p.T + kpos0 + row] : p.T;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + half * 64;
    const uint32_t t_dp = tmem + lane_off + 128 + half * 64;
    const float* lse_s = reinterpret_cast<const float*>(smem + L::kLse);
    const float* del_s = reinterpret_cast<const float*>(smem + L::kDelta);
    StageRing<QS> qr;
    StageRing<DS> dr;
    int cnt = 0;
    bool ok = true;
    // packed: the query tiles form one natural range (nothing hidden), walked here
    Walk wk;
    if constexpr (PK) walk_start(wk);
    for (int t = 0; t < n_tiles; ++t) {
      int qpos0;
      if constexpr (PK) {
        qpos0 = wk.pos();
        walk_next(wk);
      }
      if (!(ok = warp_wait(q_full(qr.stage), qr.par, abort, p.status, tmo))) break;  // -LSE log2e landed
      if constexpr (!PK) qpos0 = stage_qpos[qr.stage];
      const int cls = classify(qpos0, kpos0, lo_row);
      const float* lse_t = lse_s + qr.stage * 128 + half * 64;
      const float* del_t = del_s + dr.stage * 128 + half * 64;
      // this half's 64 per-query LSE values, fetched while S^T is still being computed
      float4 nl4[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) nl4[i] = reinterpret_cast<const float4*>(lse_t)[i];
      if (!(ok = warp_wait(s_full, cnt & 1, abort, p.status, tmo))) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(t_s, sr[0]);
      tmem_ld32(t_s + 32, sr[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_free);  // S^T is in registers: the S region may take the next S^T
      // query column j (of this half) sees this key row iff kpos0 + row <= qpos0 + 64*half + j
      const int thr = kpos0 + row - qpos0 - half * 64;
      // packed: query column j is also hidden past the key's document end
      const int thr_hi = hi_k - qpos0 - half * 64;
      float pr[64];
      const float2 sl2v = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int j0 = c * 32 + j;
          // P = 2^(S scale log2e - LSE log2e), the exponent argument two lanes at a time
          const float4 n4 = nl4[j0 >> 2];
          const float2 nl = (j0 & 2) ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y);
          const float2 x = fma2(make_float2(__uint_as_float(sr[c][j]), __uint_as_float(sr[c][j + 1])),
                                sl2v, nl);
          float p0 = ex2(x.x), p1 = ex2(x.y);
          if (cls == kDiag) {
            if (j0 < thr || (PK && j0 > thr_hi)) p0 = 0.f;
            if (j0 + 1 < thr || (PK && j0 + 1 > thr_hi)) p1 = 0.f;
          }
          pr[j0] = p0;
          pr[j0 + 1] = p1;
        }
      // -Delta of this half's 64 queries (it travels with dO), fetched before dP^T is ready
      if (!(ok = warp_wait(do_full(dr.stage), dr.par, abort, p.status, tmo))) break;
      float4 nd4[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) nd4[k] = reinterpret_cast<const float4*>(del_t)[k];
      if (!(ok = warp_wait(dp_full, cnt & 1, abort, p.status, tmo))) break;
      tc_fence_after();
      tmem_ld32(t_dp, sr[0]);
      tmem_ld32(t_dp + 32, sr[1]);
      tmem_wait_ld();
      // P^T (bf16) over the first 32 columns of this half's dP^T, already in
      // registers, so the dV product can start while dS is formed
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) pk[j >> 1] = pack_bf16(pr[c * 32 + j], pr[c * 32 + j + 1]);
        tmem_st16(t_dp + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int j0 = c * 32 + j;
          // dS = P (dP - Delta), two lanes per instruction (del_t holds -Delta)
          const float4 d4 = nd4[j0 >> 2];
          const float2 nd = (j0 & 2) ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
          const float2 d = mul2(make_float2(pr[j0], pr[j0 + 1]),
                                add2(make_float2(__uint_as_float(sr[c][j]),
                                                 __uint_as_float(sr[c][j + 1])), nd));
          pk[j >> 1] = pack_bf16(d.x, d.y);
        }
        // dS^T (bf16) over the next 32 columns of this half's dP^T
        tmem_st16(t_dp + 32 + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_full);
      ++cnt;
      qr.advance();
      dr.advance();
    }
    if (ok && cnt > 0) ok = warp_wait(final_bar, 0, abort, p.status, tmo);
    // (the TMEM loads below are warp-collective: only the global stores are guarded)
    // one ring step: the chunk's own c rows per (b, g)
    const int64_t orow = step ? ((int64_t)b * p.Hkv + g) * p.m.c + (kslot0 - p.kv_chunk * p.m.c) + row
                              : ((int64_t)b * p.Hkv + g) * p.T + kslot0 + row;
    const bool store = in_bounds(orow, 1, step ? (int64_t)p.B * p.Hkv * p.m.c : kv_rows, p.status);
    if (ok && AG && D == 128 && (cnt > 0 || !p.accumulate)) {
      // all-gather / ring step: float32 share of this rank's queries.  This thread's
      // 64 columns of its row are two 128-byte lines of each of dK and dV.  The warp
      // stages them in shared memory (the Q and dO stages, idle once the walk is
      // done) as four 32-row x 32-column boxes in the tensor maps' 128-byte swizzle
      // (chunk a of row i at slot a ^ (i & 7)), and one TMA operation per box adds
      // them into the sums (or stores them, for the first share) in L2, with no load
      // on the SM.  Each element receives one addition per launch.
      tc_fence_after();
      const uint32_t stage = sbase + L::kQ + (warp - 4) * 16384;
      float4* st4 = reinterpret_cast<float4*>(smem + L::kQ + (warp - 4) * 16384);
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK (times the scale)
        const float mul = which ? p.scale : 1.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v32[32];
          if (cnt > 0) {
            tmem_ld32(tmem + lane_off + 256 + which * D + half * 64 + c * 32, v32);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v32[j] = 0u;
          }
#pragma unroll
          for (int a = 0; a < 8; ++a)
            st4[which * 512 + c * 256 + lane * 8 + (a ^ (lane & 7))] =
                make_float4(__uint_as_float(v32[4 * a]) * mul, __uint_as_float(v32[4 * a + 1]) * mul,
                            __uint_as_float(v32[4 * a + 2]) * mul,
                            __uint_as_float(v32[4 * a + 3]) * mul);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int64_t orow0 = orow - row;  // the tile's first row
      if (lane == 0 &&
          in_bounds(orow0, kTile, step ? (int64_t)p.B * p.Hkv * p.m.c : kv_rows, p.status)) {
        const int y = (int)(orow0 + quad * 32);
#pragma unroll
        for (int which = 0; which < 2; ++which)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const CUtensorMap* map = which ? &tm_dk : &tm_dv;
            const uint32_t box = stage + which * 8192 + c * 4096;
            if (p.accumulate) tma_reduce_add_2d(map, half * 64 + c * 32, y, box);
            else tma_store_2d(map, half * 64 + c * 32, y, box);
          }
        bulk_commit_group();
        bulk_wait_all();  // the CTA's shared memory is released when it ends
      }
    } else if (ok && AG) {
      // all-gather: float32 share of this rank's queries, added to the sum so far
      tc_fence_after();
      float* dkf = static_cast<float*>(p.out0) + orow * D + half * (D / 2);
      float* dvf = static_cast<float*>(p.out1) + orow * D + half * (D / 2);
      if (cnt > 0 || !p.accumulate) {
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          for (int which = 0; which < 2; ++which) {
            uint32_t v32[32];
            if (cnt > 0) {
              tmem_ld32(tmem + lane_off + 256 + which * D + half * (D / 2) + c * 32, v32);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) v32[j] = 0u;
            }
            const float mul = which ? p.scale : 1.f;
            float4* dst = reinterpret_cast<float4*>((which ? dkf : dvf) + c * 32);
#pragma unroll
            for (int j = 0; j < 8 && store; ++j) {
              float4 x = make_float4(__uint_as_float(v32[4 * j]) * mul,
                                     __uint_as_float(v32[4 * j + 1]) * mul,
                                     __uint_as_float(v32[4 * j + 2]) * mul,
                                     __uint_as_float(v32[4 * j + 3]) * mul);
              if (p.accumulate) {
                const float4 y = dst[j];
                x.x += y.x;
                x.y += y.y;
                x.z += y.z;
                x.w += y.w;
              }
              dst[j] = x;
            }
          }
        }
      }
    } else if (ok && !AG && D == 128) {
      // bf16 dK and dV: this thread's 64 columns of its row are one 128-byte line of
      // each.  The warp's lines go through shared memory (the Q stages, idle once the
      // walk is done: chunk a of line i at slot a ^ (i & 7)) so that they leave as
      // whole boxes instead of stores that touch 32 lines each.
      tc_fence_after();
      uint4* st4 = reinterpret_cast<uint4*>(smem + L::kQ + (warp - 4) * 8192);
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK (times the scale)
        const float mul = which ? p.scale : 1.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v32[32];
          if (cnt > 0) {
            tmem_ld32(tmem + lane_off + 256 + which * D + half * 64 + c * 32, v32);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v32[j] = 0u;
          }
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const int ca = c * 4 + a;  // 16-byte chunk of the line
            st4[which * 256 + lane * 8 + (ca ^ (lane & 7))] = make_uint4(
                pack_bf16(__uint_as_float(v32[8 * a]) * mul, __uint_as_float(v32[8 * a + 1]) * mul),
                pack_bf16(__uint_as_float(v32[8 * a + 2]) * mul, __uint_as_float(v32[8 * a + 3]) * mul),
                pack_bf16(__uint_as_float(v32[8 * a + 4]) * mul, __uint_as_float(v32[8 * a + 5]) * mul),
                pack_bf16(__uint_as_float(v32[8 * a + 6]) * mul, __uint_as_float(v32[8 * a + 7]) * mul));
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      // the two areas are 32 x 64 boxes of dV and dK in the tensor maps' 128-byte
      // swizzle: one TMA store each
      const int64_t orow0 = orow - row;  // the tile's first row
      if (lane == 0 &&
          in_bounds(orow0, kTile, step ? (int64_t)p.B * p.Hkv * p.m.c : kv_rows, p.status)) {
        const uint32_t stage = sbase + L::kQ + (warp - 4) * 8192;
        tma_store_2d(&tm_dv, half * 64, (int)(orow0 + quad * 32), stage);
        tma_store_2d(&tm_dk, half * 64, (int)(orow0 + quad * 32), stage + 4096);
        bulk_commit_group();
        bulk_wait_all();  // the CTA's shared memory is released when it ends
      }
    } else if (ok) {
      tc_fence_after();
      __nv_bfloat16* dk = static_cast<__nv_bfloat16*>(p.out0) + orow * D + half * (D / 2);
      __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(p.out1) + orow * D + half * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v32[32];
        if (cnt > 0) {
          tmem_ld32(tmem + lane_off + 256 + half * (D / 2) + c * 32, v32);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v32[j] = 0u;
        }
        if (store) store_row32_bf16(dv + c * 32, v32, 1.f);
        if (cnt > 0) {
          tmem_ld32(tmem + lane_off + 256 + D + half * (D / 2) + c * 32, v32);
          tmem_wait_ld();
        }
        if (store) store_row32_bf16(dk + c * 32, v32, p.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// dQ
// ===========================================================================
template <int D>
struct DqSmem {
  // K and V have separate rings: V is last read by dP (early in a tile), K by dQ
  // (late), so each is refilled as soon as its own consumer is done, and K gets
  // the extra stage that the freed shared memory allows.
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kTB = kTile * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kDO = kTB;
  static constexpr int kK = 2 * kTB;
  static constexpr int kV = kK + kKStages * kTB;
  static constexpr int kBar = kV + kVStages * kTB;
  // qdo_full, qdo_empty (released by the S and the dP issuer), k_full[KS], k_empty[KS],
  // v_full[VS], v_empty[VS], s_full, s_free, dp_full[2], ds_full[2] (one per dP
  // buffer), dq_done[2], dq_free, final_q (dQ issuer), final_s (S issuer), final_p
  // (dP issuer), item_full[IS], item_empty[IS]
  static constexpr int kItemSlots = 4;  // claimed items passed from the producer to the other roles
  static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 12 + 2 * kItemSlots;
  static constexpr int kMisc = kBar + kNumBars * 8;
  // TMEM address, abort flag, then the item slots
  static constexpr int kItems = kMisc + 16;
  static constexpr int kBytes = kItems + 4 * kItemSlots + 1024;
};

// One work item of the dQ kernel: a 128-row query tile of one (batch, head), the
// latest query positions (the most keys) first.
struct DqItem {
  int b, h, g, qpos0, qslot0, r_own;
  int64_t qrow;  // row of q
  int64_t srow;  // row of dO, the statistics and dQ (the rank's own rows in all-gather mode)
  int kv_row_base;
};

template <int D, bool PK>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const Params p) {
  using L = DqSmem<D>;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  constexpr int kDqCol = 384;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBar;
  const uint32_t qdo_full = bars;
  const uint32_t qdo_empty = bars + 8;
  auto k_full = [&](int s) { return bars + 8 * (2 + s); };
  auto k_empty = [&](int s) { return bars + 8 * (2 + KS + s); };
  auto v_full = [&](int s) { return bars + 8 * (2 + 2 * KS + s); };
  auto v_empty = [&](int s) { return bars + 8 * (2 + 2 * KS + VS + s); };
  const uint32_t s_full = bars + 8 * (2 + 2 * KS + 2 * VS);
  const uint32_t s_free = s_full + 8;
  // per-buffer barriers: a second arrival on a buffer's barrier needs that buffer
  // to have been recycled, so no waiter can ever be two phases behind
  auto dp_full = [&](int x) { return s_full + 16 + 8 * x; };
  auto ds_full = [&](int x) { return s_full + 32 + 8 * x; };
  auto dq_done = [&](int x) { return s_full + 48 + 8 * x; };
  const uint32_t dq_free = s_full + 64;
  const uint32_t final_q = s_full + 72;
  const uint32_t final_s = s_full + 80;
  const uint32_t final_p = s_full + 88;
  constexpr int IS = L::kItemSlots;
  auto item_full = [&](int s) { return s_full + 96 + 8 * s; };
  auto item_empty = [&](int s) { return s_full + 96 + 8 * (IS + s); };
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::kItems);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = p.debug_fault ? kDebugTimeoutNs : kTimeoutNs;
  // row extents of the tensors (for the bounds checks of a CPATTN_DEBUG build): q,
  // k/v, and dO / the statistics / dQ (the rank's rows only in all-gather mode)
  const int64_t q_rows = (int64_t)p.B * p.Hq * p.T, kv_rows = (int64_t)p.B * p.Hkv * p.T;
  const int64_t s_rows = p.ag_rank >= 0 ? (int64_t)p.B * p.Hq * p.m.c : q_rows;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) {
      const uint32_t b = bars + 8 * i;
      const bool compute_arrivals = b == s_free || b == ds_full(0) || b == ds_full(1) || b == dq_free;
      // an item slot is released by one lane of each of the 11 warps other than the producer's
      const bool slot_release = b >= item_empty(0) && b < item_empty(IS);
      mbar_init(b, compute_arrivals ? 256 : b == qdo_empty ? 2 : slot_release ? 11 : 1);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Persistent: the CTAs stay resident and walk the items (latest query positions
  // first) in the order item_of gives; every pipeline keeps running across items.
  // all-gather mode: the rank's c/128 query tiles per (b, h); else all T/128
  const bool ag = p.ag_rank >= 0;
  const int n_q_tiles = (ag ? p.m.c : p.T) / kTile;
  const int n_items = p.B * p.Hq * n_q_tiles;
  auto decode = [&](int w) {
    DqItem it;
    const int units = p.B * p.Hq;
    int ti;
    if constexpr (PK) {
      // packed: items in decreasing work, every head of a (batch row, tile) together
      const int nt = p.T >> 7;
      const int ent = p.ord_q[w / p.Hq];
      it.b = ent / nt;
      it.h = w - (w / p.Hq) * p.Hq;
      ti = n_q_tiles - 1 - (ent - it.b * nt);  // the tile below is n_q_tiles - 1 - ti
    } else {
      ti = w / units;
      const int rem = w - ti * units;
      it.b = rem / p.Hq;
      it.h = rem - it.b * p.Hq;
    }
    it.g = it.h / p.n_rep;
    const int64_t bh = (int64_t)it.b * p.Hq + it.h;
    if (ag) {
      // the rank's later slots hold its later positions: heaviest first
      it.qslot0 = p.ag_rank * p.m.c + (n_q_tiles - 1 - ti) * kTile;
      it.qpos0 = p.m.pos(it.qslot0);
      it.srow = bh * p.m.c + (it.qslot0 - p.ag_rank * p.m.c);
    } else {
      it.qpos0 = (n_q_tiles - 1 - ti) * kTile;
      it.qslot0 = p.m.slot(it.qpos0);
      it.srow = bh * p.T + it.qslot0;
    }
    it.r_own = it.qslot0 / p.m.c;
    it.qrow = bh * p.T + it.qslot0;
    it.kv_row_base = (it.b * p.Hkv + it.g) * p.T;
    return it;
  };
  // K/V tiles of an item in ring order (chunks r, r-1, ...), hidden tiles skipped
  auto doc_row = [&](const DqItem& it) -> const int* {
    return PK ? p.doc_lo + (int64_t)it.b * p.T : nullptr;
  };
  // packed: the key tiles from the one holding the first row's document start up to
  // the diagonal, in natural order
  using Walk = std::conditional_t<PK, NatWalk, TileWalk>;
  auto walk_start = [&](Walk& w, const DqItem& it) {
    if constexpr (PK) {
      w.start(p.m, doc_row(it)[it.qpos0] >> 7, it.qpos0 >> 7, 1);
    } else {
      // ring order from the rank's own chunk, or the one chunk of a ring step
      if (p.kv_chunk >= 0) w.start(p.m, p.kv_chunk, 1, -1, 1);
      else w.start(p.m, it.r_own, p.m.cp, -1, 1);
      w.settle_keys(it.qpos0);
    }
  };
  auto walk_next = [&](Walk& w, const DqItem& it) {
    w.next();
    if constexpr (!PK) w.settle_keys(it.qpos0);
  };
  // The k-th item of this CTA.  Fixed shares (no counter): item_of's order.  With the
  // counter, the producer claims the next item (heaviest first over the whole grid,
  // so CTAs that start late, or run slow, simply take fewer) and passes it to the
  // other warps through a ring of shared-memory slots; -1 ends every role's loop.
  const bool claimed = p.claim != nullptr;
  auto claim_item = [&](int k, bool& ok) -> int {  // producer thread
    if (!claimed) return item_of(k, n_items);
    int w = atomicAdd(p.claim, 1);
    if (w >= n_items) w = -1;
    const int s = k % IS;
    if (k >= IS && !(ok = mbar_wait(item_empty(s), ((k / IS) - 1) & 1, abort, p.status, tmo)))
      return -1;
    item_slot[s] = w;
    mbar_arrive(item_full(s));
    return w;
  };
  auto take_item = [&](int k, bool& ok) -> int {  // whole warps
    if (!claimed) return item_of(k, n_items);
    const int s = k % IS;
    if (!(ok = warp_wait(item_full(s), (k / IS) & 1, abort, p.status, tmo))) return -1;
    const int w = item_slot[s];
    __syncwarp();
    if (lane == 0) mbar_arrive(item_empty(s));
    return w;
  };

  if (warp < 4) {
  regs_ctl();  // warpgroup 0: TMA producer (warp 0) and MMA issuers (warps 1, 2, 3)
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      StageRing<KS> kr;
      StageRing<VS> vr;
      int q_last = -1;
      bool ok = true;
      int w;
      for (int k = 0; ok && (w = claim_item(k, ok)) >= 0; ++k) {
        const DqItem it = decode(w);
        // Q and dO of this item once the S and dP issuers are done with the last one's
        if (k > 0 && !(ok = mbar_wait(qdo_empty, (k - 1) & 1, abort, p.status, tmo))) break;
        // fault hook: the first item's Q and dO never arrive, so the waits on them run out
        if (!(p.debug_fault == kFaultDq && k == 0)) {
          mbar_expect_tx(qdo_full, 2 * L::kTB);
          if (in_bounds(it.qrow, kTile, q_rows, p.status) &&
              in_bounds(it.srow, kTile, s_rows, p.status))
          for (int kb = 0; kb < D / 64; ++kb) {
            tma_load_2d(sbase + L::kQ + kb * (kTile * 128), &tm_q, kb * 64, (int)it.qrow, qdo_full);
            tma_load_2d(sbase + L::kDO + kb * (kTile * 128), &tm_do, kb * 64, (int)it.srow,
                        qdo_full);
          }
          q_last = k;
        }
        Walk wk;
        for (walk_start(wk, it); !wk.done(); walk_next(wk, it)) {
          const int row = it.kv_row_base + wk.slot();
          if (!(ok = mbar_wait(k_empty(kr.stage), kr.par ^ 1, abort, p.status, tmo))) break;
          mbar_expect_tx(k_full(kr.stage), L::kTB);
          const bool kv_ok = in_bounds(row, kTile, kv_rows, p.status);
          if (kv_ok)
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_2d(sbase + L::kK + kr.stage * L::kTB + kb * (kTile * 128), &tm_k, kb * 64,
                          row, k_full(kr.stage));
          kr.mark_issued();
          if (!(ok = mbar_wait(v_empty(vr.stage), vr.par ^ 1, abort, p.status, tmo))) break;
          mbar_expect_tx(v_full(vr.stage), L::kTB);
          if (kv_ok)
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_2d(sbase + L::kV + vr.stage * L::kTB + kb * (kTile * 128), &tm_v, kb * 64,
                          row, v_full(vr.stage));
          vr.mark_issued();
          kr.advance();
          vr.advance();
        }
      }
      if (q_last >= 0) drain_wait(qdo_full, q_last & 1);
      for (int s = 0; s < KS; ++s)
        if (kr.was_issued(s)) drain_wait(k_full(s), kr.issued_parity(s));
      for (int s = 0; s < VS; ++s)
        if (vr.was_issued(s)) drain_wait(v_full(s), vr.issued_parity(s));
    }
  } else if (warp == 1 || warp == 3) {
    // One issuer per product: warp 1 S = Q K^T, warp 3 dP = dO V^T, warp 2 dQ.  An
    // issuing thread's next memory access after a tcgen05.commit waits for the
    // committed MMAs, so one thread alternating products would keep a single group
    // in flight and wait on each product's consumers in turn.  Each issuer runs as a
    // whole warp (warp-uniform descriptors) and issues from one elected lane.
    {
      const bool leader = elect_one();
      const bool is_s = warp == 1;
      constexpr uint32_t kIdSS = idesc_bf16(128, 128, false, false);
      // descriptor bases (16-byte units), K-major
      constexpr uint32_t kTD = L::kTB >> 4;
      const uint64_t ad = sdesc_sw128(sbase + (is_s ? L::kQ : L::kDO), 16, 1024);
      const uint64_t bd0 = sdesc_sw128(sbase + (is_s ? L::kK : L::kV), 16, 1024);
      StageRing<KS> kr;
      StageRing<VS> vr;
      int g = 0;  // tiles so far over all items
      bool ok = true;
      int w;
      for (int k = 0; ok && (w = take_item(k, ok)) >= 0; ++k) {
        const DqItem it = decode(w);
        if (!(ok = warp_wait(qdo_full, k & 1, abort, p.status, tmo))) break;
        Walk wk;
        for (walk_start(wk, it); !wk.done(); walk_next(wk, it)) {
          uint32_t dst;
          uint64_t bd;
          if (is_s) {
            // S(g): the S region is free once the compute warps have read S(g-1)
            if (g > 0 && !(ok = warp_wait(s_free, (g - 1) & 1, abort, p.status, tmo))) break;
            if (!(ok = warp_wait(k_full(kr.stage), kr.par, abort, p.status, tmo))) break;
            dst = tmem;
            bd = bd0 + (uint64_t)(kr.stage * kTD);
          } else {
            // dP(g) into buffer g&1: free once dQ(g-2) has read the dS stored there
            if (g >= 2 && !(ok = warp_wait(dq_done(g & 1), ((g - 2) >> 1) & 1, abort, p.status, tmo)))
              break;
            if (!(ok = warp_wait(v_full(vr.stage), vr.par, abort, p.status, tmo))) break;
            dst = tmem + 128 + 128 * (g & 1);
            bd = bd0 + (uint64_t)(vr.stage * kTD);
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;
            if (leader) mma_ss(dst, ad + off, bd + off, kIdSS, kk > 0);
          }
          if (leader) {
            if (is_s) {
              mma_commit(s_full);
            } else {
              mma_commit(dp_full(g & 1));
              mma_commit(v_empty(vr.stage));  // V of this tile is not read again
            }
          }
          __syncwarp();
          kr.advance();
          vr.advance();
          ++g;
        }
        if (!ok) break;
        if (leader) mma_commit(qdo_empty);  // this issuer is done with the item's Q (or dO)
        __syncwarp();
      }
      if (leader) mma_commit(is_s ? final_s : final_p);
      __syncwarp();
      drain_wait(is_s ? final_s : final_p, 0);
    }
  } else if (warp == 2) {
    {
      // Gradient issuer: dQ += dS K (TS: dS in TMEM, K MN-major from shared memory);
      // whole warp, one elected lane issues
      const bool leader = elect_one();
      constexpr uint32_t kIdTS = idesc_bf16(128, D, false, true);
      constexpr uint32_t kTD = L::kTB >> 4;
      const uint64_t kd_mn0 = sdesc_sw128(sbase + L::kK, kTile * 128, 1024);
      StageRing<KS> kr;
      int g = 0;
      bool ok = true;
      int w;
      for (int k = 0; ok && (w = take_item(k, ok)) >= 0; ++k) {
        const DqItem it = decode(w);
        int t = 0;  // tile of this item
        Walk wk;
        for (walk_start(wk, it); !wk.done(); walk_next(wk, it)) {
          if (!(ok = warp_wait(ds_full(g & 1), (g >> 1) & 1, abort, p.status, tmo))) break;
          // the item's first dQ overwrites the accumulator the previous epilogue read
          if (t == 0 && k > 0 && !(ok = warp_wait(dq_free, (k - 1) & 1, abort, p.status, tmo))) break;
          tc_fence_after();
          // K(g) landed before S(g), which the compute warps read before storing dS(g)
          const uint64_t kd_mn = kd_mn0 + (uint64_t)(kr.stage * kTD);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t acol = 128 + 128 * (g & 1) + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
            if (leader)
              mma_ts(tmem + kDqCol, tmem + acol, kd_mn + kk * 128, kIdTS,
                     (t > 0 || kk > 0) ? 1u : 0u);
          }
          if (leader) {
            mma_commit(dq_done(g & 1));  // the dS buffer may take dP(g+2)
            // both S(g) and dQ(g) have read K(g) once dQ(g) completes
            mma_commit(k_empty(kr.stage));
          }
          __syncwarp();
          kr.advance();
          ++g;
          ++t;
        }
      }
      if (leader) mma_commit(final_q);
      __syncwarp();
      drain_wait(final_q, 0);
    }
  }
  } else {
    regs_math();  // warpgroups 1 and 2: softmax / gradient math
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int row = quad * 32 + lane;  // query row of the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + half * 64;
    const float2 sl2v = make_float2(p.scale_log2, p.scale_log2);
    int g = 0;
    bool ok = true;
    int w;
    for (int k = 0; ok && (w = take_item(k, ok)) >= 0; ++k) {
      const DqItem it = decode(w);
      const int* lo_row = doc_row(it);
      const int lo_q = PK ? lo_row[it.qpos0 + row] : 0;  // packed: first key of the document
      const bool row_ok = in_bounds(it.srow + row, 1, s_rows, p.status);
      const float sl = row_ok ? p.lse2[it.srow + row] : 0.f, sd = row_ok ? p.delta[it.srow + row] : 0.f;
      const float2 nl2 = make_float2(sl, sl);  // -LSE log2e
      const float2 ndl = make_float2(sd, sd);  // -Delta
      int cnt = 0;  // tiles of this item
      Walk wk;
      for (walk_start(wk, it); !wk.done(); walk_next(wk, it)) {
        const int kpos0 = wk.pos();
        const int cls = classify(it.qpos0, kpos0, lo_row);
        if (!(ok = warp_wait(s_full, g & 1, abort, p.status, tmo))) break;
        tc_fence_after();
        uint32_t sr[2][32];
        tmem_ld32(t_s, sr[0]);
        tmem_ld32(t_s + 32, sr[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_free);
        // key column j (of this half) is visible iff kpos0 + 64*half + j <= qpos0 + row
        const int thr = it.qpos0 + row - kpos0 - half * 64;
        const int thr_lo = lo_q - kpos0 - half * 64;
        float pr[64];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2) {
            const int j0 = c * 32 + jj;
            const float2 x = fma2(make_float2(__uint_as_float(sr[c][jj]), __uint_as_float(sr[c][jj + 1])),
                                  sl2v, nl2);
            float p0 = ex2(x.x), p1 = ex2(x.y);
            if (cls == kDiag) {
              if (j0 > thr || (PK && j0 < thr_lo)) p0 = 0.f;
              if (j0 + 1 > thr || (PK && j0 + 1 < thr_lo)) p1 = 0.f;
            }
            pr[j0] = p0;
            pr[j0 + 1] = p1;
          }
        if (!(ok = warp_wait(dp_full(g & 1), (g >> 1) & 1, abort, p.status, tmo))) break;
        tc_fence_after();
        const uint32_t t_dp = tmem + lane_off + 128 + 128 * (g & 1) + half * 64;
        tmem_ld32(t_dp, sr[0]);
        tmem_ld32(t_dp + 32, sr[1]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2) {
            const int j0 = c * 32 + jj;
            const float2 d = mul2(make_float2(pr[j0], pr[j0 + 1]),
                                  add2(make_float2(__uint_as_float(sr[c][jj]),
                                                   __uint_as_float(sr[c][jj + 1])), ndl));
            pk[jj >> 1] = pack_bf16(d.x, d.y);
          }
          tmem_st16(t_dp + c * 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(ds_full(g & 1));
        ++cnt;
        ++g;
      }
      if (!ok) break;
      if (cnt > 0 &&
          !(ok = warp_wait(dq_done((g - 1) & 1), ((g - 1) >> 1) & 1, abort, p.status, tmo)))
        break;
      tc_fence_after();
      const int64_t dq_off = (it.srow + row) * D + half * (D / 2);
      // (the TMEM loads are warp-collective: only the global stores are guarded)
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v32[32];
        if (cnt > 0) {
          tmem_ld32(tmem + lane_off + kDqCol + half * (D / 2) + c * 32, v32);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) v32[jj] = 0u;
        }
        if (!row_ok) continue;
        if (p.kv_chunk >= 0 && (reinterpret_cast<uintptr_t>(p.out0) & 31) == 0) {
          // one ring step: the float32 contribution, overwritten or added; 32-byte
          // loads and stores, every old value loaded before any store
          float* dst = static_cast<float*>(p.out0) + dq_off + c * 32;
          float y[32];
          if (p.accumulate) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              asm volatile("ld.global.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                           : "=f"(y[8 * j]), "=f"(y[8 * j + 1]), "=f"(y[8 * j + 2]), "=f"(y[8 * j + 3]),
                             "=f"(y[8 * j + 4]), "=f"(y[8 * j + 5]), "=f"(y[8 * j + 6]), "=f"(y[8 * j + 7])
                           : "l"(dst + 8 * j));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) y[j] = 0.f;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              // a multiply and an add, each rounded (no fused multiply-add), as below
              x[e] = __fmul_rn(__uint_as_float(v32[8 * j + e]), p.scale);
              if (p.accumulate) x[e] = __fadd_rn(x[e], y[8 * j + e]);
            }
            asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 8 * j),
                         "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
                         "f"(x[7])
                         : "memory");
          }
        } else if (p.kv_chunk >= 0) {
          // one ring step: the float32 contribution, overwritten or added
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out0) + dq_off + c * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float4 x = make_float4(__fmul_rn(__uint_as_float(v32[4 * j]), p.scale),
                                   __fmul_rn(__uint_as_float(v32[4 * j + 1]), p.scale),
                                   __fmul_rn(__uint_as_float(v32[4 * j + 2]), p.scale),
                                   __fmul_rn(__uint_as_float(v32[4 * j + 3]), p.scale));
            if (p.accumulate) {
              const float4 y = dst[j];
              x.x = __fadd_rn(x.x, y.x);
              x.y = __fadd_rn(x.y, y.y);
              x.z = __fadd_rn(x.z, y.z);
              x.w = __fadd_rn(x.w, y.w);
            }
            dst[j] = x;
          }
        } else if ((reinterpret_cast<uintptr_t>(p.out0) & 31) == 0) {
          // 32-byte stores: half as many store instructions, each touching 32 rows
          store_row32_bf16_v8(static_cast<__nv_bfloat16*>(p.out0) + dq_off + c * 32, v32, p.scale);
        } else {
          store_row32_bf16(static_cast<__nv_bfloat16*>(p.out0) + dq_off + c * 32, v32, p.scale);
        }
      }
      // the accumulator has been read: the next item's first dQ may overwrite it
      tc_fence_before();
      mbar_arrive(dq_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // launched as the dK/dV kernel's programmatic dependent: finish only after that
  // grid has completed (a no-op for any other launch)
  griddep_wait();
}

template <typename K>
static cudaError_t prep(K kern, int smem) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return check_register_split(kern, kThreads);
}

template <int D>
static cudaError_t run_bwd(const Ring& R, const Params& base, const void* q, const void* k,
                           const void* v, const void* dO, void* dq, void* dk, void* dv,
                           cudaStream_t st, const AfterDkdv* after = nullptr,
                           const AfterDqPart* dq_parts = nullptr) {
  const bool ag = base.ag_rank >= 0;
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t qrows = (uint64_t)R.B * R.Hq * R.T, krows = (uint64_t)R.B * R.Hkv * R.T;
  const uint64_t dorows = ag ? (uint64_t)R.B * R.Hq * (R.T / R.cp) : qrows;
  if (encode_tmap_2d_bf16(&tq, q, D, qrows, 64, kTile) != CUDA_SUCCESS ||
      encode_tmap_2d_bf16(&tdo, dO, D, dorows, 64, kTile) != CUDA_SUCCESS ||
      encode_tmap_2d_bf16(&tk, k, D, krows, 64, kTile) != CUDA_SUCCESS ||
      encode_tmap_2d_bf16(&tv, v, D, krows, 64, kTile) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // dK / dV as boxes of 32 rows x 64 bf16 columns (ring) or 32 x 32 float32 columns
  // (the all-gather sums and a ring step's parts), for the epilogue's TMA operations
  CUtensorMap tdk = tq, tdv = tq;
  if (D == 128) {
    const bool step_mode = ag && base.kv_chunk >= 0;
    const uint64_t orows = (uint64_t)R.B * R.Hkv * (step_mode ? R.T / R.cp : R.T);
    const CUresult r1 = ag ? encode_tmap_2d_f32(&tdk, dk, D, orows, 32, 32)
                           : encode_tmap_2d_bf16(&tdk, dk, D, orows, 64, 32);
    const CUresult r2 = ag ? encode_tmap_2d_f32(&tdv, dv, D, orows, 32, 32)
                           : encode_tmap_2d_bf16(&tdv, dv, D, orows, 64, 32);
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  Params pk = base;
  pk.out0 = dk;
  pk.out1 = dv;
  pk.claim = nullptr;
  const bool packed = base.doc_lo != nullptr;  // ring mode only (checked by the caller)
  auto kdkdv = ag ? dkdv_kernel<D, true, false>
                  : (packed ? dkdv_kernel<D, false, true> : dkdv_kernel<D, false, false>);
  cudaError_t e = prep(kdkdv, DkdvSmem<D>::kBytes);
  if (e != cudaSuccess) return e;
  const bool step = ag && base.kv_chunk >= 0;  // one ring step: the chunk's K/V tiles only
  const int kv_items = R.B * R.Hkv * ((step ? R.T / R.cp : R.T) / kTile);
  Params pq = base;
  pq.out0 = dq;
  pq.out1 = nullptr;
  auto kdq = packed ? dq_kernel<D, true> : dq_kernel<D, false>;
  e = prep(kdq, DqSmem<D>::kBytes);
  if (e != cudaSuccess) return e;
  const int q_items = R.B * R.Hq * ((ag ? R.T / R.cp : R.T) / kTile);
  // persistent: at most one resident CTA per SM, each walking its share of the items
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int q_grid = q_items < sms ? q_items : sms;
  // dQ in parts (plain ring only): part j is the j-th contiguous np-th of every tensor,
  // batch rows when np divides B, else K/V heads (with their query heads) of each row
  const int np = dq_parts != nullptr && dq_parts->fn != nullptr ? dq_parts->parts : 1;
  const bool split = np > 1 && !ag && !packed &&
                     (R.B % np == 0 || (np % R.B == 0 && R.Hkv % (np / R.B) == 0));

  // The dK/dV and dQ kernels read the same inputs and write disjoint outputs, so they
  // may overlap.  The dK/dV kernel's CTAs differ in work by up to 64 times (a key
  // tile is seen by the query tiles at or after it), and its last ones leave SMs
  // idle while they finish.  With an item counter (nothing queued between the two
  // kernels) the dQ kernel is launched as a programmatic dependent of the dK/dV
  // kernel, whose CTAs release it as they start: once the last dK/dV CTA is
  // resident, the persistent dQ CTAs take the SMs that the dK/dV kernel frees,
  // claiming their items from the counter, and each waits for the dK/dV grid to
  // complete before it exits, so the stream's next work sees both kernels' results.
  if (base.claim != nullptr && after == nullptr && np == 1) {
    if ((e = cudaMemsetAsync(base.claim, 0, sizeof(int), st)) != cudaSuccess) return e;
    timing_begin(step     ? "tc_partial_dkdv_dq"
                 : ag     ? "tc_allgather_dkdv_dq"
                 : packed ? "tc_packed_dkdv_dq"
                          : "tc_bwd_dkdv_dq",
                 st);
    kdkdv<<<kv_items, kThreads, DkdvSmem<D>::kBytes, st>>>(tq, tk, tv, tdo, tdk, tdv, pk);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)q_grid);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = DqSmem<D>::kBytes;
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, kdq, tq, tk, tv, tdo, pq);
    }
    timing_end(st);
    return e;
  }
  pq.claim = nullptr;

  timing_begin(step     ? "tc_partial_dkdv"
               : ag     ? "tc_allgather_dkdv"
               : packed ? "tc_packed_dkdv"
                        : "tc_bwd_dkdv",
               st);
  kdkdv<<<kv_items, kThreads, DkdvSmem<D>::kBytes, st>>>(tq, tk, tv, tdo, tdk, tdv, pk);
  e = cudaGetLastError();
  timing_end(st);
  if (e != cudaSuccess) return e;
  if (after != nullptr && after->fn != nullptr && (e = after->fn(after->ctx, st)) != cudaSuccess)
    return e;
  if (split) {
    const int m = R.B % np == 0 ? 1 : np / R.B;  // parts per batch row
    const int Bp = R.B % np == 0 ? R.B / np : 1, Hqp = R.Hq / m, Hkvp = R.Hkv / m;
    const uint64_t qr = (uint64_t)Bp * Hqp * R.T, kr = (uint64_t)Bp * Hkvp * R.T;
    for (int j = 0; j < np; ++j) {
      const char* qj = static_cast<const char*>(q) + j * qr * D * 2;
      const char* kj = static_cast<const char*>(k) + j * kr * D * 2;
      const char* vj = static_cast<const char*>(v) + j * kr * D * 2;
      const char* dj = static_cast<const char*>(dO) + j * qr * D * 2;
      CUtensorMap pqm, pkm, pvm, pdm;
      if (encode_tmap_2d_bf16(&pqm, qj, D, qr, 64, kTile) != CUDA_SUCCESS ||
          encode_tmap_2d_bf16(&pdm, dj, D, qr, 64, kTile) != CUDA_SUCCESS ||
          encode_tmap_2d_bf16(&pkm, kj, D, kr, 64, kTile) != CUDA_SUCCESS ||
          encode_tmap_2d_bf16(&pvm, vj, D, kr, 64, kTile) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
      Params pj = pq;
      pj.B = Bp;
      pj.Hq = Hqp;
      pj.Hkv = Hkvp;
      pj.lse2 = base.lse2 + j * qr;
      pj.delta = base.delta + j * qr;
      pj.out0 = static_cast<char*>(dq) + j * qr * D * 2;
      const int items = (int)(qr / kTile);
      timing_begin("tc_bwd_dq", st);
      kdq<<<items < sms ? items : sms, kThreads, DqSmem<D>::kBytes, st>>>(pqm, pkm, pvm, pdm, pj);
      e = cudaGetLastError();
      timing_end(st);
      if (e != cudaSuccess) return e;
      if ((e = dq_parts->fn(dq_parts->ctx, st, j)) != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  timing_begin(step     ? "tc_partial_dq"
               : ag     ? "tc_allgather_dq"
               : packed ? "tc_packed_dq"
                        : "tc_bwd_dq",
               st);
  kdq<<<q_grid, kThreads, DqSmem<D>::kBytes, st>>>(tq, tk, tv, tdo, pq);
  e = cudaGetLastError();
  timing_end(st);
  if (e == cudaSuccess && np > 1)
    for (int j = 0; j < np && e == cudaSuccess; ++j) e = dq_parts->fn(dq_parts->ctx, st, j);
  return e;
}

}  // namespace tcbwd

static tcbwd::Params bwd_params(const Ring& R, const float* lse2, const float* delta,
                                int* status) {
  tcbwd::Params p;
  p.B = R.B;
  p.Hq = R.Hq;
  p.Hkv = R.Hkv;
  p.T = R.T;
  p.n_rep = R.Hq / R.Hkv;
  p.m = SeqMap::make(R.T, R.cp, R.zz);
  p.scale = R.scale;
  p.scale_log2 = R.scale * tcbwd::kLog2e;
  p.lse2 = lse2;
  p.delta = delta;
  p.status = status;
  p.ag_rank = -1;
  p.accumulate = 0;
  p.kv_chunk = -1;
  p.doc_lo = nullptr;
  p.doc_hi = nullptr;
  p.ord_q = nullptr;
  p.ord_k = nullptr;
  p.debug_fault = R.debug_fault;
  p.claim = nullptr;
  return p;
}

cudaError_t launch_tc_bwd(const Ring& R, const void* q, const void* k, const void* v,
                          const float* lse2, const float* delta, const void* dO, void* dq,
                          void* dk, void* dv, int* status, cudaStream_t st, const int* doc_lo,
                          const int* doc_hi, const int* ord_q, const int* ord_k,
                          const AfterDkdv* after, const AfterDqPart* dq_parts, int* dq_claim) {
  tcbwd::Params p = bwd_params(R, lse2, delta, status);
  p.doc_lo = doc_lo;
  p.doc_hi = doc_hi;
  p.ord_q = ord_q;
  p.ord_k = ord_k;
  p.claim = dq_claim;
  if (R.D == 128) return tcbwd::run_bwd<128>(R, p, q, k, v, dO, dq, dk, dv, st, after, dq_parts);
  return tcbwd::run_bwd<64>(R, p, q, k, v, dO, dq, dk, dv, st, after, dq_parts);
}

cudaError_t launch_tc_partial_bwd(const Ring& R, int q_rank, int kv_rank, const void* q,
                                  const void* k, const void* v, const float* lse2,
                                  const float* delta, const void* dO, float* dq_part,
                                  float* dk_part, float* dv_part, int accumulate, int* status,
                                  cudaStream_t st, int* dq_claim) {
  tcbwd::Params p = bwd_params(R, lse2, delta, status);
  p.ag_rank = q_rank;
  p.kv_chunk = kv_rank;
  p.accumulate = accumulate ? 1 : 0;
  p.claim = dq_claim;
  if (R.D == 128) return tcbwd::run_bwd<128>(R, p, q, k, v, dO, dq_part, dk_part, dv_part, st);
  return tcbwd::run_bwd<64>(R, p, q, k, v, dO, dq_part, dk_part, dv_part, st);
}

cudaError_t launch_tc_allgather_bwd(const Ring& R, int q_rank, const void* q, const void* k,
                                    const void* v, const float* lse2, const float* delta,
                                    const void* dO, void* dq, float* dk_sum, float* dv_sum,
                                    int accumulate, int* status, cudaStream_t st,
                                    int* dq_claim) {
  tcbwd::Params p = bwd_params(R, lse2, delta, status);
  p.ag_rank = q_rank;
  p.accumulate = accumulate ? 1 : 0;
  p.claim = dq_claim;
  if (R.D == 128) return tcbwd::run_bwd<128>(R, p, q, k, v, dO, dq, dk_sum, dv_sum, st);
  return tcbwd::run_bwd<64>(R, p, q, k, v, dO, dq, dk_sum, dv_sum, st);
}

}  // namespace cpattn
