// Ring-attention forward on the 5th-generation tensor cores (sm_103a).
//
// What one work item computes: one 128-row query tile of one (batch, head) against
// every key/value tile its rows can see, visited in ring order -- step i of
// rank r holds the K/V chunk of rank (r - i) mod cp (tutorial "上下文并行",
// section "朴素 Ring Attention") -- with the running max / sum / output carried
// across steps, i.e. the per-step partials merged by the single-pass online
// softmax (pull request "Feat: Context Parallel" #181, mode "p2p").  Tiles
// wholly hidden by the causal mask (key position > query position for every
// pair) are skipped; diagonal tiles are masked per element from global
// positions.
//
// The CTAs are persistent (at most one per SM) and walk the heaviest-first item
// list in a snake order; every pipeline keeps running across items, so the next
// item's loads and first S overlap the current item's last tiles and epilogue.
//
// Two softmax threads per query row: thread (row, h) owns key columns
// [64h, 64h+64) of every tile and runs an online softmax of its own over them
// into an output accumulator of its own, O_h.  The two halves are partial
// results over disjoint key sets; the epilogue merges them once with the
// (O, LSE) merge rule (tutorial, section "朴素 Ring Attention"), so the two
// threads of a row never exchange anything per tile.
//
// Warp roles (384 threads):
//   warp 0        TMA producer: the Q tile, then the K tiles through a ring of
//                 shared-memory stages (128-byte swizzle); warp 3: the V tiles
//                 through a ring of their own.
//   warp 1        S issuer: S = Q K^T (SS form) into one of two TMEM buffers, so
//                 S of the next tile is formed while the softmax of this one runs.
//   warp 2        PV issuer: O_h += P_h V_h (TS form, P_h read from TMEM) for each
//                 half as soon as that half's P is stored.
//                 Both issuers run as whole warps with warp-uniform descriptor
//                 arithmetic and issue from one elected lane, which issues
//                 markedly faster than a lone thread.  Two issuers because a
//                 tcgen05.mma that runs 64 cycles at N = 128 takes tens of cycles
//                 to issue, the pipe queues only a few, and a thread's next memory
//                 access after a tcgen05.commit waits for the committed MMAs: one
//                 issuer that also waited on the softmax would leave the pipe idle.
//   warps 4..11   softmax: warp w serves TMEM lane quadrant w%4 (32 rows) and
//                 column half (w-4)/4.  tcgen05.ld of its 64 scores, causal
//                 mask, P = 2^(s*scale*log2e - m) rounded to bf16 into TMEM, sum
//                 in fp32.  O_h is rescaled only when the running max grows by
//                 more than 2^8 (exact after the final division); thanks to that
//                 slack P is formed against the running max in the same pass that
//                 takes the tile's max, and formed again only when a row's max
//                 rose by more than 2^8.
//   epilogue      M = max(m_0, m_1), w_h = 2^(m_h - M), L = w_0 l_0 + w_1 l_1,
//                 O = (w_0 O_0 + w_1 O_1) / L rounded once to the output dtype,
//                 LSE = ln 2 (M + log2 L).
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256, 256+D),
// O_1 [256+D, 256+2D); P of half h overwrites columns [64h, 64h+32) of its S.
// Every mbarrier wait is bounded; on time-out the CTA raises its abort flag,
// latches CPATTN_ERR_TIMEOUT in the device status word, drains its own TMA
// loads and MMAs, frees TMEM and exits.
#include <math.h>

#include "kernels.h"

namespace cpattn {
namespace tcfwd {

constexpr int kTile = 128;
constexpr int kThreads = 384;
constexpr uint64_t kTimeoutNs = 2000000000ull;     // 2 s
constexpr uint64_t kDebugTimeoutNs = 50000000ull;  // 50 ms under the fault hook
constexpr uint64_t kDrainTimeoutNs = 200000000ull;
constexpr float kLn2 = 0.69314718055994530942f;

enum : int { kEmpty = 0, kFull = 1, kDiag = 2 };

struct Params {
  int B, Hq, Hkv, T, n_rep;
  SeqMap m;
  float scale_log2;
  int q_tiles;          // 128-row query tiles per (batch, head) in the launch
  int n_items;          // work items (B * Hq * q_tiles), walked by resident CTAs
  // q_rank >= 0: only that rank's query rows, written as c rows per (b, h); with
  // kv_rank >= 0 against that one chunk (a ring step), with kv_rank < 0 against
  // every chunk (the all-gather mode)
  int q_rank, kv_rank;
  void* o;
  float* lse;
  int* status;
  int debug_fault;
  // packed sequences: lo[b * T + p] = first natural position of p's document in
  // batch row b (nullptr: one document per row, plain causal attention)
  const int* doc_lo;
  // packed sequences: (batch row, query tile) entries b * (T/128) + tile, heaviest
  // first (the order items are handed out in)
  const int* ord_q;
};

template <int D>
struct Smem {
  // one Q tile; K and V in rings of their own (K is last read by S, V by PV); at
  // D = 128 a 4 KB staging area per softmax warp for the bf16 output (a third K
  // stage in its place measured no faster); the (m, l) exchange of the two column
  // halves of each row
  static constexpr int kKStages = D == 128 ? 2 : 4;
  static constexpr int kVStages = D == 128 ? 3 : 4;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kTileBytes;
  static constexpr int kV = kK + kKStages * kTileBytes;
  static constexpr int kOst = kV + kVStages * kTileBytes;
  static constexpr int kOstBytes = D == 128 ? 8 * 32 * 128 : 0;
  static constexpr int kXch = kOst + kOstBytes;
  static constexpr int kBar = kXch + 2 * kTile * 8;
  // barriers: q_full, q_empty, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
  // s_full[2], p_full[2 buffers][2 halves], pv_done[2], o_free, xch_full, xch_free,
  // final_s, final_pv
  static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 2 + 4 + 2 + 3 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  // no alignment slack: the kernel declares its dynamic shared memory 1024-byte
  // aligned and checks it
  static constexpr int kBytes = kMisc + 16;
};

struct Item {
  int b, h, g, rank, slot0, pos0;
};

template <bool PK>
__device__ __forceinline__ Item decode(const Params& p, int w) {
  Item it;
  if constexpr (PK) {
    // packed: items in decreasing work, every head of a (batch row, tile) together
    const int nt = p.T >> 7;
    const int ent = p.ord_q[w / p.Hq];
    it.b = ent / nt;
    it.h = w - (w / p.Hq) * p.Hq;
    it.g = it.h / p.n_rep;
    it.pos0 = (ent - it.b * nt) * kTile;
    it.slot0 = p.m.slot(it.pos0);
    it.rank = it.slot0 / p.m.c;
    return it;
  }
  const int units = p.B * p.Hq;
  const int ti = w / units;
  const int rem = w - ti * units;
  it.b = rem / p.Hq;
  it.h = rem - it.b * p.Hq;
  it.g = it.h / p.n_rep;
  if (p.q_rank >= 0) {
    // the rank's later slots hold its later positions (its second zigzag half):
    // heaviest first
    it.slot0 = p.q_rank * p.m.c + (p.q_tiles - 1 - ti) * kTile;
    it.pos0 = p.m.pos(it.slot0);
  } else {
    // heaviest (latest) query positions first: causal work grows with position
    it.pos0 = (p.q_tiles - 1 - ti) * kTile;
    it.slot0 = p.m.slot(it.pos0);
  }
  it.rank = it.slot0 / p.m.c;
  return it;
}

// Tile pairs on the same 128-position grid.  Plain causal: full below the
// diagonal, empty above it, masked on it.  Packed sequences (lo_row = the batch
// row's document starts per position): also empty when every key lies before
// the first query's document, and full only when every key lies in the last
// query's document; any other pair is masked per element.
__device__ __forceinline__ int classify(int qpos0, int kpos0, const int* lo_row) {
  if (kpos0 > qpos0 + kTile - 1) return kEmpty;
  if (lo_row == nullptr) return kpos0 + kTile - 1 <= qpos0 ? kFull : kDiag;
  if (kpos0 + kTile - 1 < lo_row[qpos0]) return kEmpty;
  return kpos0 + kTile - 1 <= qpos0 && kpos0 >= lo_row[qpos0 + kTile - 1] ? kFull : kDiag;
}

// Wait in which every lane of the warp takes part; all lanes agree on the result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t par, volatile int* abort,
                                          int* status, uint64_t tmo) {
  bool ok = mbar_wait(bar, par, abort, status, tmo);
  return __all_sync(0xffffffffu, ok);
}

// Wait that ignores the abort flag (used to drain in-flight copies before exit).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t par) {
  int never = 0;
  return mbar_wait(bar, par, &never, nullptr, kDrainTimeoutNs);
}

template <int D, bool OUT_F32, bool PK>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const Params p) {
  using L = Smem<D>;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the layout has no alignment slack
    if (threadIdx.x == 0) latch_status(p.status, kStatusLaunch);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBar;
  const uint32_t q_full = bars;
  const uint32_t q_empty = bars + 8;
  auto k_full = [&](int s) { return bars + 8 * (2 + s); };
  auto k_empty = [&](int s) { return bars + 8 * (2 + KS + s); };
  auto v_full = [&](int s) { return bars + 8 * (2 + 2 * KS + s); };
  auto v_empty = [&](int s) { return bars + 8 * (2 + 2 * KS + VS + s); };
  const uint32_t tile_bars = bars + 8 * (2 + 2 * KS + 2 * VS);
  auto s_full = [&](int b) { return tile_bars + 8 * b; };
  auto p_full = [&](int b, int h) { return tile_bars + 8 * (2 + 2 * b + h); };
  auto pv_done = [&](int b) { return tile_bars + 8 * (6 + b); };
  const uint32_t o_free = tile_bars + 8 * 8;
  const uint32_t xch_full = tile_bars + 8 * 9;
  const uint32_t xch_free = tile_bars + 8 * 10;
  const uint32_t final_s = tile_bars + 8 * 11;
  const uint32_t final_pv = tile_bars + 8 * 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  float2* xch = reinterpret_cast<float2*>(smem + L::kXch);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = p.debug_fault ? kDebugTimeoutNs : kTimeoutNs;
  // row extents of the tensors (for the bounds checks of a CPATTN_DEBUG build)
  const int64_t q_rows = (int64_t)p.B * p.Hq * p.T, kv_rows = (int64_t)p.B * p.Hkv * p.T;
  const int64_t o_rows = p.q_rank >= 0 ? (int64_t)p.B * p.Hq * p.m.c : q_rows;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) {
      const uint32_t b = bars + 8 * i;
      // p_full: the 128 softmax threads of one column half; o_free / xch_*: all 256
      const bool half_arrivals = b >= p_full(0, 0) && b <= p_full(1, 1);
      const bool all_arrivals = b == o_free || b == xch_full || b == xch_free;
      mbar_init(b, half_arrivals ? 128 : all_arrivals ? 256 : 1);
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

  // K/V tiles of an item in ring order: chunks r, r-1, ..., r-cp+1 (mod cp), or one
  // chunk; every role walks the same list and skips the tiles the causal mask hides
  const bool one_chunk = p.q_rank >= 0 && p.kv_rank >= 0;
  // packed sequences only in the PK instantiation, so the plain path keeps its code
  auto doc_row = [&](const Item& it) -> const int* {
    return PK ? p.doc_lo + (int64_t)it.b * p.T : nullptr;
  };
  // packed: the key tiles of the query tile's visible range, from the tile holding
  // its first row's document start up to the diagonal, in natural order
  using Walk = std::conditional_t<PK, NatWalk, TileWalk>;
  auto walk_start = [&](Walk& w, const Item& it) {
    if constexpr (PK) {
      w.start(p.m, doc_row(it)[it.pos0] >> 7, it.pos0 >> 7, 1);
    } else {
      w.start(p.m, one_chunk ? p.kv_rank : it.rank, one_chunk ? 1 : p.m.cp, -1, 1);
      w.settle_keys(it.pos0);
    }
  };
  auto walk_next = [&](Walk& w, const Item& it) {
    w.next();
    if constexpr (!PK) w.settle_keys(it.pos0);
  };

  if (warp < 4) {
  regs_ctl();  // warpgroup 0: TMA producers (warps 0, 3) and MMA issuers (warps 1, 2)
  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ producers
    // warp 0: each item's Q tile, then its K tiles; warp 3: the V tiles
    if (lane == 0) {
      const bool is_k = warp == 0;
      const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
      tma_prefetch_desc(tm);
      if (is_k) tma_prefetch_desc(&tm_q);
      const int nst = is_k ? KS : VS;
      const uint32_t base = sbase + (is_k ? L::kK : L::kV);
      int stage = 0, par = 0, q_last = -1;
      uint32_t issued = 0, issued_par = 0;  // bit s: stage s loaded / its phase parity
      bool ok = true;
      int w;
      for (int k = 0; ok && (w = item_of(k, p.n_items)) >= 0; ++k) {
        const Item it = decode<PK>(p, w);
        const int kv_row_base = (it.b * p.Hkv + it.g) * p.T;
        if (is_k) {
          // the Q buffer is free once the last S of the previous item has read it
          if (k > 0 && !(ok = mbar_wait(q_empty, (k - 1) & 1, abort, p.status, tmo))) break;
          if (!(k == 0 && p.debug_fault == 1)) {  // fault hook: the first Q load never happens
            mbar_expect_tx(q_full, L::kTileBytes);
            const int row = (it.b * p.Hq + it.h) * p.T + it.slot0;
            if (in_bounds(row, kTile, q_rows, p.status))
              for (int kb = 0; kb < D / 64; ++kb)
                tma_load_2d(sbase + L::kQ + kb * (kTile * 128), &tm_q, kb * 64, row, q_full);
            q_last = k;
          }
        }
        Walk wk;
        for (walk_start(wk, it); !wk.done(); walk_next(wk, it)) {
          const uint32_t empty = is_k ? k_empty(stage) : v_empty(stage);
          const uint32_t full = is_k ? k_full(stage) : v_full(stage);
          if (!(ok = mbar_wait(empty, par ^ 1, abort, p.status, tmo))) break;
          const int row = kv_row_base + wk.slot();
          mbar_expect_tx(full, L::kTileBytes);
          if (in_bounds(row, kTile, kv_rows, p.status))
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_2d(base + stage * L::kTileBytes + kb * (kTile * 128), tm, kb * 64, row, full);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | ((uint32_t)par << stage);
          if (++stage == nst) stage = 0, par ^= 1;
        }
      }
      // never leave with a copy still writing into this CTA's shared memory
      if (q_last >= 0) drain_wait(q_full, q_last & 1);
      for (int st = 0; st < nst; ++st)
        if ((issued >> st) & 1u)
          drain_wait(is_k ? k_full(st) : v_full(st), (issued_par >> st) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    // (whole warp, warp-uniform descriptors; one elected lane issues)
    {
      const bool leader = elect_one();
      constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kTileDesc = L::kTileBytes >> 4;
      // descriptor bases; per k-step offsets are compile-time constants (16-byte units)
      const uint64_t qd = sdesc_sw128(sbase + L::kQ, 16, 1024);
      const uint64_t kd0 = sdesc_sw128(sbase + L::kK, 16, 1024);
      StageRing<KS> kr;
      int g = 0;  // tiles so far over all items: buffer g&1, its phase (g>>1)&1
      bool ok = true;
      int w;
      for (int k = 0; ok && (w = item_of(k, p.n_items)) >= 0; ++k) {
        const Item it = decode<PK>(p, w);
        if (!(ok = warp_wait(q_full, k & 1, abort, p.status, tmo))) break;
        Walk wk;
        for (walk_start(wk, it); !wk.done(); walk_next(wk, it)) {
          const int b = g & 1;
          if (!(ok = warp_wait(k_full(kr.stage), kr.par, abort, p.status, tmo))) break;
          // buffer b is free once PV of tile g-2 has read the P stored there
          if (g >= 2 && !(ok = warp_wait(pv_done(b), ((g - 2) >> 1) & 1, abort, p.status, tmo)))
            break;
          tc_fence_after();
          const uint64_t kd = kd0 + (uint64_t)(kr.stage * kTileDesc);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;  // 16 KiB blocks, 32 B steps
            if (leader) mma_ss(tmem + b * 128, qd + off, kd + off, kIdescS, kk > 0);
          }
          if (leader) {
            mma_commit(s_full(b));
            mma_commit(k_empty(kr.stage));
          }
          __syncwarp();
          kr.advance();
          ++g;
        }
        if (!ok) break;
        if (leader) mma_commit(q_empty);  // the Q buffer may take the next item's tile
        __syncwarp();
      }
      // every MMA this warp issued has finished before TMEM can be freed
      if (leader) mma_commit(final_s);
      __syncwarp();
      drain_wait(final_s, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    // (whole warp, one elected lane issues)
    {
      const bool leader = elect_one();
      constexpr uint32_t kIdescPV = idesc_bf16(128, D, false, true);
      constexpr uint32_t kTileDesc = L::kTileBytes >> 4;
      const uint64_t vd0 = sdesc_sw128(sbase + L::kV, kTile * 128, 1024);
      StageRing<VS> vr;
      int g = 0;
      bool ok = true;
      int w;
      for (int k = 0; ok && (w = item_of(k, p.n_items)) >= 0; ++k) {
        const Item it = decode<PK>(p, w);
        int t = 0;  // tile of this item
        Walk wk;
        for (walk_start(wk, it); !wk.done(); walk_next(wk, it)) {
          const int b = g & 1;
          if (!(ok = warp_wait(v_full(vr.stage), vr.par, abort, p.status, tmo))) break;
          // the first PV of an item overwrites O: the previous item's epilogue has read it
          if (t == 0 && k > 0 && !(ok = warp_wait(o_free, (k - 1) & 1, abort, p.status, tmo)))
            break;
          const uint64_t vd = vd0 + (uint64_t)(vr.stage * kTileDesc);
          for (int h = 0; h < 2 && ok; ++h) {
            // O_h += P_h V_h: keys [64h, 64h+64), 16 key rows = 2048 B per k-step
            if (!(ok = warp_wait(p_full(b, h), (g >> 1) & 1, abort, p.status, tmo))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (leader)
                mma_ts(tmem + 256 + h * D, tmem + b * 128 + h * 64 + kk * 8,
                       vd + (uint64_t)((h * 4 + kk) * 128), kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
            __syncwarp();
          }
          if (!ok) break;
          if (leader) {
            mma_commit(pv_done(b));
            mma_commit(v_empty(vr.stage));
          }
          __syncwarp();
          vr.advance();
          ++g;
          ++t;
        }
      }
      if (leader) mma_commit(final_pv);
      __syncwarp();
      drain_wait(final_pv, 0);
    }
  }
  } else {
    regs_math();  // warpgroups 1 and 2: softmax
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;         // TMEM lane quadrant this warp may access
    const int half = (warp - 4) >> 2;  // key columns [64 half, 64 half + 64) of a tile
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_o = tmem + lane_off + 256 + half * D;
    const float2 sl2v = make_float2(p.scale_log2, p.scale_log2);
    int g = 0;
    bool ok = true;
    int w;
    for (int k = 0; ok && (w = item_of(k, p.n_items)) >= 0; ++k) {
      const Item it = decode<PK>(p, w);
      const int* lo_row = doc_row(it);
      // packed: this row's keys start at its document's first position
      const int lo_q = PK ? lo_row[it.pos0 + row] : 0;
      float m_run = -INFINITY, l_run = 0.f;
      int cnt = 0;  // tiles of this item
      Walk wk;
      for (walk_start(wk, it); !wk.done(); walk_next(wk, it)) {
        const int kpos = wk.pos();
        const int cls = classify(it.pos0, kpos, lo_row);
        const int b = g & 1;
        const uint32_t t_s = tmem + lane_off + b * 128 + half * 64;
        if (!(ok = warp_wait(s_full(b), (g >> 1) & 1, abort, p.status, tmo))) break;
        tc_fence_after();
        uint32_t r[2][32];
        tmem_ld32(t_s, r[0]);
        tmem_ld32(t_s + 32, r[1]);
        tmem_wait_ld();
        if (cls == kDiag) {
          // key column j of this half is visible iff lo_q <= kpos + 64 half + j <= qpos + row
          const int thr = row + it.pos0 - kpos - half * 64;
          const int thr_lo = lo_q - kpos - half * 64;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j > thr || (PK && c * 32 + j < thr_lo))
                r[c][j] = __float_as_uint(-INFINITY);
        }
        // P = 2^(s * scale * log2e - mu) for the 64 scores: exponent arguments and row
        // sums two lanes per instruction (packed fp32x2), 2^x on the special-function
        // unit, P stored as bf16 over the scores.  With with_max set, the tile's max
        // is taken in the same pass (4 independent chains of three-input max).
        auto form_p = [&](auto with_max, float mu, float& mx) -> float {
          const float2 nmu = make_float2(-mu, -mu);
          float2 l4[4];
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < 4; ++i) l4[i] = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float s0 = __uint_as_float(r[c][2 * j]), s1 = __uint_as_float(r[c][2 * j + 1]);
              if (decltype(with_max)::value) m4[(c * 16 + j) & 3] = max3(m4[(c * 16 + j) & 3], s0, s1);
              const float2 x = fma2(make_float2(s0, s1), sl2v, nmu);
              const float2 pp = make_float2(ex2(x.x), ex2(x.y));
              l4[j & 3] = add2(l4[j & 3], pp);
              pk[j] = pack_bf16(pp.x, pp.y);
            }
            tmem_st16(t_s + c * 16, pk);
          }
          if (decltype(with_max)::value) mx = fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]);
          return ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) + ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));
        };
        bool rescale = false;
        float factor = 1.f;
        float lsum;
        // form_p's TMEM stores are warp-collective: every branch around it is taken
        // by the whole warp
        if (cnt > 0 && __all_sync(0xffffffffu, m_run != -INFINITY)) {
          // Against the running max straight away, the tile's max alongside: P stays
          // below 2^8 unless the tile's max exceeds the running max by more than 8
          // (log2 units).  Only then (rarely after an item's first tiles) is the
          // running max raised and the tile's P formed again over what was stored,
          // by the whole warp (a row whose max did not move forms the same P again).
          float mx;
          lsum = form_p(std::true_type{}, m_run, mx);
          const float m_tile = mx * p.scale_log2;
          const bool jump = m_tile > m_run + 8.f;
          if (jump) {
            factor = ex2(m_run - m_tile);
            l_run *= factor;
            m_run = m_tile;
            rescale = true;
          }
          if (__any_sync(0xffffffffu, jump)) {
            tmem_wait_st();
            lsum = form_p(std::false_type{}, m_run, mx);
          }
        } else {
          float mx;
          {
            // 4 independent chains of three-input max over the 64 scores
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int j = 0; j < 32; j += 2)
                m4[(c * 16 + j / 2) & 3] = max3(m4[(c * 16 + j / 2) & 3], __uint_as_float(r[c][j]),
                                                __uint_as_float(r[c][j + 1]));
            mx = fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]);
          }
          const float m_new = fmaxf(m_run, mx * p.scale_log2);
          if (cnt == 0) {
            m_run = m_new;
          } else if (m_new > m_run + 8.f) {
            factor = ex2(m_run - m_new);
            l_run *= factor;
            m_run = m_new;
            rescale = true;
          }
          lsum = form_p(std::false_type{}, m_run == -INFINITY ? 0.f : m_run, mx);
        }
        l_run += lsum;
        tmem_wait_st();
        if (cnt > 0 && __any_sync(0xffffffffu, rescale)) {
          // O_h so far must be final in TMEM before it is rescaled
          if (!(ok = warp_wait(pv_done((g - 1) & 1), ((g - 1) >> 1) & 1, abort, p.status, tmo)))
            break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o32[32];
            tmem_ld32(t_o + c * 32, o32);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o32[j] = __float_as_uint(__uint_as_float(o32[j]) * factor);
            tmem_st32(t_o + c * 32, o32);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(p_full(b, half));
        ++cnt;
        ++g;
      }
      if (!ok) break;
      // ------------------------------------------------------ epilogue of the item
      if (cnt > 0 && !(ok = warp_wait(pv_done((g - 1) & 1), ((g - 1) >> 1) & 1, abort, p.status,
                                      tmo)))
        break;
      // the two halves' (m, l) meet in shared memory; the slot is free once the
      // partner has read the previous item's value
      if (k > 0 && !(ok = warp_wait(xch_free, (k - 1) & 1, abort, p.status, tmo))) break;
      xch[half * 128 + row] = make_float2(m_run, l_run);
      mbar_arrive(xch_full);
      if (!(ok = warp_wait(xch_full, k & 1, abort, p.status, tmo))) break;
      const float2 other = xch[(1 - half) * 128 + row];
      mbar_arrive(xch_free);
      tc_fence_after();
      const float m0 = half == 0 ? m_run : other.x, l0 = half == 0 ? l_run : other.y;
      const float m1 = half == 0 ? other.x : m_run, l1 = half == 0 ? other.y : l_run;
      const float mm = fmaxf(m0, m1);
      float w0 = 0.f, w1 = 0.f;
      if (mm != -INFINITY) {
        w0 = ex2(m0 - mm);
        w1 = ex2(m1 - mm);
      }
      const float lsum = w0 * l0 + w1 * l1;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const float a0 = w0 * inv, a1 = w1 * inv;
      const bool local = p.q_rank >= 0;
      const int64_t bh = (int64_t)it.b * p.Hq + it.h;
      const int64_t orow = local ? bh * p.m.c + (it.slot0 - p.q_rank * p.m.c) + row
                                 : bh * p.T + it.slot0 + row;
      if constexpr (D == 128 && !OUT_F32) {
        // This thread's 64 output columns [64 half, 64 half + 64) of its row, as bf16:
        // one 128-byte line in eight 16-byte chunks.  Stored from registers, every
        // store instruction of the warp would touch 32 lines (one per row); instead
        // the warp's 32 lines go to shared memory and leave as one TMA store.
        uint32_t wd[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o0[32], o1[32];
          if (cnt > 0) {
            tmem_ld32(tmem + lane_off + 256 + half * 64 + c * 32, o0);
            tmem_ld32(tmem + lane_off + 256 + D + half * 64 + c * 32, o1);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o0[j] = o1[j] = 0u;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j)
            wd[c * 16 + j] = pack_bf16(a0 * __uint_as_float(o0[2 * j]) + a1 * __uint_as_float(o1[2 * j]),
                                       a0 * __uint_as_float(o0[2 * j + 1]) +
                                           a1 * __uint_as_float(o1[2 * j + 1]));
        }
        // This warp's staging area holds line i (row 32 quad + i) at 128 i, its chunk
        // a at slot a ^ (i & 7): the tensor map's 128-byte swizzle of a 32 x 64 box
        // (the area starts on a 1024-byte boundary), and eight lanes writing chunk a
        // of eight lines meet eight different bank groups.  One TMA store writes the
        // box out while the warp goes on to the next item; the area is written again
        // only once that store has read it.
        const uint32_t ost = sbase + L::kOst + (warp - 4) * 4096;
        uint4* st4 = reinterpret_cast<uint4*>(smem + L::kOst + (warp - 4) * 4096);
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int a = 0; a < 8; ++a)
          st4[lane * 8 + (a ^ (lane & 7))] = make_uint4(wd[4 * a], wd[4 * a + 1], wd[4 * a + 2],
                                                        wd[4 * a + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        const int64_t tile_row0 = orow - row;
        if (lane == 0 && in_bounds(tile_row0, kTile, o_rows, p.status)) {
          tma_store_2d(&tm_o, half * 64, (int)(tile_row0 + quad * 32), ost);
          bulk_commit_group();
        }
      } else {
        // this thread writes output columns [D/2 half, D/2 half + D/2) of its row
        // (the TMEM loads are warp-collective: only the global stores are guarded)
        const bool store = in_bounds(orow, 1, o_rows, p.status);
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          const int col = half * (D / 2) + c * 32;
          uint32_t o0[32], o1[32];
          if (cnt > 0) {
            tmem_ld32(tmem + lane_off + 256 + col, o0);
            tmem_ld32(tmem + lane_off + 256 + D + col, o1);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o0[j] = o1[j] = 0u;
          }
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] = a0 * __uint_as_float(o0[j]) + a1 * __uint_as_float(o1[j]);
          if (store && OUT_F32 && (reinterpret_cast<uintptr_t>(p.o) & 31) == 0) {
            // 32-byte stores: half as many store instructions, each touching 32 rows
            float* dst = static_cast<float*>(p.o) + orow * D + col;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 8 * j),
                           "f"(v[8 * j]), "f"(v[8 * j + 1]), "f"(v[8 * j + 2]), "f"(v[8 * j + 3]),
                           "f"(v[8 * j + 4]), "f"(v[8 * j + 5]), "f"(v[8 * j + 6]), "f"(v[8 * j + 7])
                           : "memory");
          } else if (store && OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * D + col);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else if (store) {
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D + col);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pack_bf16(v[8 * j], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                                  pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                                  pack_bf16(v[8 * j + 6], v[8 * j + 7]));
          }
        }
      }
      if (half == 0 && in_bounds(orow, 1, o_rows, p.status))
        p.lse[orow] = lsum > 0.f ? (mm + log2f(lsum)) * kLn2 : -INFINITY;
      // O has been read: the next item's first PV may overwrite it
      tc_fence_before();
      mbar_arrive(o_free);
    }
  }

  // every output store of this CTA is complete before it ends
  if constexpr (D == 128 && !OUT_F32)
    if (warp >= 4 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace tcfwd

bool tc_supported(const Ring& R) {
  if (!R.bf16 || (R.D != 64 && R.D != 128)) return false;
  const int c = R.T / R.cp;
  const int seg = R.zz ? c / 2 : c;
  if (seg % tcfwd::kTile) return false;
  if ((double)R.B * R.Hq * R.T >= 2147483647.0) return false;
  return true;
}

template <int D, bool F32, bool PK = false>
static cudaError_t run_fwd(const Ring& R, const tcfwd::Params& p, int items, const void* q,
                           const void* k, const void* v, cudaStream_t st) {
  CUtensorMap tq, tk, tv, to;
  if (encode_tmap_2d_bf16(&tq, q, D, (uint64_t)R.B * R.Hq * R.T, 64, tcfwd::kTile) != CUDA_SUCCESS ||
      encode_tmap_2d_bf16(&tk, k, D, (uint64_t)R.B * R.Hkv * R.T, 64, tcfwd::kTile) != CUDA_SUCCESS ||
      encode_tmap_2d_bf16(&tv, v, D, (uint64_t)R.B * R.Hkv * R.T, 64, tcfwd::kTile) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // the bf16 output as 32-row, 64-column boxes (one softmax warp's rows and half); the
  // float32 outputs of a ring step are stored by the threads themselves
  to = tq;
  if (!F32 && D == 128) {
    const uint64_t o_rows = (uint64_t)R.B * R.Hq * (p.q_rank >= 0 ? R.T / R.cp : R.T);
    if (encode_tmap_2d_bf16(&to, p.o, D, o_rows, 64, 32) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  constexpr int kSmem = tcfwd::Smem<D>::kBytes;
  auto kern = tcfwd::fwd_kernel<D, F32, PK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if ((e = check_register_split(kern, tcfwd::kThreads)) != cudaSuccess) return e;
  // persistent: at most one resident CTA per SM, each walking its share of the items
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int grid = items < sms ? items : sms;
  kern<<<grid, tcfwd::kThreads, kSmem, st>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

cudaError_t launch_tc_fwd(const Ring& R, int q_rank, int kv_rank, const void* q, const void* k,
                          const void* v, void* o, float* lse, int* status, cudaStream_t st,
                          const int* doc_lo, const int* ord_q) {
  tcfwd::Params p;
  p.B = R.B;
  p.Hq = R.Hq;
  p.Hkv = R.Hkv;
  p.T = R.T;
  p.n_rep = R.Hq / R.Hkv;
  p.m = SeqMap::make(R.T, R.cp, R.zz);
  p.scale_log2 = R.scale * 1.44269504088896340736f;
  // q_rank >= 0: one rank's rows; with kv_rank >= 0 one ring step (float32 out),
  // with kv_rank < 0 the all-gather mode (output dtype)
  const bool local = q_rank >= 0;
  const bool partial = local && kv_rank >= 0;
  p.q_tiles = (local ? p.m.c : R.T) / tcfwd::kTile;
  p.q_rank = local ? q_rank : -1;
  p.kv_rank = partial ? kv_rank : -1;
  p.o = o;
  p.lse = lse;
  p.status = status;
  p.debug_fault = R.debug_fault;
  p.doc_lo = doc_lo;
  p.ord_q = ord_q;
  const int items = R.B * R.Hq * p.q_tiles;
  if (items == 0) return cudaSuccess;
  p.n_items = items;
  const bool packed = doc_lo != nullptr;  // ring mode only (checked by the caller)
  timing_begin(partial  ? "tc_partial_fwd"
               : local  ? "tc_allgather_fwd"
               : packed ? "tc_packed_fwd"
                        : "tc_ring_fwd",
               st);
  cudaError_t e;
  if (R.D == 128)
    e = partial  ? run_fwd<128, true>(R, p, items, q, k, v, st)
        : packed ? run_fwd<128, false, true>(R, p, items, q, k, v, st)
                 : run_fwd<128, false>(R, p, items, q, k, v, st);
  else
    e = partial  ? run_fwd<64, true>(R, p, items, q, k, v, st)
        : packed ? run_fwd<64, false, true>(R, p, items, q, k, v, st)
                 : run_fwd<64, false>(R, p, items, q, k, v, st);
  timing_end(st);
  return e;
}

}  // namespace cpattn
