// Ring-attention forward on the 5th-generation tensor cores (sm_103a).
//
// What one CTA computes: two 128-row query tiles (A and B) of one sequence
// against every key/value tile their rows can see, visited in ring order --
// step i of rank r holds the K/V chunk of rank (r - i) mod cp (tutorial
// "上下文并行", section "朴素 Ring Attention") -- with the running max / sum /
// output carried across steps, i.e. the per-step partials merged by the
// single-pass online softmax (pull request "Feat: Context Parallel" #181, mode
// "p2p").  Tiles wholly hidden by the causal mask (key position > query
// position for every pair) are skipped; diagonal tiles are masked per element
// from global positions.  Pairing: with an even number of query heads per K/V
// head the two tiles are two query heads of the same group at the same rows
// (they share every K/V tile and every mask decision); otherwise they are two
// consecutive 128-token tiles of one head.
//
// Warp roles (384 threads):
//   warp 0        TMA producer: Q tiles once, then K tiles through a ring of
//                 shared-memory stages (128-byte swizzle); warp 3: V tiles
//                 through a ring of their own.
//   warps 1, 2    MMA issuers, one thread each, warp 1 for tile A and warp 2
//                 for tile B: S_X = Q_X K^T into TMEM (SS form), O_X += P_X V
//                 with P read from TMEM (TS form).
//   warps 4..7    softmax of tile A; warps 8..11 softmax of tile B.  Thread =
//                 row: tcgen05.ld of its S row, causal mask, row max, P =
//                 2^(s*scale*log2e - m) rounded to bf16 into TMEM, row sum in
//                 fp32.  The output is rescaled only when the running max grows
//                 by more than 2^8 (exact after the final division by the sum).
//   epilogue      O / l rounded once to the output dtype, LSE = ln(l) + m.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256, 256+D),
// O_B [256+D, 256+2D); P_X overwrites the first 64 columns of S_X.
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

enum : int { kEmpty = 0, kFull = 1, kDiag = 2 };

struct Params {
  int B, Hq, Hkv, T, n_rep;
  SeqMap m;
  float scale_log2;
  int head_pairs;      // 1: tiles A/B are query heads 2u, 2u+1 at the same rows
  int tiles_per_item;  // row pairing: 2 consecutive 128-token tiles, or 1
  int n_hu;            // head units per batch (H_q/2 with head pairs, else H_q)
  int q_tiles;         // 128-row query tiles per sequence in the launch
  int q_rank, kv_rank; // partial mode when q_rank >= 0
  void* o;
  float* lse;
  int* status;
  int debug_fault;
};

template <int D>
struct Smem {
  // K and V have rings of their own: K is last read by the S products early in a
  // step, V by the PV products at its end, so K is refilled a step sooner and
  // takes the extra stage.
  static constexpr int kKStages = D == 128 ? 3 : 5;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = 2 * kTileBytes;
  static constexpr int kV = kK + kKStages * kTileBytes;
  static constexpr int kBar = kV + kVStages * kTileBytes;
  // barriers: q_full[2], k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2],
  // p_full[2], pv_done[2], final[2] (one per issuer)
  static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 6 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16 + 1024;  // + alignment slack
};

struct Item {
  int b, g, rank;
  int h[2], slot0[2], pos0[2];
  int active[2];
};

__device__ __forceinline__ Item decode(const Params& p, int w) {
  Item it;
  const int units = p.B * p.n_hu;
  const int ti = w / units;
  const int rem = w - ti * units;
  it.b = rem / p.n_hu;
  const int hu = rem - it.b * p.n_hu;
  const int tpi = p.tiles_per_item;
  if (p.q_rank >= 0) {
    it.slot0[0] = p.q_rank * p.m.c + ti * tpi * kTile;
    it.pos0[0] = p.m.pos(it.slot0[0]);
  } else {
    // heaviest (latest) query positions first: causal work grows with position
    const int n_pos_items = p.q_tiles / tpi;
    it.pos0[0] = (n_pos_items - 1 - ti) * tpi * kTile;
    it.slot0[0] = p.m.slot(it.pos0[0]);
  }
  if (p.head_pairs) {
    it.h[0] = 2 * hu;
    it.h[1] = 2 * hu + 1;
    it.slot0[1] = it.slot0[0];
    it.pos0[1] = it.pos0[0];
    it.active[1] = 1;
  } else {
    it.h[0] = hu;
    it.h[1] = hu;
    it.slot0[1] = it.slot0[0] + kTile;
    it.pos0[1] = it.pos0[0] + kTile;
    it.active[1] = tpi == 2;
  }
  it.active[0] = 1;
  it.g = it.h[0] / p.n_rep;
  it.rank = it.slot0[0] / p.m.c;
  return it;
}

__device__ __forceinline__ int classify(int qpos0, int kpos0) {
  if (kpos0 + kTile - 1 <= qpos0) return kFull;
  if (kpos0 > qpos0 + kTile - 1) return kEmpty;
  return kDiag;  // tiles are aligned on the same 128-position grid: kpos0 == qpos0
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

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using L = Smem<D>;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBar;
  auto q_full = [&](int x) { return bars + 8 * x; };
  auto k_full = [&](int s) { return bars + 8 * (2 + s); };
  auto k_empty = [&](int s) { return bars + 8 * (2 + KS + s); };
  auto v_full = [&](int s) { return bars + 8 * (2 + 2 * KS + s); };
  auto v_empty = [&](int s) { return bars + 8 * (2 + 2 * KS + VS + s); };
  const uint32_t tile_bars = bars + 8 * (2 + 2 * KS + 2 * VS);
  auto s_full = [&](int x) { return tile_bars + 8 * x; };
  auto p_full = [&](int x) { return tile_bars + 8 * (2 + x); };
  auto pv_done = [&](int x) { return tile_bars + 8 * (4 + x); };
  auto final_bar = [&](int x) { return tile_bars + 8 * (6 + x); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = p.debug_fault ? kDebugTimeoutNs : kTimeoutNs;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) {
      const uint32_t b = bars + 8 * i;
      const bool softmax_arrivals = b == p_full(0) || b == p_full(1);
      // a K or V stage is free once both issuers' MMAs that read it have completed
      const bool both_issuers = (b >= k_empty(0) && b < k_empty(0) + 8 * KS) ||
                                (b >= v_empty(0) && b < v_empty(0) + 8 * VS);
      mbar_init(b, softmax_arrivals ? 128 : both_issuers ? 2 : 1);
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

  const Item it = decode(p, blockIdx.x);
  // K/V tiles in ring order: chunks r, r-1, ..., r-cp+1 (mod cp), or one chunk
  const int kv_first = p.q_rank >= 0 ? p.kv_rank : it.rank;
  const int kv_chunks = p.q_rank >= 0 ? 1 : p.m.cp;
  const int kv_row_base = (it.b * p.Hkv + it.g) * p.T;

  if (warp < 4) {
  regs_ctl();  // warpgroup 0: TMA producers (warps 0, 3) and MMA issuers (warps 1, 2)
  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ producers
    // warp 0: the Q tiles, then the K tiles; warp 3: the V tiles
    if (lane == 0) {
      const bool is_k = warp == 0;
      const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
      tma_prefetch_desc(tm);
      int q_issued[2] = {0, 0};
      if (is_k) {
        tma_prefetch_desc(&tm_q);
        for (int x = 0; x < 2; ++x) {
          if (!it.active[x]) continue;
          if (x == 0 && p.debug_fault) continue;  // fault hook: this load never happens
          mbar_expect_tx(q_full(x), L::kTileBytes);
          const int row = (it.b * p.Hq + it.h[x]) * p.T + it.slot0[x];
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_2d(sbase + L::kQ + x * L::kTileBytes + kb * (kTile * 128), &tm_q, kb * 64,
                        row, q_full(x));
          q_issued[x] = 1;
        }
      }
      const int nst = is_k ? KS : VS;
      const uint32_t base = sbase + (is_k ? L::kK : L::kV);
      int stage = 0, par = 0;
      uint32_t issued = 0, issued_par = 0;  // bit s: stage s loaded / its phase parity
      TileWalk wk;
      for (wk.start(p.m, kv_first, kv_chunks, -1, 1); !wk.done(); wk.next()) {
        const int kpos = wk.pos();
        const int ca = classify(it.pos0[0], kpos);
        const int cb = it.active[1] ? classify(it.pos0[1], kpos) : kEmpty;
        if (ca == kEmpty && cb == kEmpty) continue;
        const uint32_t empty = is_k ? k_empty(stage) : v_empty(stage);
        const uint32_t full = is_k ? k_full(stage) : v_full(stage);
        if (!mbar_wait(empty, par ^ 1, abort, p.status, tmo)) break;
        const int row = kv_row_base + wk.slot();
        mbar_expect_tx(full, L::kTileBytes);
        for (int kb = 0; kb < D / 64; ++kb)
          tma_load_2d(base + stage * L::kTileBytes + kb * (kTile * 128), tm, kb * 64, row, full);
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | ((uint32_t)par << stage);
        if (++stage == nst) stage = 0, par ^= 1;
      }
      // never leave with a copy still writing into this CTA's shared memory
      for (int x = 0; x < 2; ++x)
        if (q_issued[x]) drain_wait(q_full(x), 0);
      for (int st = 0; st < nst; ++st)
        if ((issued >> st) & 1u)
          drain_wait(is_k ? k_full(st) : v_full(st), (issued_par >> st) & 1u);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // One issuer per query tile (warp 1: A, warp 2: B).  A tcgen05.mma takes a
    // thread about 35-50 cycles to issue against 64 cycles to run at N = 128 and
    // the tensor pipe queues only a few, so a single thread serving both softmax
    // warpgroups in turn puts one tile's PV and the next step's waits on the other
    // tile's S -> softmax -> PV chain; with a thread per tile each chain runs on
    // its own.  Both issuers wait for every K and V load, even one their tile does
    // not use, so their k_empty / v_empty arrivals stay one per load.
    if (lane == 0) {
      const int x = warp - 1;
      constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(128, D, false, true);
      bool ok = true;
      if (it.active[x]) ok = mbar_wait(q_full(x), 0, abort, p.status, tmo);
      tc_fence_after();
      // descriptor bases; per k-step offsets are compile-time constants (16-byte units)
      constexpr uint32_t kTileDesc = L::kTileBytes >> 4;
      const uint64_t qd = sdesc_sw128(sbase + L::kQ, 16, 1024) + (uint64_t)(x * kTileDesc);
      const uint64_t kd0 = sdesc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t vd0 = sdesc_sw128(sbase + L::kV, kTile * 128, 1024);
      StageRing<KS> kr;
      StageRing<VS> vr;
      int cnt = 0, cnt_other = 0;  // S products issued so far by this / the other issuer
      TileWalk wk;
      for (wk.start(p.m, kv_first, kv_chunks, -1, 1); !wk.done() && ok; wk.next()) {
        const int kpos = wk.pos();
        const int ca = classify(it.pos0[0], kpos);
        const int cb = it.active[1] ? classify(it.pos0[1], kpos) : kEmpty;
        if (ca == kEmpty && cb == kEmpty) continue;  // the producers skip these too
        const bool mine = (x == 0 ? ca : cb) != kEmpty;
        const bool other = (x == 0 ? cb : ca) != kEmpty;
        if (!(ok = mbar_wait(k_full(kr.stage), kr.par, abort, p.status, tmo))) break;
        if (mine) {
          // S_X = Q_X K^T; the S region is free once the previous PV has read P_X
          if (cnt > 0 && !(ok = mbar_wait(pv_done(x), (cnt - 1) & 1, abort, p.status, tmo)))
            break;
          // Ping-pong: the S products alternate A(j), B(j), A(j+1), ... -- S_B of a
          // K/V tile waits for S_A of the same tile and S_A for S_B of the tile
          // before -- so one tile's softmax runs while the tensor pipe serves the
          // other tile instead of both softmax warpgroups contending at once.  Each
          // issuer is thereby at most one S phase ahead of the other, which keeps
          // these parity waits unambiguous.
          if (x == 1 && other &&
              !(ok = mbar_wait(s_full(0), cnt_other & 1, abort, p.status, tmo)))
            break;
          if (x == 0 && cnt_other > 0 &&
              !(ok = mbar_wait(s_full(1), (cnt_other - 1) & 1, abort, p.status, tmo)))
            break;
          tc_fence_after();
          const uint64_t kd = kd0 + (uint64_t)(kr.stage * kTileDesc);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;  // 16 KiB blocks, 32 B steps
            mma_ss(tmem + x * 128, qd + off, kd + off, kIdescS, kk > 0);
          }
          mma_commit(s_full(x));
        }
        mma_commit(k_empty(kr.stage));  // arrives at once if nothing was issued
        if (!(ok = mbar_wait(v_full(vr.stage), vr.par, abort, p.status, tmo))) break;
        if (mine) {
          // O_X += P_X V
          if (!(ok = mbar_wait(p_full(x), cnt & 1, abort, p.status, tmo))) break;
          tc_fence_after();
          const uint64_t vd = vd0 + (uint64_t)(vr.stage * kTileDesc);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)  // 16 key rows = 2048 B per k-step
            mma_ts(tmem + 256 + x * D, tmem + x * 128 + kk * 8, vd + kk * 128, kIdescPV,
                   (cnt > 0 || kk > 0) ? 1u : 0u);
          mma_commit(pv_done(x));
          ++cnt;
        }
        mma_commit(v_empty(vr.stage));
        if (other) ++cnt_other;
        kr.advance();
        vr.advance();
      }
      // every MMA this thread issued has finished before TMEM can be freed
      mma_commit(final_bar(x));
      drain_wait(final_bar(x), 0);
    }
  }
  } else {
    regs_math();  // warpgroups 1 and 2: softmax / gradient math
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;  // tile A (warps 4..7) or B (warps 8..11)
    const int quad = warp & 3;      // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + x * 128;
    const uint32_t t_o = tmem + lane_off + 256 + x * D;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    int cnt = 0;
    bool ok = true;
    if (it.active[x]) {
      TileWalk wk;
      for (wk.start(p.m, kv_first, kv_chunks, -1, 1); !wk.done(); wk.next()) {
        const int kpos = wk.pos();
        const int cls = classify(it.pos0[x], kpos);
        if (cls == kEmpty) continue;
        if (!(ok = warp_wait(s_full(x), cnt & 1, abort, p.status, tmo))) break;
        tc_fence_after();
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, r[c]);
        tmem_wait_ld();
        float mx = -INFINITY;
        if (cls == kDiag) {
          // key column j is visible iff kpos + j <= qpos + row
          const int thr = row + it.pos0[x] - kpos;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j > thr) r[c][j] = __float_as_uint(-INFINITY);
        }
        {
          // 8 independent chains of three-input max over the 128 scores
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 32; j += 2)
              m8[(c * 16 + j / 2) & 7] = max3(m8[(c * 16 + j / 2) & 7], __uint_as_float(r[c][j]),
                                              __uint_as_float(r[c][j + 1]));
          mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        }
        const float m_new = fmaxf(m_run, mx * sl2);
        bool rescale = false;
        float factor = 1.f;
        if (cnt == 0) {
          m_run = m_new;
        } else if (m_new > m_run + 8.f) {
          factor = ex2(m_run - m_new);
          l_run *= factor;
          m_run = m_new;
          rescale = true;
        }
        const float mu = m_run == -INFINITY ? 0.f : m_run;
        // P = 2^(s * scale * log2e - m): exponent arguments and row sums two lanes per
        // instruction (packed fp32x2), 2^x on the special-function unit
        const float2 sl2v = make_float2(sl2, sl2), nmu = make_float2(-mu, -mu);
        float2 l4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) l4[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 x = fma2(make_float2(__uint_as_float(r[c][2 * j]),
                                              __uint_as_float(r[c][2 * j + 1])), sl2v, nmu);
            const float2 pp = make_float2(ex2(x.x), ex2(x.y));
            l4[j & 3] = add2(l4[j & 3], pp);
            pk[j] = pack_bf16(pp.x, pp.y);
          }
          tmem_st16(t_s + c * 16, pk);
        }
        l_run += ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) + ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));
        tmem_wait_st();
        if (cnt > 0 && __any_sync(0xffffffffu, rescale)) {
          // the output so far must be final in TMEM before it is rescaled
          if (!(ok = warp_wait(pv_done(x), (cnt - 1) & 1, abort, p.status, tmo))) break;
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
        mbar_arrive(p_full(x));
        ++cnt;
      }
      // -------------------------------------------------------- epilogue
      if (ok && cnt > 0) ok = warp_wait(pv_done(x), (cnt - 1) & 1, abort, p.status, tmo);
      if (ok) {
        tc_fence_after();
        const bool partial = p.q_rank >= 0;
        const int64_t bh = (int64_t)it.b * p.Hq + it.h[x];
        const int64_t orow = partial ? bh * p.m.c + (it.slot0[x] - p.q_rank * p.m.c) + row
                                     : bh * p.T + it.slot0[x] + row;
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o32[32];
          if (cnt > 0) {
            tmem_ld32(t_o + c * 32, o32);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o32[j] = 0u;
          }
          if (OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * D + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(o32[4 * j]) * inv,
                                   __uint_as_float(o32[4 * j + 1]) * inv,
                                   __uint_as_float(o32[4 * j + 2]) * inv,
                                   __uint_as_float(o32[4 * j + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D +
                                                  c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 v4;
              v4.x = pack_bf16(__uint_as_float(o32[8 * j + 0]) * inv,
                               __uint_as_float(o32[8 * j + 1]) * inv);
              v4.y = pack_bf16(__uint_as_float(o32[8 * j + 2]) * inv,
                               __uint_as_float(o32[8 * j + 3]) * inv);
              v4.z = pack_bf16(__uint_as_float(o32[8 * j + 4]) * inv,
                               __uint_as_float(o32[8 * j + 5]) * inv);
              v4.w = pack_bf16(__uint_as_float(o32[8 * j + 6]) * inv,
                               __uint_as_float(o32[8 * j + 7]) * inv);
              dst[j] = v4;
            }
          }
        }
        p.lse[orow] = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
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

}  // namespace tcfwd

bool tc_supported(const Ring& R) {
  if (!R.bf16 || (R.D != 64 && R.D != 128)) return false;
  const int c = R.T / R.cp;
  const int seg = R.zz ? c / 2 : c;
  if (seg % tcfwd::kTile) return false;
  if ((double)R.B * R.Hq * R.T >= 2147483647.0) return false;
  return true;
}

template <int D, bool F32>
static cudaError_t run_fwd(const Ring& R, const tcfwd::Params& p, int items, const void* q,
                           const void* k, const void* v, cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  if (encode_tmap_2d_bf16(&tq, q, D, (uint64_t)R.B * R.Hq * R.T, 64, tcfwd::kTile) != CUDA_SUCCESS ||
      encode_tmap_2d_bf16(&tk, k, D, (uint64_t)R.B * R.Hkv * R.T, 64, tcfwd::kTile) != CUDA_SUCCESS ||
      encode_tmap_2d_bf16(&tv, v, D, (uint64_t)R.B * R.Hkv * R.T, 64, tcfwd::kTile) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  constexpr int kSmem = tcfwd::Smem<D>::kBytes;
  auto kern = tcfwd::fwd_kernel<D, F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if ((e = check_register_split(kern, tcfwd::kThreads)) != cudaSuccess) return e;
  kern<<<items, tcfwd::kThreads, kSmem, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_tc_fwd(const Ring& R, int q_rank, int kv_rank, const void* q, const void* k,
                          const void* v, void* o, float* lse, int* status, cudaStream_t st) {
  tcfwd::Params p;
  p.B = R.B;
  p.Hq = R.Hq;
  p.Hkv = R.Hkv;
  p.T = R.T;
  p.n_rep = R.Hq / R.Hkv;
  p.m = SeqMap::make(R.T, R.cp, R.zz);
  p.scale_log2 = R.scale * 1.44269504088896340736f;
  p.head_pairs = (p.n_rep % 2) == 0;
  const int seg_tiles = (R.zz ? p.m.c / 2 : p.m.c) / tcfwd::kTile;
  p.tiles_per_item = (!p.head_pairs && seg_tiles % 2 == 0) ? 2 : 1;
  p.n_hu = p.head_pairs ? R.Hq / 2 : R.Hq;
  const bool partial = q_rank >= 0;
  p.q_tiles = (partial ? p.m.c : R.T) / tcfwd::kTile;
  p.q_rank = partial ? q_rank : -1;
  p.kv_rank = partial ? kv_rank : -1;
  p.o = o;
  p.lse = lse;
  p.status = status;
  p.debug_fault = R.debug_fault;
  const int items = R.B * p.n_hu * (p.q_tiles / p.tiles_per_item);
  if (items == 0) return cudaSuccess;
  timing_begin(partial ? "tc_partial_fwd" : "tc_ring_fwd", st);
  cudaError_t e;
  if (R.D == 128)
    e = partial ? run_fwd<128, true>(R, p, items, q, k, v, st)
                : run_fwd<128, false>(R, p, items, q, k, v, st);
  else
    e = partial ? run_fwd<64, true>(R, p, items, q, k, v, st)
                : run_fwd<64, false>(R, p, items, q, k, v, st);
  timing_end(st);
  return e;
}

}  // namespace cpattn
