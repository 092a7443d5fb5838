// Shared device helpers: token position maps of the emulated ranks, the device
// status word, bounded mbarrier waits, and thin inline-PTX wrappers for TMA,
// tcgen05 (MMA, TMEM alloc/ld/st) on sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace cpattn {

// Device status codes (the values of cpattn_status).
constexpr int kStatusLaunch = 3;   // a kernel found its launch unusable (reported as a CUDA error)
constexpr int kStatusTimeout = 4;
constexpr int kStatusBounds = 5;   // a bounds check of a CPATTN_DEBUG build failed

// ---------------------------------------------------------------------------
// Token position maps.  Slot = index on the layout-order token axis; position =
// natural (global) index.  Contiguous: identity.  Zigzag over `cp` ranks
// (tutorial "上下文并行", section "Zig-Zag Ring Attention"): 2*cp chunks of
// h = T/(2cp) tokens; rank r's slots [r*c, (r+1)*c) hold chunk r then chunk
// 2cp-1-r.
// ---------------------------------------------------------------------------
struct SeqMap {
  int T, cp, c, h, zz;

  __host__ __device__ static SeqMap make(int T, int cp, int zigzag) {
    SeqMap m;
    m.T = T;
    m.cp = cp;
    m.c = T / cp;
    m.h = m.c / 2;
    m.zz = zigzag;
    return m;
  }
  __host__ __device__ __forceinline__ int pos(int slot) const {
    if (!zz) return slot;
    int r = slot / c, w = slot - r * c;
    return w < h ? r * h + w : (2 * cp - 1 - r) * h + (w - h);
  }
  __host__ __device__ __forceinline__ int slot(int p) const {
    if (!zz) return p;
    int ch = p / h, w = p - ch * h;
    return ch < cp ? ch * c + w : (2 * cp - 1 - ch) * c + h + w;
  }
  __host__ __device__ __forceinline__ int rank_of_slot(int s) const { return s / c; }
};

// Walk over the 128-token tiles of consecutive ring chunks without integer
// divisions: `nchunks` chunks starting at `first`, stepping by `dir` (-1: the
// order in which a rank receives K/V chunks, +1: the order in which a chunk's
// gradient travels back), `reps` passes over each chunk's tiles (the query heads
// of a K/V group), tiles of a chunk in slot order.
struct TileWalk {
  int cp, c, h, zz, tpc, reps, dir, nchunks;
  int i, rep, t, s;
  __device__ __forceinline__ void start(const SeqMap& m, int first, int n, int direction,
                                        int repeats) {
    cp = m.cp;
    c = m.c;
    h = m.h;
    zz = m.zz;
    tpc = m.c >> 7;
    reps = repeats;
    dir = direction;
    nchunks = n;
    i = 0;
    rep = 0;
    t = 0;
    s = first;
  }
  __device__ __forceinline__ bool done() const { return i >= nchunks; }
  __device__ __forceinline__ int slot() const { return s * c + (t << 7); }
  __device__ __forceinline__ int pos() const {
    const int w = t << 7;
    if (!zz) return s * c + w;
    return w < h ? s * h + w : (2 * cp - 1 - s) * h + (w - h);
  }
  __device__ __forceinline__ void next() {
    if (++t == tpc) end_pass();
  }
  // The next pass over this chunk's tiles, or the next chunk after the last pass.
  __device__ __forceinline__ void end_pass() {
    t = 0;
    if (++rep == reps) {
      rep = 0;
      ++i;
      s += dir;
      if (s < 0) s += cp;
      else if (s >= cp) s -= cp;
    }
  }
  // The next chunk, whatever pass this is.
  __device__ __forceinline__ void end_chunk() {
    rep = reps - 1;
    end_pass();
  }

  // Query-stationary walks over key tiles: move to the next key tile that the
  // query tile at q0 sees (a key tile is hidden when its first position is past
  // the query tile's last row).  Inside a chunk the tile positions grow with t (in
  // the zigzag layout the late half follows the early one), so the visible key
  // tiles of a chunk are a prefix: the first hidden tile ends the pass, and a chunk
  // whose first tile is hidden is left at once.  The tiles visited, and their
  // order, are those of stepping through every tile and skipping the hidden ones.
  __device__ __forceinline__ void settle_keys(int q0) {
    while (!done() && pos() > q0 + 127) {
      if (t == 0) end_chunk();  // the chunk's first tile is hidden: all of it is
      else end_pass();          // the rest of this pass is hidden
    }
  }

  // Key-stationary walks over query tiles (a K/V tile at k0 is seen by the query
  // tiles at or after its position): inside a pass the visible query tiles are a
  // suffix, so at the start of each pass jump to its first visible tile, or past the
  // chunk when none of its tiles is visible.  The tiles visited, and their order, are
  // those of stepping through every tile and skipping the hidden ones.
  __device__ __forceinline__ void settle_queries(int k0) {
    while (!done() && t == 0) {
      int f;  // first tile of the pass at or after k0 (tpc: none)
      if (!zz) {
        const int p0 = s * c;
        f = k0 <= p0 ? 0 : k0 < p0 + c ? (k0 - p0) >> 7 : tpc;
      } else {
        const int e0 = s * h, l0 = (2 * cp - 1 - s) * h, th = h >> 7;
        f = k0 <= e0 ? 0
            : k0 < e0 + h ? (k0 - e0) >> 7
            : k0 <= l0 ? th
            : k0 < l0 + h ? th + ((k0 - l0) >> 7)
            : tpc;
      }
      if (f < tpc) {
        t = f;
        return;
      }
      end_chunk();
    }
  }
};

// Walk over the 128-token tiles of a range of NATURAL positions, tiles
// [first, last] in order, `reps` passes (the query heads of a K/V group).  Packed
// sequences use it: the tiles a tile pair can see form one contiguous natural
// range (a document's), so nothing has to be skipped.  Same interface as TileWalk.
struct NatWalk {
  SeqMap m;
  int t, first, last, rep, reps;
  __device__ __forceinline__ void start(const SeqMap& mm, int first_tile, int last_tile,
                                        int repeats) {
    m = mm;
    first = first_tile;
    last = last_tile;
    t = first_tile;
    rep = 0;
    reps = first_tile <= last_tile ? repeats : 0;
  }
  __device__ __forceinline__ bool done() const { return rep >= reps; }
  __device__ __forceinline__ int pos() const { return t << 7; }
  __device__ __forceinline__ int slot() const { return m.slot(t << 7); }
  __device__ __forceinline__ void next() {
    if (++t > last) {
      t = first;
      ++rep;
    }
  }
};

// Position in a ring of N shared-memory stages fed by TMA: the current stage,
// the parity of its current mbarrier phase, and (for the producer's drain
// before exit) which stages ever received a copy and the parity of the last one.
template <int N>
struct StageRing {
  int stage = 0;
  uint32_t par = 0;
  uint32_t issued = 0, ipar = 0;
  __device__ __forceinline__ void advance() {
    if (++stage == N) {
      stage = 0;
      par ^= 1u;
    }
  }
  __device__ __forceinline__ void mark_issued() {
    issued |= 1u << stage;
    ipar = (ipar & ~(1u << stage)) | (par << stage);
  }
  __device__ __forceinline__ bool was_issued(int st) const { return (issued >> st) & 1u; }
  __device__ __forceinline__ uint32_t issued_parity(int st) const { return (ipar >> st) & 1u; }
};

// The k-th work item of a persistent CTA, or -1: resident CTAs walk a
// heaviest-first item list in a snake (rounds of gridDim.x items, every other
// round reversed), which evens out the per-CTA totals.
// Programmatic dependent launch: let the grid launched after this one as its
// programmatic dependent start once every CTA here has executed this (or exited) ...
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// ... and, in that dependent, wait until the grids it depends on have completed and
// their memory operations are visible (returns at once in a grid launched normally).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ int item_of(int k, int n_items) {
  const int G = gridDim.x;
  const int w = k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  return w < n_items ? w : -1;
}

__device__ __forceinline__ void latch_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Bounds checks of the tensor-core kernels' hand-computed global rows (TMA tile
// rows, statistics loads, epilogue stores).  A build with CPATTN_DEBUG defined
// evaluates them: a failed check latches CPATTN_ERR_BOUNDS in the device status
// word and the caller skips the access (a skipped load then also ends in a
// bounded-wait time-out).  Other builds compile them away.
__device__ __forceinline__ bool in_bounds(int64_t first, int64_t count, int64_t extent,
                                          int* status) {
#ifdef CPATTN_DEBUG
  if (first >= 0 && count >= 0 && first + count <= extent) return true;
  latch_status(status, kStatusBounds);
  return false;
#else
  (void)first, (void)count, (void)extent, (void)status;
  return true;
#endif
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// elect.sync: true in exactly one lane of the (converged) warp.  The MMA issuers
// run as whole warps, so that descriptor arithmetic stays warp-uniform, and issue
// each tcgen05 instruction from the elected lane.
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(e));
  return e != 0;
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.  Gives up (returns
// false) when *abort becomes non-zero or after timeout_ns of wall time; an
// iteration cap backs the time limit up.  On its own time-out it raises *abort
// and latches the device status word, so every other role of the CTA stops too.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) break;
    }
  }
  *abort = 1;
  latch_status(status, kStatusTimeout);
  return false;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk) loads into shared memory, completing on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Plain bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA tensor store of one box from shared memory (this CTA's) to global memory,
// tracked by the issuing thread's bulk groups.  x: innermost coordinate (elements).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
// The same box added element-wise into global memory (the tensor map's element type;
// float32 adds round to nearest even, as a plain add would).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, int x, int y,
                                                  uint32_t src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The issuing thread's bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// The issuing thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA (cta_group::1).
// TMEM address: bits 31..16 lane, 15..0 column.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier arrives once every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor of kind::f16: bf16 A and B, f32 accumulator, M x N.
// a_mn / b_mn select the MN-major (transposed) operand layout.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                              // accumulator format: f32
         | (1u << 7)                            // A format: bf16
         | (1u << 10)                           // B format: bf16
         | ((a_mn ? 1u : 0u) << 15)             // A major-ness
         | ((b_mn ? 1u : 0u) << 16)             // B major-ness
         | ((uint32_t)(N >> 3) << 17)           // N / 8
         | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// Shared-memory matrix descriptor with 128-byte swizzling.
//  K-major operand (rows of 128 bytes, 8-row groups of 1024 bytes): sbo = 1024,
//    lbo unused (16).
//  MN-major operand: lbo = byte distance between 64-element blocks along M/N,
//    sbo = byte distance between 8-row groups along K (1024).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;   // swizzle: 128 B
  return d;
}

// ---- TMEM <-> registers, 32 lanes x 32-bit, one row per thread ------------
#define CPATTN_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                     "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define CPATTN_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                     "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : CPATTN_R8(0), CPATTN_R8(8), CPATTN_R8(16), CPATTN_R8(24)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : CPATTN_R8(0), CPATTN_R8(8)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      CPATTN_W8(0), CPATTN_W8(8), CPATTN_W8(16), CPATTN_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      CPATTN_W8(0), CPATTN_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Register split between warpgroups (setmaxnreg): the control warpgroup (TMA
// producer, MMA issuer) gives registers back, the math warpgroups take them.
// The sum over the block must not exceed what the launch allocated (checked on
// the host against the kernel's compiled register count before every launch).
constexpr uint32_t kRegsCtl = 80;
constexpr uint32_t kRegsMath = 208;
__device__ __forceinline__ void regs_ctl() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
}
__device__ __forceinline__ void regs_math() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsMath));
}

// ---------------------------------------------------------------------------
// Small arithmetic helpers
// ---------------------------------------------------------------------------
// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed two-lane fp32 arithmetic (sm_100 and later): one issue slot for two
// lanes' worth of FP32 work.  The kernels' softmax phases are issue-bound, so
// these halve their FMA/ADD/MUL instruction count.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// max(a, b, c) in one instruction (three-input form of max.f32, sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace cpattn
