// cpattn_ring_step_host: one forward + backward step of the ring over tensors that
// live in host memory, with the host<->device transfers overlapping the compute.
//
// The problem splits into n independent groups: batch rows when B is even, else
// (B = 1) K/V heads with their query heads when H_kv is even.  Group j of every
// tensor is the j-th contiguous n-th of it, so each group is a smaller problem of
// the same kind.  Two copy streams per device, created once, carry the transfers:
//
//   upload stream    q, k, v of group 0, 1, ...; then dO of group 0, 1, ...
//   caller's stream  per group: permute q, k, v to layout order, ring forward,
//                    permute o and LSE back; then per group: permute dO, ring
//                    backward, permute dq, dk, dv back
//   download stream  o and LSE of a group as soon as its forward is done; dq, dk,
//                    dv of a group as soon as its backward is done
//
// so a group's uploads run while the previous group computes, and its downloads
// while the next one does.  The caller's stream waits for the last download, so
// the call's work is complete when that stream's work is.
#include <mutex>

#include "../../include/cpattn.h"
#include "kernels.h"

namespace cpattn {
namespace {

constexpr int kMaxGroups = 2;
// events per device: start, end, and per group: inputs landed, dO landed, forward
// outputs ready, gradients ready
constexpr int kEventsPerGroup = 4;
constexpr int kNumEvents = 2 + kEventsPerGroup * kMaxGroups;

struct CopyStreams {
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t ev[kNumEvents] = {};
  std::mutex mu;  // one call's enqueue at a time per device (the events are shared)
  bool ready = false;
};
CopyStreams g_copy[128];
std::mutex g_copy_mu;

CopyStreams* copy_streams() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(g_copy_mu);
  CopyStreams& c = g_copy[dev];
  if (!c.ready) {
    if (cudaStreamCreateWithFlags(&c.up, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c.down, cudaStreamNonBlocking) != cudaSuccess)
      return nullptr;
    for (auto& e : c.ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    c.ready = true;
  }
  return &c;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Device workspace of a step: natural-order staging of q, k, v, dO (reused for the
// natural-order o, dk, dv, dq on the way back), the layout-order q, k, v, dO, o,
// LSE, dq, dk, dv, the natural-order LSE, and the backward's own workspace (sized
// for one group; the groups run one after another on the caller's stream).
struct StepLayout {
  size_t q, kv, lse, bwd;  // bytes of a q-sized and a k-sized tensor, an LSE, bwd workspace
  size_t stage_q, stage_k, stage_v, stage_do;
  size_t lay_q, lay_k, lay_v, lay_do, lay_o, lay_lse, lay_dq, lay_dk, lay_dv;
  size_t nat_lse, bwd_ws, total;
};

// Two groups when the problem splits into independent halves whose slices of every
// tensor (q, k, the LSE) start on 16-byte boundaries; else one.
int groups_of(const cpattn_desc* d) {
  if (!(d->B % 2 == 0 || (d->B == 1 && d->H_kv % 2 == 0))) return 1;
  const size_t elt = d->dtype == CPATTN_BF16 ? 2 : 4;
  const size_t q = (size_t)d->B * d->H_q * d->T * d->D * elt / 2;
  const size_t k = (size_t)d->B * d->H_kv * d->T * d->D * elt / 2;
  const size_t l = (size_t)d->B * d->H_q * d->T * sizeof(float) / 2;
  return q % 16 == 0 && k % 16 == 0 && l % 16 == 0 ? 2 : 1;
}

cpattn_desc group_desc(const cpattn_desc* d, int n) {
  cpattn_desc g = *d;
  if (n > 1) {
    if (d->B % n == 0) {
      g.B = d->B / n;
    } else {
      g.H_q = d->H_q / n;
      g.H_kv = d->H_kv / n;
    }
  }
  return g;
}

StepLayout layout_of(const cpattn_desc* d) {
  StepLayout s;
  const size_t elt = d->dtype == CPATTN_BF16 ? 2 : 4;
  s.q = round256((size_t)d->B * d->H_q * d->T * d->D * elt);
  s.kv = round256((size_t)d->B * d->H_kv * d->T * d->D * elt);
  s.lse = round256((size_t)d->B * d->H_q * d->T * sizeof(float));
  const cpattn_desc g = group_desc(d, groups_of(d));
  s.bwd = round256(cpattn_ring_bwd_workspace(&g));
  size_t off = 0;
  auto take = [&](size_t b) {
    const size_t at = off;
    off += b;
    return at;
  };
  s.stage_q = take(s.q);
  s.stage_k = take(s.kv);
  s.stage_v = take(s.kv);
  s.stage_do = take(s.q);
  s.lay_q = take(s.q);
  s.lay_k = take(s.kv);
  s.lay_v = take(s.kv);
  s.lay_do = take(s.q);
  s.lay_o = take(s.q);
  s.lay_lse = take(s.lse);
  s.lay_dq = take(s.q);
  s.lay_dk = take(s.kv);
  s.lay_dv = take(s.kv);
  s.nat_lse = take(s.lse);
  s.bwd_ws = take(s.bwd);
  s.total = off;
  return s;
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" size_t cpattn_ring_step_host_workspace(const cpattn_desc* desc) {
  if (cpattn_ring_bwd_workspace(desc) == 0 || desc->a2a != 1) return 0;
  return layout_of(desc).total;
}

extern "C" cpattn_status cpattn_ring_step_host(const cpattn_desc* desc, const void* q,
                                               const void* k, const void* v, const void* dO,
                                               void* o, float* lse, void* dq, void* dk, void* dv,
                                               void* workspace, size_t ws_bytes, void* stream) {
  if (cpattn_ring_bwd_workspace(desc) == 0) {  // the descriptor is not valid
    return cpattn_ring_fwd(desc, nullptr, nullptr, nullptr, nullptr, nullptr, stream);
  }
  if (desc->a2a != 1) return CPATTN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !dO || !o || !lse || !dq || !dk || !dv) return CPATTN_ERR_INVALID_ARG;
  if (!workspace || ((uintptr_t)workspace & 255u)) return CPATTN_ERR_INVALID_ARG;
  const StepLayout L = layout_of(desc);
  if (ws_bytes < L.total) return CPATTN_ERR_INVALID_ARG;
  CopyStreams* cs = copy_streams();
  if (!cs) return CPATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(cs->mu);
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();

  const int n = groups_of(desc);
  const cpattn_desc gd = group_desc(desc, n);
  cpattn_desc gd_lse = gd;  // the LSE permuted as rows of one float32
  gd_lse.D = 1;
  gd_lse.dtype = CPATTN_F32;
  char* w = static_cast<char*>(workspace);
  const size_t elt = desc->dtype == CPATTN_BF16 ? 2 : 4;
  const size_t qb = (size_t)desc->B * desc->H_q * desc->T * desc->D * elt / n;   // per group
  const size_t kb = (size_t)desc->B * desc->H_kv * desc->T * desc->D * elt / n;
  const size_t lb = (size_t)desc->B * desc->H_q * desc->T * sizeof(float) / n;
  auto dev_at = [&](size_t section, int j, size_t per) { return w + section + j * per; };
  auto host_at = [&](const void* p, int j, size_t per) {
    return static_cast<const char*>(p) + j * per;
  };
  auto host_out = [&](void* p, int j, size_t per) { return static_cast<char*>(p) + j * per; };
  cudaEvent_t* ev = cs->ev;
  cudaEvent_t ev_start = ev[0], ev_end = ev[1];
  auto ev_in = [&](int j) { return ev[2 + kEventsPerGroup * j]; };
  auto ev_do = [&](int j) { return ev[3 + kEventsPerGroup * j]; };
  auto ev_fwd = [&](int j) { return ev[4 + kEventsPerGroup * j]; };
  auto ev_grad = [&](int j) { return ev[5 + kEventsPerGroup * j]; };
  const int Hq = gd.H_q, Hkv = gd.H_kv;

#define CPATTN_TRY(x)                         \
  do {                                        \
    if ((x) != cudaSuccess) return CPATTN_ERR_CUDA; \
  } while (0)
#define CPATTN_TRY_S(x)                       \
  do {                                        \
    const cpattn_status s_ = (x);             \
    if (s_ != CPATTN_OK) return s_;           \
  } while (0)

  // the copies follow what the caller's stream already holds
  CPATTN_TRY(cudaEventRecord(ev_start, st));
  CPATTN_TRY(cudaStreamWaitEvent(cs->up, ev_start, 0));
  CPATTN_TRY(cudaStreamWaitEvent(cs->down, ev_start, 0));
  // uploads: q, k, v of every group, then dO of every group
  for (int j = 0; j < n; ++j) {
    CPATTN_TRY(cudaMemcpyAsync(dev_at(L.stage_q, j, qb), host_at(q, j, qb), qb,
                               cudaMemcpyHostToDevice, cs->up));
    CPATTN_TRY(cudaMemcpyAsync(dev_at(L.stage_k, j, kb), host_at(k, j, kb), kb,
                               cudaMemcpyHostToDevice, cs->up));
    CPATTN_TRY(cudaMemcpyAsync(dev_at(L.stage_v, j, kb), host_at(v, j, kb), kb,
                               cudaMemcpyHostToDevice, cs->up));
    CPATTN_TRY(cudaEventRecord(ev_in(j), cs->up));
  }
  for (int j = 0; j < n; ++j) {
    CPATTN_TRY(cudaMemcpyAsync(dev_at(L.stage_do, j, qb), host_at(dO, j, qb), qb,
                               cudaMemcpyHostToDevice, cs->up));
    CPATTN_TRY(cudaEventRecord(ev_do(j), cs->up));
  }
  // forward of every group; o and LSE go back to natural order and home
  for (int j = 0; j < n; ++j) {
    CPATTN_TRY(cudaStreamWaitEvent(st, ev_in(j), 0));
    const void* src[3] = {dev_at(L.stage_q, j, qb), dev_at(L.stage_k, j, kb),
                          dev_at(L.stage_v, j, kb)};
    void* dst[3] = {dev_at(L.lay_q, j, qb), dev_at(L.lay_k, j, kb), dev_at(L.lay_v, j, kb)};
    const int heads[3] = {Hq, Hkv, Hkv};
    CPATTN_TRY_S(cpattn_layout_batch(CPATTN_ZIGZAG_FWD, &gd, 3, src, dst, heads, st));
    float* lay_lse = reinterpret_cast<float*>(dev_at(L.lay_lse, j, lb));
    CPATTN_TRY_S(cpattn_ring_fwd(&gd, dst[0], dst[1], dst[2], dev_at(L.lay_o, j, qb), lay_lse,
                                 st));
    // the natural-order o takes q's staging (q was permuted above, on this stream)
    CPATTN_TRY_S(cpattn_layout(CPATTN_ZIGZAG_INV, &gd, dev_at(L.lay_o, j, qb),
                               dev_at(L.stage_q, j, qb), Hq, st));
    CPATTN_TRY_S(cpattn_layout(CPATTN_ZIGZAG_INV, &gd_lse, lay_lse, dev_at(L.nat_lse, j, lb), Hq,
                               st));
    CPATTN_TRY(cudaEventRecord(ev_fwd(j), st));
    CPATTN_TRY(cudaStreamWaitEvent(cs->down, ev_fwd(j), 0));
    CPATTN_TRY(cudaMemcpyAsync(host_out(o, j, qb), dev_at(L.stage_q, j, qb), qb,
                               cudaMemcpyDeviceToHost, cs->down));
    CPATTN_TRY(cudaMemcpyAsync(host_out(lse, j, lb), dev_at(L.nat_lse, j, lb), lb,
                               cudaMemcpyDeviceToHost, cs->down));
  }
  // backward of every group; dq, dk, dv go back to natural order and home
  for (int j = 0; j < n; ++j) {
    CPATTN_TRY(cudaStreamWaitEvent(st, ev_do(j), 0));
    CPATTN_TRY_S(cpattn_layout(CPATTN_ZIGZAG_FWD, &gd, dev_at(L.stage_do, j, qb),
                               dev_at(L.lay_do, j, qb), Hq, st));
    CPATTN_TRY_S(cpattn_ring_bwd(&gd, dev_at(L.lay_q, j, qb), dev_at(L.lay_k, j, kb),
                                 dev_at(L.lay_v, j, kb), dev_at(L.lay_o, j, qb),
                                 reinterpret_cast<float*>(dev_at(L.lay_lse, j, lb)),
                                 dev_at(L.lay_do, j, qb), dev_at(L.lay_dq, j, qb),
                                 dev_at(L.lay_dk, j, kb), dev_at(L.lay_dv, j, kb),
                                 w + L.bwd_ws, L.bwd, st));
    // natural-order dq, dk, dv take the staging of dO, k and v
    const void* src[3] = {dev_at(L.lay_dq, j, qb), dev_at(L.lay_dk, j, kb),
                          dev_at(L.lay_dv, j, kb)};
    void* dst[3] = {dev_at(L.stage_do, j, qb), dev_at(L.stage_k, j, kb),
                    dev_at(L.stage_v, j, kb)};
    const int heads[3] = {Hq, Hkv, Hkv};
    CPATTN_TRY_S(cpattn_layout_batch(CPATTN_ZIGZAG_INV, &gd, 3, src, dst, heads, st));
    CPATTN_TRY(cudaEventRecord(ev_grad(j), st));
    CPATTN_TRY(cudaStreamWaitEvent(cs->down, ev_grad(j), 0));
    CPATTN_TRY(cudaMemcpyAsync(host_out(dq, j, qb), dst[0], qb, cudaMemcpyDeviceToHost,
                               cs->down));
    CPATTN_TRY(cudaMemcpyAsync(host_out(dk, j, kb), dst[1], kb, cudaMemcpyDeviceToHost,
                               cs->down));
    CPATTN_TRY(cudaMemcpyAsync(host_out(dv, j, kb), dst[2], kb, cudaMemcpyDeviceToHost,
                               cs->down));
  }
  // the caller's stream completes with the last download
  CPATTN_TRY(cudaEventRecord(ev_end, cs->down));
  CPATTN_TRY(cudaStreamWaitEvent(st, ev_end, 0));
#undef CPATTN_TRY
#undef CPATTN_TRY_S
  return CPATTN_OK;
}
