// cpattn_ring_step_host: one forward + backward step of the ring over tensors that
// live in host memory, with the host<->device transfers overlapping the compute.
//
// The problem splits into independent groups: batch rows, or K/V heads with their
// query heads.  Group j of n of every tensor is its j-th contiguous n-th, so each
// group is a smaller problem of the same kind.  The backward runs in nb groups (two
// when the problem splits so), the forward in nf = 2 nb groups when it splits that
// far (the forward's kernels lose little on a quarter of the problem, the
// backward's dK/dV kernel would), so backward group j covers forward groups 2j and
// 2j + 1.  Two copy streams per device, created once, carry the transfers:
//
//   upload stream    q, k, v of forward group 2j, of 2j + 1, then dO of backward
//                    group j; then the same for j + 1
//   caller's stream  per backward group j: for its forward groups, permute q, k, v
//                    to layout order, ring forward, permute o and LSE back; then
//                    permute dO, ring backward (its dQ kernel overlapping the end of
//                    its dK/dV kernel), permute dk, dv and dq back; in the last group
//                    dk and dv are permuted back between the two kernels instead
//   download stream  (once every upload is done: the two directions share the host
//                    link, and only the first uploads are on the compute's path)
//                    o and LSE of a forward group as soon as it is done; dk and dv
//                    of a backward group once permuted (the last group's while its
//                    dQ kernel runs); dq once its backward is done (the last group's
//                    in two parts, the first while the second part's dQ kernel runs)
//
// so the first kernel waits only for the first forward group's inputs, uploads
// run while earlier groups compute, downloads while later ones do, and only the
// last group's dq is left to download after the last kernel.  The caller's stream
// waits for the last download, so the call's work is complete when that stream's
// work is.
#include <mutex>

#include "../../include/cpattn.h"
#include "api_internal.h"
#include "kernels.h"

namespace cpattn {
namespace {

constexpr int kMaxBwdGroups = 2, kMaxFwdGroups = 2 * kMaxBwdGroups;
// events per device: start, end; per forward group: inputs landed, outputs ready;
// per backward group: dO landed, dk and dv ready, dq ready
// plus the two parts of the last backward group's dq
constexpr int kDqParts = 2;
constexpr int kNumEvents = 2 + 2 * kMaxFwdGroups + 3 * kMaxBwdGroups + kDqParts;

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

// Whether the j-th contiguous n-th of every tensor is an independent problem of the
// same kind (n divides B, or each batch row splits into n / B groups of K/V heads)
// whose slices of q, k and the LSE start on 16-byte boundaries.
bool splits(const cpattn_desc* d, int n) {
  if (n == 1) return true;
  if (!(d->B % n == 0 || (n % d->B == 0 && d->H_kv % (n / d->B) == 0))) return false;
  const size_t elt = d->dtype == CPATTN_BF16 ? 2 : 4;
  const size_t q = (size_t)d->B * d->H_q * d->T * d->D * elt / n;
  const size_t k = (size_t)d->B * d->H_kv * d->T * d->D * elt / n;
  const size_t l = (size_t)d->B * d->H_q * d->T * sizeof(float) / n;
  return q % 16 == 0 && k % 16 == 0 && l % 16 == 0;
}

int bwd_groups(const cpattn_desc* d) { return splits(d, 2) ? 2 : 1; }
int fwd_groups(const cpattn_desc* d) {
  const int nb = bwd_groups(d);
  return splits(d, 2 * nb) ? 2 * nb : nb;
}

cpattn_desc group_desc(const cpattn_desc* d, int n) {
  cpattn_desc g = *d;
  if (n > 1) {
    if (d->B % n == 0) {
      g.B = d->B / n;
    } else {
      const int m = n / d->B;  // groups per batch row
      g.B = 1;
      g.H_q = d->H_q / m;
      g.H_kv = d->H_kv / m;
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
  const cpattn_desc g = group_desc(d, bwd_groups(d));
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

// Queued by the backward between its dK/dV and dQ kernels: dk and dv back to
// natural order, then the event the download stream waits for.
struct DkdvOut {
  const cpattn_desc* gd;
  const void* src[2];
  void* dst[2];
  int heads[2];
  cudaEvent_t done;
};

cudaError_t dkdv_out(void* ctx, cudaStream_t st) {
  DkdvOut* d = static_cast<DkdvOut*>(ctx);
  if (cpattn_layout_batch(CPATTN_ZIGZAG_INV, d->gd, 2, d->src, d->dst, d->heads, st) != CPATTN_OK)
    return cudaErrorLaunchFailure;
  return cudaEventRecord(d->done, st);
}

// Queued by the backward after each part of its dQ kernel: that part's dq back to
// natural order, then the event the download stream waits for.
struct DqOut {
  cpattn_desc gp;  // one part
  const char* src;
  char* dst;
  size_t bytes;  // of one part
  cudaEvent_t done[kDqParts];
};

cudaError_t dq_out(void* ctx, cudaStream_t st, int part) {
  DqOut* d = static_cast<DqOut*>(ctx);
  if (cpattn_layout(CPATTN_ZIGZAG_INV, &d->gp, d->src + part * d->bytes, d->dst + part * d->bytes,
                    d->gp.H_q, st) != CPATTN_OK)
    return cudaErrorLaunchFailure;
  return cudaEventRecord(d->done[part], st);
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

  const int nb = bwd_groups(desc), nf = fwd_groups(desc), r = nf / nb;
  const cpattn_desc gb = group_desc(desc, nb), gf = group_desc(desc, nf);
  cpattn_desc gf_lse = gf;  // the LSE permuted as rows of one float32
  gf_lse.D = 1;
  gf_lse.dtype = CPATTN_F32;
  char* w = static_cast<char*>(workspace);
  const size_t elt = desc->dtype == CPATTN_BF16 ? 2 : 4;
  const size_t q_all = (size_t)desc->B * desc->H_q * desc->T * desc->D * elt;
  const size_t k_all = (size_t)desc->B * desc->H_kv * desc->T * desc->D * elt;
  const size_t l_all = (size_t)desc->B * desc->H_q * desc->T * sizeof(float);
  // bytes of one group's slice: backward groups (b) and forward groups (f)
  const size_t qb = q_all / nb, kb = k_all / nb, lb = l_all / nb;
  const size_t qf = q_all / nf, kf = k_all / nf, lf = l_all / nf;
  auto dev_at = [&](size_t section, int j, size_t per) { return w + section + j * per; };
  auto host_at = [&](const void* p, int j, size_t per) {
    return static_cast<const char*>(p) + j * per;
  };
  auto host_out = [&](void* p, int j, size_t per) { return static_cast<char*>(p) + j * per; };
  cudaEvent_t* ev = cs->ev;
  cudaEvent_t ev_start = ev[0], ev_end = ev[1];
  auto ev_in = [&](int f) { return ev[2 + f]; };                  // forward group f
  auto ev_fwd = [&](int f) { return ev[2 + kMaxFwdGroups + f]; };
  auto ev_do = [&](int j) { return ev[2 + 2 * kMaxFwdGroups + j]; };  // backward group j
  auto ev_dkdv = [&](int j) { return ev[2 + 2 * kMaxFwdGroups + kMaxBwdGroups + j]; };
  auto ev_grad = [&](int j) { return ev[2 + 2 * kMaxFwdGroups + 2 * kMaxBwdGroups + j]; };
  auto ev_dq = [&](int part) { return ev[2 + 2 * kMaxFwdGroups + 3 * kMaxBwdGroups + part]; };

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
  // uploads in the order the groups use them
  for (int j = 0; j < nb; ++j) {
    for (int f = j * r; f < (j + 1) * r; ++f) {
      CPATTN_TRY(cudaMemcpyAsync(dev_at(L.stage_q, f, qf), host_at(q, f, qf), qf,
                                 cudaMemcpyHostToDevice, cs->up));
      CPATTN_TRY(cudaMemcpyAsync(dev_at(L.stage_k, f, kf), host_at(k, f, kf), kf,
                                 cudaMemcpyHostToDevice, cs->up));
      CPATTN_TRY(cudaMemcpyAsync(dev_at(L.stage_v, f, kf), host_at(v, f, kf), kf,
                                 cudaMemcpyHostToDevice, cs->up));
      CPATTN_TRY(cudaEventRecord(ev_in(f), cs->up));
    }
    CPATTN_TRY(cudaMemcpyAsync(dev_at(L.stage_do, j, qb), host_at(dO, j, qb), qb,
                               cudaMemcpyHostToDevice, cs->up));
    CPATTN_TRY(cudaEventRecord(ev_do(j), cs->up));
  }
  // downloads start once every upload is done: the two directions share the host
  // link, and the first uploads are on the compute's critical path
  CPATTN_TRY(cudaStreamWaitEvent(cs->down, ev_do(nb - 1), 0));
  for (int j = 0; j < nb; ++j) {
    // forward of the group's forward groups; o and LSE go back to natural order and home
    for (int f = j * r; f < (j + 1) * r; ++f) {
      CPATTN_TRY(cudaStreamWaitEvent(st, ev_in(f), 0));
      const void* src[3] = {dev_at(L.stage_q, f, qf), dev_at(L.stage_k, f, kf),
                            dev_at(L.stage_v, f, kf)};
      void* dst[3] = {dev_at(L.lay_q, f, qf), dev_at(L.lay_k, f, kf), dev_at(L.lay_v, f, kf)};
      const int heads[3] = {gf.H_q, gf.H_kv, gf.H_kv};
      CPATTN_TRY_S(cpattn_layout_batch(CPATTN_ZIGZAG_FWD, &gf, 3, src, dst, heads, st));
      float* lay_lse = reinterpret_cast<float*>(dev_at(L.lay_lse, f, lf));
      CPATTN_TRY_S(cpattn_ring_fwd(&gf, dst[0], dst[1], dst[2], dev_at(L.lay_o, f, qf), lay_lse,
                                   st));
      // the natural-order o takes q's staging (q was permuted above, on this stream)
      CPATTN_TRY_S(cpattn_layout(CPATTN_ZIGZAG_INV, &gf, dev_at(L.lay_o, f, qf),
                                 dev_at(L.stage_q, f, qf), gf.H_q, st));
      CPATTN_TRY_S(cpattn_layout(CPATTN_ZIGZAG_INV, &gf_lse, lay_lse, dev_at(L.nat_lse, f, lf),
                                 gf.H_q, st));
      CPATTN_TRY(cudaEventRecord(ev_fwd(f), st));
      CPATTN_TRY(cudaStreamWaitEvent(cs->down, ev_fwd(f), 0));
      CPATTN_TRY(cudaMemcpyAsync(host_out(o, f, qf), dev_at(L.stage_q, f, qf), qf,
                                 cudaMemcpyDeviceToHost, cs->down));
      CPATTN_TRY(cudaMemcpyAsync(host_out(lse, f, lf), dev_at(L.nat_lse, f, lf), lf,
                                 cudaMemcpyDeviceToHost, cs->down));
    }
    // backward (its layout-order q, k, v, o, LSE are those of its forward groups, end
    // to end); natural-order dk and dv take the staging of k and v (read by the
    // forward's permutes above), dq that of dO
    CPATTN_TRY(cudaStreamWaitEvent(st, ev_do(j), 0));
    CPATTN_TRY_S(cpattn_layout(CPATTN_ZIGZAG_FWD, &gb, dev_at(L.stage_do, j, qb),
                               dev_at(L.lay_do, j, qb), gb.H_q, st));
    DkdvOut out;
    out.gd = &gb;
    out.src[0] = dev_at(L.lay_dk, j, kb);
    out.src[1] = dev_at(L.lay_dv, j, kb);
    out.dst[0] = dev_at(L.stage_k, j, kb);
    out.dst[1] = dev_at(L.stage_v, j, kb);
    out.heads[0] = out.heads[1] = gb.H_kv;
    out.done = ev_dkdv(j);
    const AfterDkdv after{dkdv_out, &out};
    // the last group's dq is the one download left after the last kernel: its dQ
    // kernel runs in two parts, and the first part goes home while the second computes
    const bool parts = j == nb - 1 && splits(&gb, kDqParts);
    DqOut dqo;
    dqo.gp = group_desc(&gb, kDqParts);
    dqo.src = dev_at(L.lay_dq, j, qb);
    dqo.dst = dev_at(L.stage_do, j, qb);
    dqo.bytes = qb / kDqParts;
    for (int part = 0; part < kDqParts; ++part) dqo.done[part] = ev_dq(part);
    const AfterDqPart after_dq{dq_out, &dqo, kDqParts};
    // Before the last group, nothing waits for dk and dv: the group's dQ kernel may then
    // overlap the end of its dK/dV kernel (nothing queued between them), and dk, dv go
    // back to natural order after both.  The last group's dk and dv go home while its
    // dQ kernel runs.
    const bool last = j == nb - 1;
    CPATTN_TRY_S(ring_bwd_after_dkdv(&gb, dev_at(L.lay_q, j, qb), dev_at(L.lay_k, j, kb),
                                     dev_at(L.lay_v, j, kb), dev_at(L.lay_o, j, qb),
                                     reinterpret_cast<float*>(dev_at(L.lay_lse, j, lb)),
                                     dev_at(L.lay_do, j, qb), dev_at(L.lay_dq, j, qb),
                                     dev_at(L.lay_dk, j, kb), dev_at(L.lay_dv, j, kb),
                                     w + L.bwd_ws, L.bwd, st, last ? &after : nullptr,
                                     parts ? &after_dq : nullptr));
    if (!last) CPATTN_TRY(dkdv_out(&out, st));
    CPATTN_TRY(cudaStreamWaitEvent(cs->down, ev_dkdv(j), 0));
    CPATTN_TRY(cudaMemcpyAsync(host_out(dk, j, kb), out.dst[0], kb, cudaMemcpyDeviceToHost,
                               cs->down));
    CPATTN_TRY(cudaMemcpyAsync(host_out(dv, j, kb), out.dst[1], kb, cudaMemcpyDeviceToHost,
                               cs->down));
    if (parts) {
      for (int part = 0; part < kDqParts; ++part) {
        CPATTN_TRY(cudaStreamWaitEvent(cs->down, ev_dq(part), 0));
        CPATTN_TRY(cudaMemcpyAsync(host_out(dq, j, qb) + part * dqo.bytes,
                                   dqo.dst + part * dqo.bytes, dqo.bytes, cudaMemcpyDeviceToHost,
                                   cs->down));
      }
    } else {
      CPATTN_TRY_S(cpattn_layout(CPATTN_ZIGZAG_INV, &gb, dev_at(L.lay_dq, j, qb),
                                 dev_at(L.stage_do, j, qb), gb.H_q, st));
      CPATTN_TRY(cudaEventRecord(ev_grad(j), st));
      CPATTN_TRY(cudaStreamWaitEvent(cs->down, ev_grad(j), 0));
      CPATTN_TRY(cudaMemcpyAsync(host_out(dq, j, qb), dev_at(L.stage_do, j, qb), qb,
                                 cudaMemcpyDeviceToHost, cs->down));
    }
  }
  // the caller's stream completes with the last download
  CPATTN_TRY(cudaEventRecord(ev_end, cs->down));
  CPATTN_TRY(cudaStreamWaitEvent(st, ev_end, 0));
#undef CPATTN_TRY
#undef CPATTN_TRY_S
  return CPATTN_OK;
}
