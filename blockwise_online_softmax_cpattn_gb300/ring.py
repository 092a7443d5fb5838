"""The ring across context-parallel ranks: one process (one GPU) per rank, K/V
chunks exchanged point to point.

Tutorial "上下文并行", section "朴素 Ring Attention": every rank sends the K/V
chunk it holds to the next rank and receives one from the previous rank while it
computes the partial result of the chunk it holds, so at step i rank r holds the
chunk of rank (r - i) mod cp; after cp steps every rank has met every chunk, and
the partial results are merged by the online softmax.  Pull request "Feat:
Context Parallel" #181, mode table row "p2p": the backward recomputes each
step's probabilities, and each chunk's K/V gradient travels the ring with the
chunk and arrives back at its owner; the exchange overlaps the step's compute
(the pull request's "overlap" bullet: communication and computation on separate
streams).

This module holds the schedule and the exchange only.  Every step's arithmetic
runs in libcpattn (cpattn_partial_fwd, cpattn_merge, cpattn_partial_bwd) through
``LibrarySteps``; the exchange is torch.distributed point-to-point
(``DistExchange``: NCCL between GPUs, whose transfers run on the communicator's
stream while the library's kernels run on the compute stream).  The kernels only
ever read this GPU's own memory: a received chunk lands in a buffer of the
receiving rank before any kernel touches it.

Per rank and step:
  forward   post the exchange of the held K/V (send to next, receive from
            previous; not after the last step), compute the step's partial and
            merge it into the running (O, LSE), wait for the exchange.
  backward  post the K/V exchange as above, add the step's contributions into
            the rank's dQ and into the held chunk's dK/dV accumulators, then pass
            those accumulators on (after the last step that pass brings every
            chunk's accumulators home to its owner).  dK/dV travel in float32.
The dK/dV pass waits for the step's compute, so it is not hidden behind it; the
K/V transfer for the next step is.

``emulate_ring_forward`` / ``emulate_ring_backward`` run all cp ranks in one
process in lockstep and hand the chunks over by reference: the same per-rank
steps on one GPU.
"""
from __future__ import annotations

from typing import List, Sequence


def ring_source(rank: int, step: int, cp: int) -> int:
    """The rank whose K/V chunk `rank` holds at `step` (send to next, receive from
    previous)."""
    return (rank - step) % cp


def next_rank(rank: int, cp: int) -> int:
    return (rank + 1) % cp


def prev_rank(rank: int, cp: int) -> int:
    return (rank - 1) % cp


# ---------------------------------------------------------------------------
# per-rank state
# ---------------------------------------------------------------------------
class _FwdRank:
    """One rank's forward: its query chunk, the K/V chunk it holds, the merged
    (O, LSE) so far, and which chunk it held at every step."""

    def __init__(self, steps, rank: int, cp: int, q, k, v):
        self.steps, self.rank, self.cp, self.q = steps, rank, cp, q
        self.kv = [k, v]
        self.o = self.lse = None
        self.held: List[int] = []

    def step(self, i: int) -> None:
        s = ring_source(self.rank, i, self.cp)
        self.held.append(s)
        o, lse = self.steps.partial_fwd(self.rank, s, self.q, *self.kv)
        if self.o is None:
            self.o, self.lse = o, lse
        else:
            self.steps.merge_into(self.o, self.lse, o, lse)


class _BwdRank:
    """One rank's backward: its rows (q, o, lse, dO), its dQ so far, the K/V chunk
    it holds and that chunk's travelling dK/dV accumulators."""

    def __init__(self, steps, rank: int, cp: int, q, k, v, o, lse, do):
        self.steps, self.rank, self.cp = steps, rank, cp
        self.rows = (q, do)
        # the rank's row statistics, once for all of its steps
        steps.bwd_stats(rank, o, lse, do)
        self.kv = [k, v]
        self.dq = steps.new_q_grad()
        self.dkv = list(steps.new_kv_grads())
        self.held: List[int] = []

    def step(self, i: int) -> None:
        s = ring_source(self.rank, i, self.cp)
        self.held.append(s)
        q, do = self.rows
        # step 0: the rank's own chunk, whose accumulators start here; later steps
        # add to what the previous ranks left in them
        self.steps.partial_bwd(self.rank, s, q, self.kv[0], self.kv[1], do, self.dq,
                               self.dkv[0], self.dkv[1], accumulate=i > 0)


# ---------------------------------------------------------------------------
# one process per rank
# ---------------------------------------------------------------------------
class DistExchange:
    """Point-to-point exchange around the ring over torch.distributed: send to the
    next rank, receive from the previous one, as one group of operations (so no
    rank's send waits behind its own receive)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def _global(self, r: int) -> int:
        return r if self.group is None else self.dist.get_global_rank(self.group, r)

    def start(self, send: Sequence, recv: Sequence):
        nxt = self._global(next_rank(self.rank, self.world))
        prv = self._global(prev_rank(self.rank, self.world))
        ops = []
        for t in send:
            ops.append(self.dist.P2POp(self.dist.isend, t, nxt, self.group))
        for t in recv:
            ops.append(self.dist.P2POp(self.dist.irecv, t, prv, self.group))
        return self.dist.batch_isend_irecv(ops), list(recv)

    @staticmethod
    def wait(handle):
        reqs, recv = handle
        for r in reqs:
            r.wait()
        return recv


class HostExchange(DistExchange):
    """The same exchange staged through host memory, for process groups whose backend
    moves host tensors only (gloo): each outgoing device tensor is copied to the
    host (which waits for the work that produced it), sent, and received into host
    buffers that are copied to the device on wait.  No transfer overlaps compute."""

    def start(self, send: Sequence, recv: Sequence):
        host_send = [t.detach().to("cpu") for t in send]
        host_recv = [t.new_empty(t.shape, device="cpu") for t in recv]
        reqs, _ = super().start(host_send, host_recv)
        return reqs, (host_send, host_recv, list(recv))

    @staticmethod
    def wait(handle):
        reqs, (_, host_recv, recv) = handle
        for r in reqs:
            r.wait()
        for dst, src in zip(recv, host_recv):
            dst.copy_(src)
        return recv


def ring_forward(steps, exch, q, k, v):
    """Rank exch.rank's forward over a ring of exch.world ranks.  q, k, v are the
    rank's own chunks ([B, H, c, D], layout order); returns its (O, LSE) rows and
    the chunks it held, step by step."""
    cp = exch.world
    st = _FwdRank(steps, exch.rank, cp, q, k, v)
    for i in range(cp):
        h = exch.start(st.kv, [t.new_empty(t.shape) for t in st.kv]) if i + 1 < cp else None
        st.step(i)
        if h is not None:
            st.kv = exch.wait(h)
    o, lse = steps.finish_fwd(st.o, st.lse)
    return o, lse, st.held


def ring_backward(steps, exch, q, k, v, o, lse, do):
    """Rank exch.rank's backward: its rows (q, o, lse, dO) and its own K/V chunk;
    returns dQ of its rows and dK, dV of its own chunk (brought home by the last
    pass), plus the chunks it held, step by step."""
    cp = exch.world
    st = _BwdRank(steps, exch.rank, cp, q, k, v, o, lse, do)
    for i in range(cp):
        h = exch.start(st.kv, [t.new_empty(t.shape) for t in st.kv]) if i + 1 < cp else None
        st.step(i)
        if cp > 1:
            st.dkv = exch.wait(exch.start(st.dkv, [t.new_empty(t.shape) for t in st.dkv]))
        if h is not None:
            st.kv = exch.wait(h)
    dq, dk, dv = steps.finish_bwd(st.dq, *st.dkv)
    return dq, dk, dv, st.held


# ---------------------------------------------------------------------------
# all ranks in one process
# ---------------------------------------------------------------------------
def emulate_ring_forward(steps, cp: int, qs, ks, vs):
    """All cp ranks in lockstep in one process; the per-rank steps of
    ring_forward, with the K/V handed to the next rank by reference."""
    ranks = [_FwdRank(steps, r, cp, qs[r], ks[r], vs[r]) for r in range(cp)]
    for i in range(cp):
        for st in ranks:
            st.step(i)
        if i + 1 < cp:
            held = [st.kv for st in ranks]
            for r, st in enumerate(ranks):
                st.kv = held[prev_rank(r, cp)]
    out = [steps.finish_fwd(st.o, st.lse) for st in ranks]
    return [o for o, _ in out], [lse for _, lse in out], [st.held for st in ranks]


def emulate_ring_backward(steps, cp: int, qs, ks, vs, os_, lses, dos):
    """All cp ranks in lockstep in one process; the per-rank steps of
    ring_backward."""
    ranks = [_BwdRank(steps, r, cp, qs[r], ks[r], vs[r], os_[r], lses[r], dos[r])
             for r in range(cp)]
    for i in range(cp):
        for st in ranks:
            st.step(i)
        held_kv = [st.kv for st in ranks]
        held_g = [st.dkv for st in ranks]
        for r, st in enumerate(ranks):
            st.dkv = held_g[prev_rank(r, cp)]
            if i + 1 < cp:
                st.kv = held_kv[prev_rank(r, cp)]
    out = [steps.finish_bwd(st.dq, *st.dkv) for st in ranks]
    return ([x[0] for x in out], [x[1] for x in out], [x[2] for x in out],
            [st.held for st in ranks])


# ---------------------------------------------------------------------------
# the library's steps
# ---------------------------------------------------------------------------
class LibrarySteps:
    """Every step's arithmetic in libcpattn on this process's GPU.

    The library's ring-step calls take full layout-order tensors, so the rank's
    query chunk and the K/V chunk held at a step are placed at their slots in
    full-length buffers of this GPU (device copies) before each call; a call
    reads only those slots.  desc: a cpattn_desc of the whole problem (a2a = 1).
    Partial outputs, dQ and the travelling dK/dV are float32; finish_* rounds
    them to the tensor dtype (the same once-after-the-sum rounding the fused
    kernels apply)."""

    def __init__(self, desc, device=None, stream=None):
        import torch

        from . import cpattn_partial_bwd_workspace
        if desc.a2a != 1:
            raise ValueError("the point-to-point ring runs the plain ring (a2a = 1)")
        self.torch = torch
        self.desc = desc
        self.stream = stream
        self.dtype = torch.bfloat16 if desc.dtype == 1 else torch.float32
        self.device = torch.device("cuda") if device is None else torch.device(device)
        B, Hq, Hkv, T, D = desc.B, desc.H_q, desc.H_kv, desc.T, desc.D
        self.c = T // desc.cp
        self.q_shape = (B, Hq, self.c, D)
        self.kv_shape = (B, Hkv, self.c, D)
        kw = dict(dtype=self.dtype, device=self.device)
        self.q_full = torch.zeros(B, Hq, T, D, **kw)
        self.k_full = torch.zeros(B, Hkv, T, D, **kw)
        self.v_full = torch.zeros(B, Hkv, T, D, **kw)
        self.ws_bytes = cpattn_partial_bwd_workspace(desc)
        self.stats = {}  # rank -> its row statistics (one workspace per rank)

    def _place(self, r: int, s: int, q, k, v) -> None:
        c = self.c
        self.q_full[:, :, r * c:(r + 1) * c].copy_(q)
        self.k_full[:, :, s * c:(s + 1) * c].copy_(k)
        self.v_full[:, :, s * c:(s + 1) * c].copy_(v)

    def partial_fwd(self, r: int, s: int, q, k, v):
        from . import check, cpattn_partial_fwd
        self._place(r, s, q, k, v)
        t = self.torch
        o = t.empty(self.q_shape, dtype=t.float32, device=self.device)
        lse = t.empty(self.q_shape[:3], dtype=t.float32, device=self.device)
        check(cpattn_partial_fwd(self.desc, r, s, self.q_full, self.k_full, self.v_full, o, lse,
                                 self.stream))
        return o, lse

    def merge_into(self, o, lse, o2, lse2) -> None:
        from . import check, cpattn_merge
        rows = o.numel() // o.shape[-1]
        check(cpattn_merge(rows, o.shape[-1], o, lse, o2, lse2, o, lse, self.stream))

    def new_q_grad(self):
        return self.torch.empty(self.q_shape, dtype=self.torch.float32, device=self.device)

    def new_kv_grads(self):
        t = self.torch
        return (t.empty(self.kv_shape, dtype=t.float32, device=self.device),
                t.empty(self.kv_shape, dtype=t.float32, device=self.device))

    def bwd_stats(self, r: int, o, lse, do) -> None:
        from . import check, cpattn_partial_bwd_stats
        if r not in self.stats:
            self.stats[r] = self.torch.empty(self.ws_bytes, dtype=self.torch.uint8,
                                             device=self.device)
        check(cpattn_partial_bwd_stats(self.desc, o, lse, do, self.stats[r], None, self.stream))

    def partial_bwd(self, r, s, q, k, v, do, dq, dk, dv, accumulate) -> None:
        from . import check, cpattn_partial_bwd
        self._place(r, s, q, k, v)
        check(cpattn_partial_bwd(self.desc, r, s, self.q_full, self.k_full, self.v_full, do, dq,
                                 dk, dv, 1 if accumulate else 0, self.stats[r], None,
                                 self.stream))

    def finish_fwd(self, o, lse):
        return o.to(self.dtype), lse

    def finish_bwd(self, dq, dk, dv):
        return dq.to(self.dtype), dk.to(self.dtype), dv.to(self.dtype)


def rank_chunks(x, cp: int) -> list:
    """A layout-order tensor [B, H, T, D] cut into the cp ranks' chunks
    [B, H, T/cp, D] (contiguous copies)."""
    c = x.shape[2] // cp
    return [x[:, :, r * c:(r + 1) * c].contiguous() for r in range(cp)]


__all__ = ["ring_source", "next_rank", "prev_rank", "DistExchange", "HostExchange", "ring_forward",
           "ring_backward", "emulate_ring_forward", "emulate_ring_backward", "LibrarySteps",
           "rank_chunks"]
