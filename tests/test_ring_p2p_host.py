"""Host (CPU, gloo): the point-to-point ring across ranks, one process per rank.

The schedule and the exchange of blockwise_online_softmax_cpattn_gb300.ring run
over torch.distributed with the gloo backend, world size 2, 3 and 4.  Each step's
arithmetic is supplied by the test from the FP64 oracle (the product supplies it
from libcpattn; here it is the checker), and every step checks that the K/V it is
handed are exactly the chunk the ring should deliver: at step i rank r holds the
chunk of rank (r - i) mod cp.  The merged forward rows and the backward's dQ rows
and home-coming dK/dV chunks are compared with the oracle's full attention.  The
same steps also run in the one-process lockstep emulation."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT, rel_err
from oracle import attention as OA
from oracle import layouts as OL


def _load_ring():
    """The ring module by path: it is pure Python, and importing it through the
    package would load the CUDA library, which these host tests do not need."""
    import importlib.util
    path = os.path.join(ROOT, "blockwise_online_softmax_cpattn_gb300", "ring.py")
    spec = importlib.util.spec_from_file_location("cpattn_ring_schedule", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


R = _load_ring()


def _problem(cp, layout, T=48, B=1, Hq=4, Hkv=2, D=6, seed=0):
    rng = np.random.default_rng(seed + 10 * cp)
    q, k, v, do = (rng.standard_normal((B, h, T, D)) for h in (Hq, Hkv, Hkv, Hq))
    pos = OL.positions(T, cp, layout)
    lay = [x[:, :, pos] for x in (q, k, v, do)]   # layout order
    return (q, k, v, do), lay, pos


class OracleSteps:
    """The ring steps computed by the FP64 oracle on CPU tensors (float64), with
    a check that every step is handed the right chunks."""

    def __init__(self, lay, pos, cp, scale):
        self.q, self.k, self.v, self.do = lay
        self.pos, self.cp, self.scale = pos, cp, scale
        self.c = self.q.shape[2] // cp
        self.n_rep = self.q.shape[1] // self.k.shape[1]

    def _sl(self, r):
        return slice(r * self.c, (r + 1) * self.c)

    def _check(self, r, s, q, k, v):
        assert np.array_equal(q.numpy(), self.q[:, :, self._sl(r)]), ("query chunk", r)
        assert np.array_equal(k.numpy(), self.k[:, :, self._sl(s)]), ("K chunk", r, s)
        assert np.array_equal(v.numpy(), self.v[:, :, self._sl(s)]), ("V chunk", r, s)

    def partial_fwd(self, r, s, q, k, v):
        self._check(r, s, q, k, v)
        qp, kp = self.pos[self._sl(r)], self.pos[self._sl(s)]
        B, H, c, D = q.shape
        o, lse = np.zeros((B, H, c, D)), np.zeros((B, H, c))
        for b in range(B):
            for h in range(H):
                g = h // self.n_rep
                o[b, h], lse[b, h] = OA.partial_attention(q[b, h].numpy(), k[b, g].numpy(),
                                                          v[b, g].numpy(), qp, kp, self.scale)
        return torch.from_numpy(o), torch.from_numpy(lse)

    def merge_into(self, o, lse, o2, lse2):
        mo, ml = OA.merge(o.numpy(), lse.numpy(), o2.numpy(), lse2.numpy())
        o.copy_(torch.from_numpy(mo))
        lse.copy_(torch.from_numpy(ml))

    def new_q_grad(self):
        return torch.full(self.q[:, :, :self.c].shape, float("nan"), dtype=torch.float64)

    def new_kv_grads(self):
        shape = self.k[:, :, :self.c].shape
        return (torch.full(shape, float("nan"), dtype=torch.float64),
                torch.full(shape, float("nan"), dtype=torch.float64))

    def bwd_stats(self, r, o, lse, do):
        self.rank_stats = getattr(self, "rank_stats", {})
        self.rank_stats[r] = (o.clone(), lse.clone())

    def partial_bwd(self, r, s, q, k, v, do, dq, dk, dv, accumulate):
        self._check(r, s, q, k, v)
        o, lse = self.rank_stats[r]
        qp, kp = self.pos[self._sl(r)], self.pos[self._sl(s)]
        B, H = q.shape[:2]
        gq, gk, gv = np.zeros(dq.shape), np.zeros(dk.shape), np.zeros(dv.shape)
        for b in range(B):
            for h in range(H):
                g = h // self.n_rep
                a, bb, e = OA.partial_attention_bwd(q[b, h].numpy(), k[b, g].numpy(),
                                                    v[b, g].numpy(), do[b, h].numpy(),
                                                    o[b, h].numpy(), lse[b, h].numpy(), qp, kp,
                                                    self.scale)
                gq[b, h] += a
                gk[b, g] += bb
                gv[b, g] += e
        for t, x in ((dq, gq), (dk, gk), (dv, gv)):
            if accumulate:
                t.add_(torch.from_numpy(x))
            else:
                t.copy_(torch.from_numpy(x))

    def finish_fwd(self, o, lse):
        return o, lse

    def finish_bwd(self, dq, dk, dv):
        return dq, dk, dv


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, layout, out, exchange="dist"):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        nat, lay, pos = _problem(world, layout)
        scale = 0.4
        steps = OracleSteps(lay, pos, world, scale)
        c = lay[0].shape[2] // world
        mine = [torch.from_numpy(np.ascontiguousarray(x[:, :, rank * c:(rank + 1) * c]))
                for x in lay]
        exch = R.DistExchange() if exchange == "dist" else R.HostExchange()
        o, lse, held_f = R.ring_forward(steps, exch, mine[0], mine[1], mine[2])
        dq, dk, dv, held_b = R.ring_backward(steps, exch, mine[0], mine[1], mine[2], o, lse,
                                             mine[3])
        out.put((rank, o.numpy(), lse.numpy(), dq.numpy(), dk.numpy(), dv.numpy(), held_f,
                 held_b))
    finally:
        dist.destroy_process_group()


def _reference(nat, scale):
    q, k, v, do = nat
    o, lse = OA.attention_fwd(q, k, v, scale)
    dq, dk, dv = OA.attention_bwd(q, k, v, do, scale)
    return o, lse, dq, dk, dv


def _check_rank(world, layout, res, nat, pos):
    o, lse, dq, dk, dv = _reference(nat, 0.4)
    r, go, gl, gdq, gdk, gdv, held_f, held_b = res
    want = [OL.ring_source(r, i, world) for i in range(world)]
    assert held_f == want and held_b == want, (r, held_f, held_b)
    c = o.shape[2] // world
    p = pos[r * c:(r + 1) * c]   # natural positions of rank r's slots (and of chunk r)
    assert rel_err(go, o[:, :, p]) < 1e-12 and np.max(np.abs(gl - lse[:, :, p])) < 1e-12
    assert rel_err(gdq, dq[:, :, p]) < 1e-12, ("dq", r)
    assert rel_err(gdk, dk[:, :, p]) < 1e-12, ("dk home", r)
    assert rel_err(gdv, dv[:, :, p]) < 1e-12, ("dv home", r)


@pytest.mark.parametrize("world,layout,exchange", [(2, "zigzag", "dist"), (3, "contiguous", "dist"),
                                                   (4, "zigzag", "dist"), (3, "zigzag", "host")])
def test_ring_over_gloo_ranks(world, layout, exchange):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, layout, out, exchange))
             for r in range(world)]
    for p in procs:
        p.start()
    results = [out.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    nat, _, pos = _problem(world, layout)
    for res in sorted(results, key=lambda x: x[0]):
        _check_rank(world, layout, res, nat, pos)


@pytest.mark.parametrize("cp,layout", [(1, "contiguous"), (3, "zigzag"), (4, "contiguous")])
def test_ring_emulated_in_one_process(cp, layout):
    nat, lay, pos = _problem(cp, layout)
    steps = OracleSteps(lay, pos, cp, 0.4)
    chunks = [[torch.from_numpy(np.ascontiguousarray(x[:, :, r * (x.shape[2] // cp):
                                                       (r + 1) * (x.shape[2] // cp)]))
               for r in range(cp)] for x in lay]
    os_, lses, held_f = R.emulate_ring_forward(steps, cp, *chunks[:3])
    dqs, dks, dvs, held_b = R.emulate_ring_backward(steps, cp, *chunks[:3], os_, lses, chunks[3])
    for r in range(cp):
        res = (r, os_[r].numpy(), lses[r].numpy(), dqs[r].numpy(), dks[r].numpy(),
               dvs[r].numpy(), held_f[r], held_b[r])
        _check_rank(cp, layout, res, nat, pos)


def test_schedule_tables():
    """Send to next, receive from previous: the chunk held at step i is the one
    (r - i) mod cp, every chunk is met once, and cp steps bring a chunk's
    gradient back home."""
    for cp in (1, 2, 5, 8):
        for r in range(cp):
            held = [R.ring_source(r, i, cp) for i in range(cp)]
            assert sorted(held) == list(range(cp)) and held[0] == r
            for i in range(1, cp):
                # what r holds at step i is what its predecessor held at step i - 1
                assert held[i] == R.ring_source(R.prev_rank(r, cp), i - 1, cp)
            # chunk r's accumulator: after cp passes to the next rank it is back at r
            at = r
            for _ in range(cp):
                at = R.next_rank(at, cp)
            assert at == r
