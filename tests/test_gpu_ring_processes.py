"""GPU: the ring across ranks as each rank runs it (ring.py's ring_forward and
ring_backward in a process of its own, every step's arithmetic in the library),
two and three processes sharing this one GPU.

The exchange is the host-staged one over gloo: each process's kernels run on their
own and only the host waits for the other ranks, so no kernel waits on a kernel of
another process (NCCL's point-to-point kernels between processes on one GPU would).
Checked: every rank held the chunk (r - i) mod cp at step i, and its forward rows,
dQ rows and home-coming dK/dV chunk equal the oracle's."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import workloads as W
from gpu_helpers import LSE_ABS_TOL, TOL, full_reference, rel
from oracle import layouts as OL

pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("rp_tc_T1024_cp2_zz_gqa2", 1, 4, 2, 1024, 128, 2, "zigzag", "bf16"),
    W.Workload("rp_tc_T768_cp3_contig_D64", 2, 2, 2, 768, 64, 3, "contiguous", "bf16"),
    W.Workload("rp_simt_f32_T96_cp3_zz", 1, 2, 1, 96, 20, 3, "zigzag", "f32"),
]


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, w, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import blockwise_online_softmax_cpattn_gb300 as cp
        from blockwise_online_softmax_cpattn_gb300 import ring as R
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        nat = W.draw_cast(w)
        pos = torch.from_numpy(OL.positions(w.T, w.cp, w.layout))
        c = w.T // w.cp
        mine = [x[:, :, pos][:, :, rank * c:(rank + 1) * c].contiguous().to(dev) for x in nat]
        d = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype)
        steps = R.LibrarySteps(d, device=dev)
        exch = R.HostExchange()
        o, lse, held_f = R.ring_forward(steps, exch, mine[0], mine[1], mine[2])
        dq, dk, dv, held_b = R.ring_backward(steps, exch, mine[0], mine[1], mine[2], o, lse,
                                             mine[3])
        cp.check(cp.cpattn_check())
        out.put((rank, [t.cpu() for t in (o, lse, dq, dk, dv)], held_f, held_b))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_ring_ranks_as_processes_match_oracle(w):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_rank, args=(r, w.cp, port, w, out)) for r in range(w.cp)]
    for p in procs:
        p.start()
    results = sorted((out.get(timeout=300) for _ in range(w.cp)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    ref = full_reference(w, W.draw_cast(w))
    pos = OL.positions(w.T, w.cp, w.layout)
    c = w.T // w.cp
    tol = TOL[w.dtype]
    for r, (o, lse, dq, dk, dv), held_f, held_b in results:
        assert held_f == held_b == [OL.ring_source(r, i, w.cp) for i in range(w.cp)]
        p = pos[r * c:(r + 1) * c]
        assert rel(W.as_f64(o), ref["o"][:, :, p]) <= tol["o"], (w.name, "o", r)
        assert float(np.max(np.abs(lse.numpy() - ref["lse"][:, :, p]))) <= LSE_ABS_TOL[w.dtype]
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert rel(W.as_f64(got), ref[name][:, :, p]) <= tol["grad"], (w.name, name, r)
