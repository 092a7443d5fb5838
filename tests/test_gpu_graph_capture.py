"""GPU: the ring forward and backward captured in a CUDA graph.

The backward launches its dQ kernel as a programmatic dependent of its dK/dV
kernel and zeroes the dQ kernel's item counter with a memset on the call's
stream; a stream capture turns both into graph nodes (a programmatic edge and a
memset node).  A replay must give the eager calls' results bit for bit (the
kernels are deterministic), for the plain ring and for packed sequences, and the
replay must leave the counter ready for the next one."""
import pytest
import torch

import workloads as W
from gpu_helpers import cp_mod, desc_of, dev, ring_inputs

pytestmark = pytest.mark.gpu

W_RING = W.Workload("graph_gqa4_T1024_D128_cp4_zz", 1, 8, 2, 1024, 128, 4, "zigzag", "bf16")


def _capture_and_compare(step):
    eager = [x.clone() for x in step()]
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        captured = step()
    for rep in range(2):  # two replays: the first must leave the counter ready
        for x in captured:
            x.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        cp_mod().check(cp_mod().cpattn_check())
        for a, b in zip(captured, eager):
            assert torch.equal(a, b), rep


def test_ring_fwd_bwd_replays_from_a_cuda_graph():
    cp = cp_mod()
    w = W_RING
    _, (ql, kl, vl, dol) = ring_inputs(w)
    d = desc_of(w)
    o, lse = torch.empty_like(ql), torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    dq, dk, dv = torch.empty_like(ql), torch.empty_like(kl), torch.empty_like(vl)
    ws = torch.empty(cp.cpattn_ring_bwd_workspace(d), dtype=torch.uint8, device=dev())

    def step():
        cp.check(cp.cpattn_ring_fwd(d, ql, kl, vl, o, lse))
        cp.check(cp.cpattn_ring_bwd(d, ql, kl, vl, o, lse, dol, dq, dk, dv, ws))
        return [o, lse, dq, dk, dv]

    _capture_and_compare(step)


def test_packed_fwd_bwd_replays_from_a_cuda_graph():
    cp = cp_mod()
    w = W_RING
    _, (ql, kl, vl, dol) = ring_inputs(w)
    d = desc_of(w)
    starts = torch.from_numpy(W.packed_starts(w, 4, 7)).to(dev())
    o, lse = torch.empty_like(ql), torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    dq, dk, dv = torch.empty_like(ql), torch.empty_like(kl), torch.empty_like(vl)
    ws = torch.empty(cp.cpattn_packed_workspace(d), dtype=torch.uint8, device=dev())

    def step():
        cp.check(cp.cpattn_ring_fwd_packed(d, starts, 4, ql, kl, vl, o, lse, ws))
        cp.check(cp.cpattn_ring_bwd_packed(d, starts, 4, ql, kl, vl, o, lse, dol, dq, dk, dv, ws))
        return [o, lse, dq, dk, dv]

    _capture_and_compare(step)
