"""GPU: the all-gather mode (pull request "Feat: Context Parallel" #181, mode table
row "all_gather": each rank runs its own queries over the gathered K/V; the K/V
gradients of all ranks are summed by a ReduceScatter) against the oracle.

Per rank: cpattn_allgather_fwd's rows and LSE and cpattn_allgather_bwd's dQ rows
against the oracle's all-gather functions at that rank's positions; the first
rank's K/V gradient share alone (accumulate = 0); and the float32 sums after all
ranks (accumulate = 1) against the full backward.  Outputs are brought to natural
order with the oracle's own index maps."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import LSE_ABS_TOL, TOL, cp_mod, desc_of, dev, rel, ring_inputs
from oracle import attention as OA
from oracle import layouts as OL

pytestmark = pytest.mark.gpu

CASES = [
    # tensor-core path: several 128-token tiles per chunk half, zigzag and contiguous,
    # grouped queries, both head dimensions
    W.Workload("ag_tc_T2048_cp4_zz_gqa4", 1, 8, 2, 2048, 128, 4, "zigzag", "bf16"),
    W.Workload("ag_tc_T1024_cp2_contig", 2, 2, 2, 1024, 64, 2, "contiguous", "bf16"),
    W.Workload("ag_tc_T1024_cp4_zz_gqa3", 1, 3, 1, 1024, 128, 4, "zigzag", "bf16"),
    W.Workload("ag_tc_T512_cp1", 1, 2, 1, 512, 64, 1, "zigzag", "bf16"),
    W.Workload("ag_tc_T2048_cp8_zz_D64_gqa2", 2, 4, 2, 2048, 64, 8, "zigzag", "bf16"),
    # SIMT paths: exact float32, and bf16 with a head dimension the tensor cores skip
    W.Workload("ag_simt_f32_T96_cp3_zz", 1, 2, 1, 96, 20, 3, "zigzag", "f32"),
    W.Workload("ag_simt_f32_T64_cp4", 2, 4, 2, 64, 16, 4, "contiguous", "f32"),
    W.Workload("ag_simt_bf16_T128_cp2_D32", 1, 2, 2, 128, 32, 2, "zigzag", "bf16"),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_allgather_matches_oracle(w):
    cp = cp_mod()
    nat, lay = ring_inputs(w)
    ql, kl, vl, dol = lay
    q, k, v, do = (W.as_f64(x) for x in nat)
    desc = desc_of(w)
    c = w.T // w.cp
    tol = TOL[w.dtype]
    tdt = ql.dtype
    dk_sum = torch.empty(w.B, w.H_kv, w.T, w.D, dtype=torch.float32, device=dev())
    dv_sum = torch.empty_like(dk_sum)
    ws = torch.empty(cp.cpattn_allgather_bwd_workspace(desc), dtype=torch.uint8, device=dev())
    for r in range(w.cp):
        pos = OL.rank_positions(w.T, w.cp, w.layout, r)
        o = torch.empty(w.B, w.H_q, c, w.D, dtype=tdt, device=dev())
        lse = torch.empty(w.B, w.H_q, c, dtype=torch.float32, device=dev())
        cp.check(cp.cpattn_allgather_fwd(desc, r, ql, kl, vl, o, lse))
        ro, rlse = OA.allgather_fwd(q, k, v, w.scale, pos)
        assert rel(W.as_f64(o), ro) <= tol["o"], (w.name, r)
        assert float(np.max(np.abs(lse.cpu().numpy() - rlse))) <= LSE_ABS_TOL[w.dtype]
        dq = torch.empty_like(o)
        do_r = dol[:, :, r * c:(r + 1) * c].contiguous()
        cp.check(cp.cpattn_allgather_bwd(desc, r, ql, kl, vl, o, lse, do_r, dq, dk_sum, dv_sum,
                                         r > 0, ws))
        rdq, rdk, rdv = OA.allgather_bwd(q, k, v, do, w.scale, pos)
        assert rel(W.as_f64(dq), rdq) <= tol["grad"], (w.name, r, "dq")
        if r == 0:
            # one rank's share alone, before any other rank adds to it
            gk = OL.to_natural(dk_sum.cpu().double().numpy(), w.cp, w.layout, axis=2)
            gv = OL.to_natural(dv_sum.cpu().double().numpy(), w.cp, w.layout, axis=2)
            assert rel(gk, rdk) <= tol["grad"], (w.name, "dk share")
            assert rel(gv, rdv) <= tol["grad"], (w.name, "dv share")
    cp.check(cp.cpattn_check())
    _, fdk, fdv = OA.attention_bwd(q, k, v, do, w.scale)
    gk = OL.to_natural(dk_sum.cpu().double().numpy(), w.cp, w.layout, axis=2)
    gv = OL.to_natural(dv_sum.cpu().double().numpy(), w.cp, w.layout, axis=2)
    assert rel(gk, fdk) <= tol["grad"], (w.name, "dk sum")
    assert rel(gv, fdv) <= tol["grad"], (w.name, "dv sum")


def test_allgather_equals_ring():
    """Ranks' all-gather rows put side by side are the ring's output (same kernels'
    arithmetic over the same keys, in another order): close to bf16 rounding."""
    w = W.Workload("ag_vs_ring", 1, 4, 2, 1024, 128, 4, "zigzag", "bf16")
    cp = cp_mod()
    _, lay = ring_inputs(w)
    ql, kl, vl, _ = lay
    desc = desc_of(w)
    c = w.T // w.cp
    o_ring = torch.empty_like(ql)
    lse_ring = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    cp.check(cp.cpattn_ring_fwd(desc, ql, kl, vl, o_ring, lse_ring))
    for r in range(w.cp):
        o = torch.empty(w.B, w.H_q, c, w.D, dtype=ql.dtype, device=dev())
        lse = torch.empty(w.B, w.H_q, c, dtype=torch.float32, device=dev())
        cp.check(cp.cpattn_allgather_fwd(desc, r, ql, kl, vl, o, lse))
        sl = slice(r * c, (r + 1) * c)
        assert torch.allclose(lse, lse_ring[:, :, sl], atol=1e-4, rtol=0)
        assert (o.float() - o_ring[:, :, sl].float()).abs().max().item() <= 1e-2
    cp.check(cp.cpattn_check())


def test_allgather_backward_is_deterministic():
    """Each rank's dQ kernel overlaps the end of its dK/dV kernel and its CTAs claim
    their query tiles from a counter, so which CTA computes a tile changes from run
    to run; each tile is still computed the same way, and the K/V sums get one float32
    addition per element per rank in rank order.  Two runs give identical bits."""
    cp = cp_mod()
    w = CASES[0]
    _, lay = ring_inputs(w)
    ql, kl, vl, dol = lay
    desc = desc_of(w)
    c = w.T // w.cp
    ws = torch.empty(cp.cpattn_allgather_bwd_workspace(desc), dtype=torch.uint8, device=dev())

    def run():
        dk_sum = torch.empty(w.B, w.H_kv, w.T, w.D, dtype=torch.float32, device=dev())
        dv_sum = torch.empty_like(dk_sum)
        dqs = []
        for r in range(w.cp):
            o = torch.empty(w.B, w.H_q, c, w.D, dtype=ql.dtype, device=dev())
            lse = torch.empty(w.B, w.H_q, c, dtype=torch.float32, device=dev())
            cp.check(cp.cpattn_allgather_fwd(desc, r, ql, kl, vl, o, lse))
            dq = torch.empty_like(o)
            do_r = dol[:, :, r * c:(r + 1) * c].contiguous()
            cp.check(cp.cpattn_allgather_bwd(desc, r, ql, kl, vl, o, lse, do_r, dq, dk_sum,
                                             dv_sum, r > 0, ws))
            dqs.append(dq)
        cp.check(cp.cpattn_check())
        return dqs + [dk_sum, dv_sum]

    for a, b in zip(run(), run()):
        assert torch.equal(a, b)
