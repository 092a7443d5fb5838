"""GPU: cpattn_partial_fwd (one ring step) against the oracle's partial attention,
and merging the partials of all steps with cpattn_merge in ring order against
full causal attention (tutorial "上下文并行", section "朴素 Ring Attention": the
block order does not matter when the running O, max and sum are carried)."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import TOL, cp_mod, desc_of, dev, full_reference, rel, ring_inputs
from oracle import attention as OA
from oracle import layouts as OL

pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("p_tc_T1024_cp4_zz", 1, 4, 2, 1024, 64, 4, "zigzag", "bf16"),
    W.Workload("p_tc_T1024_cp2_contig", 1, 2, 2, 1024, 128, 2, "contiguous", "bf16"),
    W.Workload("p_tc_T1024_cp2_zz_gqa3", 1, 3, 1, 1024, 128, 2, "zigzag", "bf16"),
    W.Workload("p_simt_f32_T64_cp4", 1, 2, 2, 64, 16, 4, "contiguous", "f32"),
    W.Workload("p_simt_f32_T96_cp3_zz", 1, 2, 1, 96, 20, 3, "zigzag", "f32"),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_partials_and_merge(w):
    cp = cp_mod()
    nat, lay = ring_inputs(w)
    ql, kl, vl, _ = lay
    q, k, v, _ = (W.as_f64(x) for x in nat)
    desc = desc_of(w)
    c = w.T // w.cp
    pos = OL.positions(w.T, w.cp, w.layout)
    n_rep = w.H_q // w.H_kv
    ref = full_reference(w, nat, bwd=False)
    tol = TOL[w.dtype]["o"]
    for r in range(w.cp):
        qp = pos[r * c:(r + 1) * c]
        acc_o = torch.zeros(w.B, w.H_q, c, w.D, dtype=torch.float32, device=dev())
        acc_l = torch.full((w.B, w.H_q, c), -float("inf"), dtype=torch.float32, device=dev())
        for i in range(w.cp):
            s = OL.ring_source(r, i, w.cp)
            kp = pos[s * c:(s + 1) * c]
            o = torch.empty(w.B, w.H_q, c, w.D, dtype=torch.float32, device=dev())
            lse = torch.empty(w.B, w.H_q, c, dtype=torch.float32, device=dev())
            cp.check(cp.cpattn_partial_fwd(desc, r, s, ql, kl, vl, o, lse))
            go, gl = o.cpu().numpy(), lse.cpu().numpy()
            for b in range(w.B):
                for h in range(w.H_q):
                    ro, rl = OA.partial_attention(q[b, h, qp], k[b, h // n_rep, kp],
                                                  v[b, h // n_rep, kp], qp, kp, w.scale)
                    empty = ~np.isfinite(rl)
                    assert np.array_equal(~np.isfinite(gl[b, h]), empty), (r, s, b, h)
                    assert np.all(go[b, h][empty] == 0)
                    if (~empty).any():
                        assert rel(go[b, h][~empty], ro[~empty]) <= tol, (r, s, b, h)
                        assert np.max(np.abs(gl[b, h][~empty] - rl[~empty])) <= 2e-3
            cp.check(cp.cpattn_merge(w.B * w.H_q * c, w.D, acc_o, acc_l, o, lse, acc_o, acc_l))
        got = acc_o.cpu().numpy()
        want = ref["o"][:, :, qp]
        assert rel(got, want) <= tol, r
        assert np.max(np.abs(acc_l.cpu().numpy() - ref["lse"][:, :, qp])) <= 2e-3
    cp.check(cp.cpattn_check())
