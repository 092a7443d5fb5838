"""GPU: cpattn_ring_step_host (one forward + backward step over tensors in host
memory, transfers overlapping the compute) gives what the device-resident path
gives (cpattn_layout to layout order, cpattn_ring_fwd, cpattn_ring_bwd, cpattn_layout
back to natural order), bit for bit: its halves are independent problems run by the
same kernels with the same per-tile arithmetic.  Pinned and pageable host buffers;
splits by K/V heads (B = 1: halves, and a forward in quarters), by batch rows (B 4:
halves, forward quarters), by batch rows for the backward and heads within a row
for the forward (B 2); an unsplit float32 problem and a split one (whose dk and dv
come back after both backward kernels)."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import TOL, cp_mod, desc_of, dev, full_reference, rel

pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("hs_tc_B1_H8x2_T2048_cp4_zz", 1, 8, 2, 2048, 128, 4, "zigzag", "bf16"),
    W.Workload("hs_tc_B2_H4x4_T1024_cp2_contig_D64", 2, 4, 4, 1024, 64, 2, "contiguous", "bf16"),
    W.Workload("hs_tc_B1_H8x4_T1024_cp2_zz", 1, 8, 4, 1024, 128, 2, "zigzag", "bf16"),
    W.Workload("hs_tc_B4_H2x1_T512_cp2_zz_D64", 4, 2, 1, 512, 64, 2, "zigzag", "bf16"),
    W.Workload("hs_simt_B3_H2x1_T96_cp3_zz_f32", 3, 2, 1, 96, 20, 3, "zigzag", "f32"),
    W.Workload("hs_simt_B2_H4x2_T64_cp2_zz_f32", 2, 4, 2, 64, 16, 2, "zigzag", "f32"),
]


def _device_path(cp, w, nat_dev):
    """The same step with every tensor already on the device."""
    d = desc_of(w)
    H = [w.H_q, w.H_kv, w.H_kv, w.H_q]
    lay = [torch.empty_like(x) for x in nat_dev]
    cp.check(cp.cpattn_layout_batch(cp.ZIGZAG_FWD, d, nat_dev, lay, H))
    o = torch.empty_like(lay[0])
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    cp.check(cp.cpattn_ring_fwd(d, lay[0], lay[1], lay[2], o, lse))
    dq, dk, dv = torch.empty_like(lay[0]), torch.empty_like(lay[1]), torch.empty_like(lay[2])
    ws = torch.empty(cp.cpattn_ring_bwd_workspace(d), dtype=torch.uint8, device=dev())
    cp.check(cp.cpattn_ring_bwd(d, lay[0], lay[1], lay[2], o, lse, lay[3], dq, dk, dv, ws))
    outs = [torch.empty_like(x) for x in (o, dq, dk, dv)]
    cp.check(cp.cpattn_layout_batch(cp.ZIGZAG_INV, d, [o, dq, dk, dv], outs,
                                    [w.H_q, w.H_q, w.H_kv, w.H_kv]))
    d_lse = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, 1, w.cp, w.layout, "f32")
    lse_nat = torch.empty_like(lse)
    cp.check(cp.cpattn_layout(cp.ZIGZAG_INV, d_lse, lse, lse_nat, w.H_q))
    cp.check(cp.cpattn_check())
    return {"o": outs[0], "lse": lse_nat, "dq": outs[1], "dk": outs[2], "dv": outs[3]}


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_host_step_equals_the_device_path(w, pinned):
    cp = cp_mod()
    nat = W.draw_cast(w)
    d = desc_of(w)
    host_in = [x.pin_memory() if pinned else x.clone() for x in nat]

    def host_like(x, dtype=None):
        t = torch.full(x.shape, float("nan"), dtype=dtype or x.dtype)
        return t.pin_memory() if pinned else t

    out = {"o": host_like(nat[0]), "lse": host_like(nat[0][..., 0], torch.float32),
           "dq": host_like(nat[0]), "dk": host_like(nat[1]), "dv": host_like(nat[2])}
    ws = torch.empty(cp.cpattn_ring_step_host_workspace(d), dtype=torch.uint8, device=dev())
    for _ in range(2):  # twice in a row: the staging and the shared copy streams are reused
        cp.check(cp.cpattn_ring_step_host(d, *host_in, out["o"], out["lse"], out["dq"], out["dk"],
                                          out["dv"], ws))
        cp.check(cp.cpattn_check())
        ref = _device_path(cp, w, [x.to(dev()) for x in nat])
        for key in ("o", "lse", "dq", "dk", "dv"):
            assert torch.equal(out[key], ref[key].cpu()), (w.name, key)
    oracle = full_reference(w, nat)
    tol = TOL[w.dtype]
    assert rel(W.as_f64(out["o"]), oracle["o"]) <= tol["o"]
    for key in ("dq", "dk", "dv"):
        assert rel(W.as_f64(out[key]), oracle[key]) <= tol["grad"], key
    assert float(np.max(np.abs(out["lse"].double().numpy() - oracle["lse"]))) <= 2e-3
