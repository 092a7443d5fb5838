"""GPU: outputs that start on a 16-byte but not a 32-byte boundary.  The dQ
epilogue (bf16, and a ring step's float32 dQ) and a ring step's float32 forward
output use 32-byte stores when the output is 32-byte aligned and 16-byte stores
otherwise; the C ABI asks for 16-byte alignment only.  Both paths must give the
same values bit for bit (the same arithmetic, stored differently)."""
import pytest
import torch

import workloads as W
from gpu_helpers import cp_mod, desc_of, dev, ring_inputs

pytestmark = pytest.mark.gpu

W_TC = W.Workload("al_tc_T1024_cp4_zz_gqa2", 1, 4, 2, 1024, 128, 4, "zigzag", "bf16")


def _offset_like(x, nbytes=16):
    """An uninitialised tensor shaped like x whose data starts nbytes past a 256-byte
    boundary (so 16-byte but not 32-byte aligned for nbytes = 16)."""
    n = x.numel() + 256 // x.element_size()
    buf = torch.full((n,), float("nan"), dtype=x.dtype, device=x.device)
    off = nbytes // x.element_size()
    t = buf[off:off + x.numel()].view(x.shape)
    assert t.data_ptr() % 32 == 16
    return t


def test_ring_bwd_dq_16_byte_aligned_equals_32_byte_aligned():
    cp = cp_mod()
    w = W_TC
    _, lay = ring_inputs(w)
    ql, kl, vl, dol = lay
    d = desc_of(w)
    o = torch.empty_like(ql)
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    cp.check(cp.cpattn_ring_fwd(d, ql, kl, vl, o, lse))
    ws = torch.empty(cp.cpattn_ring_bwd_workspace(d), dtype=torch.uint8, device=dev())
    outs = {}
    def aligned_like(x):
        return torch.full_like(x, float("nan"))

    for name, make in (("aligned", aligned_like), ("offset", _offset_like)):
        dq, dk, dv = make(ql), make(kl), make(vl)
        cp.check(cp.cpattn_ring_bwd(d, ql, kl, vl, o, lse, dol, dq, dk, dv, ws))
        outs[name] = (dq.clone(), dk.clone(), dv.clone())
    cp.check(cp.cpattn_check())
    for a, b in zip(outs["aligned"], outs["offset"]):
        assert torch.equal(a, b)


def test_ring_step_outputs_16_byte_aligned_equal_32_byte_aligned():
    """A ring step's float32 forward output and its float32 dQ contribution (first
    step and accumulated)."""
    cp = cp_mod()
    w = W_TC
    _, lay = ring_inputs(w)
    ql, kl, vl, dol = lay
    d = desc_of(w)
    c = w.T // w.cp
    f32 = dict(dtype=torch.float32, device=dev())
    o = torch.empty_like(ql)
    lse = torch.empty(w.B, w.H_q, w.T, **f32)
    cp.check(cp.cpattn_ring_fwd(d, ql, kl, vl, o, lse))
    r = 2
    o_r, lse_r, do_r = (x[:, :, r * c:(r + 1) * c].contiguous() for x in (o, lse, dol))
    stats = torch.empty(cp.cpattn_partial_bwd_workspace(d), dtype=torch.uint8, device=dev())
    cp.check(cp.cpattn_partial_bwd_stats(d, o_r, lse_r, do_r, stats))
    res = {}
    def aligned_like(x):
        return torch.full_like(x, float("nan"))

    for name, make in (("aligned", aligned_like), ("offset", _offset_like)):
        op = make(torch.empty(w.B, w.H_q, c, w.D, **f32))
        lp = torch.empty(w.B, w.H_q, c, **f32)
        cp.check(cp.cpattn_partial_fwd(d, r, 1, ql, kl, vl, op, lp))
        dqp = make(torch.empty(w.B, w.H_q, c, w.D, **f32))
        dkp = torch.empty(w.B, w.H_kv, c, w.D, **f32)
        dvp = torch.empty_like(dkp)
        # step r (its own chunk), then step 1 added on top
        cp.check(cp.cpattn_partial_bwd(d, r, r, ql, kl, vl, do_r, dqp, dkp, dvp, 0, stats))
        cp.check(cp.cpattn_partial_bwd(d, r, 1, ql, kl, vl, do_r, dqp, dkp, dvp, 1, stats))
        res[name] = (op.clone(), lp.clone(), dqp.clone())
    cp.check(cp.cpattn_check())
    for key, a, b in zip(("o", "lse", "dq"), res["aligned"], res["offset"]):
        assert not torch.isnan(a).any() and not torch.isnan(b).any(), key
        assert torch.equal(a, b), (key, float((a - b).abs().max()))
