"""Helpers of the GPU parity tests: run the CUDA path through the C ABI on seeded
inputs and bring its outputs back to natural order with the ORACLE's own index
maps (never with the library's permute kernels)."""
import numpy as np
import torch

import workloads as W
from oracle import attention as OA
from oracle import layouts as OL

TOL = {"f32": {"o": 1e-5, "grad": 1e-5}, "bf16": {"o": 1e-2, "grad": 3e-2}}
LSE_ABS_TOL = {"f32": 1e-5, "bf16": 2e-3}


def cp_mod():
    import blockwise_online_softmax_cpattn_gb300 as cp
    return cp


def dev():
    return torch.device("cuda:0")


def ring_inputs(w, seed=None):
    """Seeded inputs in the workload dtype: natural-order host copies and
    layout-order device copies."""
    q, k, v, do = W.draw_cast(w, seed)
    pos = torch.from_numpy(OL.positions(w.T, w.cp // w.a2a, w.layout))
    lay = [x[:, :, pos].contiguous().to(dev()) for x in (q, k, v, do)]
    return (q, k, v, do), lay


def desc_of(w, **kw):
    cp = cp_mod()
    return cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype, a2a=w.a2a, **kw)


def run_ring(w, lay, bwd=True):
    cp = cp_mod()
    ql, kl, vl, dol = lay
    desc = desc_of(w)
    o = torch.empty_like(ql)
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    cp.check(cp.cpattn_ring_fwd(desc, ql, kl, vl, o, lse))
    out = {"o": o, "lse": lse}
    if bwd:
        dq, dk, dv = torch.empty_like(ql), torch.empty_like(kl), torch.empty_like(vl)
        ws = torch.empty(cp.cpattn_ring_bwd_workspace(desc), dtype=torch.uint8, device=dev())
        cp.check(cp.cpattn_ring_bwd(desc, ql, kl, vl, o, lse, dol, dq, dk, dv, ws))
        out.update(dq=dq, dk=dk, dv=dv)
    cp.check(cp.cpattn_check())
    return out


def to_nat(x, w):
    """Layout-order [B, H, T, ...] device tensor -> natural-order float64 numpy."""
    a = W.as_f64(x)
    return OL.to_natural(a, w.cp // w.a2a, w.layout, axis=2)


def rel(x, ref):
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(x - ref)) / den) if den > 0 else float(np.max(np.abs(x)))


def full_reference(w, nat_inputs, bwd=True):
    q, k, v, do = (W.as_f64(x) for x in nat_inputs)
    o, lse = OA.attention_fwd(q, k, v, w.scale)
    ref = {"o": o, "lse": lse}
    if bwd:
        ref["dq"], ref["dk"], ref["dv"] = OA.attention_bwd(q, k, v, do, w.scale)
    return ref


def assert_close(w, got, ref, keys=("o", "dq", "dk", "dv")):
    tol = TOL[w.dtype]
    errs = {}
    for key in keys:
        if key not in got:
            continue
        e = rel(to_nat(got[key], w), ref[key])
        errs[key] = e
        lim = tol["o"] if key == "o" else tol["grad"]
        assert e <= lim, f"{w.name} {key}: {e:.3e} > {lim:.0e} ({errs})"
    if "lse" in got:
        lse = to_nat(got["lse"].unsqueeze(-1), w)[..., 0]
        e = float(np.max(np.abs(lse - ref["lse"])))
        errs["lse_abs"] = e
        assert e <= LSE_ABS_TOL[w.dtype], f"{w.name} lse: {e:.3e}"
    return errs
