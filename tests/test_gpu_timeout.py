"""GPU: the bounded-wait protocol of the tensor-core kernels.

With the descriptor's test hook set, one kernel's producer withholds one load
(1: the forward's first query tile; 2: the dK/dV kernel's first query tile; 3:
the dQ kernel's first query and dO tiles), so the bounded waits on it run out
(~50 ms).  The kernel must then latch CPATTN_ERR_TIMEOUT in the device status
word, stop its other roles, drain its own copies, free its tensor memory and
exit; cpattn_check reports the error once, and the context keeps working for the
next call.  Nothing here faults or hangs the GPU: the wait that runs out is on a
barrier that nothing completes."""
import pytest
import torch

import workloads as W
from gpu_helpers import assert_close, full_reference, ring_inputs, run_ring, cp_mod, desc_of, dev

pytestmark = pytest.mark.gpu

HOOK_FWD, HOOK_DKDV, HOOK_DQ = 1, 2, 3


def test_timeout_is_reported_and_context_survives():
    cp = cp_mod()
    w = W.Workload("fault_hook", 1, 2, 2, 256, 64, 1, "contiguous", "bf16")
    nat, lay = ring_inputs(w)
    ql, kl, vl, _ = lay
    assert cp.cpattn_check() == cp.OK
    d = desc_of(w, debug_fault=HOOK_FWD)
    o = torch.empty_like(ql)
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    assert cp.cpattn_ring_fwd(d, ql, kl, vl, o, lse) == cp.OK   # enqueued fine
    assert cp.cpattn_check() == cp.ERR_TIMEOUT
    assert cp.cpattn_check() == cp.OK                           # cleared once read
    got = run_ring(w, lay)                                      # the context still works
    assert_close(w, got, full_reference(w, nat))


@pytest.mark.parametrize("hook", [HOOK_DKDV, HOOK_DQ], ids=["dkdv", "dq"])
def test_backward_timeout_is_reported_and_context_survives(hook):
    cp = cp_mod()
    # GQA and zigzag, so the withheld tile sits inside a real multi-tile walk
    w = W.Workload("fault_hook_bwd", 1, 4, 2, 1024, 128, 2, "zigzag", "bf16")
    nat, lay = ring_inputs(w)
    ql, kl, vl, dol = lay
    assert cp.cpattn_check() == cp.OK
    d = desc_of(w)
    o = torch.empty_like(ql)
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    cp.check(cp.cpattn_ring_fwd(d, ql, kl, vl, o, lse))
    assert cp.cpattn_check() == cp.OK
    dq, dk, dv = torch.empty_like(ql), torch.empty_like(kl), torch.empty_like(vl)
    ws = torch.empty(cp.cpattn_ring_bwd_workspace(d), dtype=torch.uint8, device=dev())
    dh = desc_of(w, debug_fault=hook)
    assert cp.cpattn_ring_bwd(dh, ql, kl, vl, o, lse, dol, dq, dk, dv, ws) == cp.OK
    assert cp.cpattn_check() == cp.ERR_TIMEOUT
    assert cp.cpattn_check() == cp.OK
    got = run_ring(w, lay)                                      # both kernels work again
    assert_close(w, got, full_reference(w, nat))
