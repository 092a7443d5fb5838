"""GPU: the bounded-wait protocol of the tensor-core forward.

With the descriptor's test hook set, the producer withholds one query-tile load,
so the MMA issuer's bounded wait on it runs out (~50 ms).  The kernel must then
latch CPATTN_ERR_TIMEOUT in the device status word, stop its other roles, drain
its own copies, free its tensor memory and exit; cpattn_check reports the error
once, and the context keeps working for the next call.  Nothing here faults or
hangs the GPU: the wait that runs out is on a flag nothing sets."""
import pytest
import torch

import workloads as W
from gpu_helpers import assert_close, full_reference, ring_inputs, run_ring, cp_mod, desc_of, dev

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_context_survives():
    cp = cp_mod()
    w = W.Workload("fault_hook", 1, 2, 2, 256, 64, 1, "contiguous", "bf16")
    nat, lay = ring_inputs(w)
    ql, kl, vl, _ = lay
    assert cp.cpattn_check() == cp.OK
    d = desc_of(w, debug_fault=1)
    o = torch.empty_like(ql)
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    assert cp.cpattn_ring_fwd(d, ql, kl, vl, o, lse) == cp.OK   # enqueued fine
    assert cp.cpattn_check() == cp.ERR_TIMEOUT
    assert cp.cpattn_check() == cp.OK                           # cleared once read
    got = run_ring(w, lay)                                      # the context still works
    assert_close(w, got, full_reference(w, nat))
