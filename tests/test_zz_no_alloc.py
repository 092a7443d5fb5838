"""cpattn_ring_bwd_noalloc: the backward for callers that cannot allocate device
memory (engine plugins that may only use buffers handed to them, programs that
reserve all memory up front).  It runs the same deterministic kernels as
cpattn_ring_bwd, only with the library's own scratch in place of the caller's
workspace, so on the same inputs its gradients must equal cpattn_ring_bwd's bit
for bit, on consecutive calls that share that scratch; and it must refuse
problems larger than the scratch before enqueueing anything.

This file is collected last so that, in a run that stops at the first failure,
every other test has already run."""
import pytest
import torch

import workloads as W
from gpu_helpers import TOL, cp_mod, desc_of, dev, full_reference, rel, ring_inputs, to_nat

FAKE = 0x10000  # aligned, never dereferenced: the call returns before any launch


@pytest.fixture(scope="module")
def cp():
    import __graft_entry__
    __graft_entry__.build()
    return cp_mod()


def _reference_and_noalloc(cp, w, seed):
    nat, (q, k, v, do) = ring_inputs(w, seed)
    d = desc_of(w)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    cp.check(cp.cpattn_ring_fwd(d, q, k, v, o, lse))
    ref = [torch.empty_like(x) for x in (q, k, v)]
    ws = torch.empty(cp.cpattn_ring_bwd_workspace(d), dtype=torch.uint8, device=dev())
    cp.check(cp.cpattn_ring_bwd(d, q, k, v, o, lse, do, *ref, ws))
    got = [torch.full_like(x, float("nan")) for x in (q, k, v)]
    cp.check(cp.cpattn_ring_bwd_noalloc(d, q, k, v, o, lse, do, *got))
    cp.check(cp.cpattn_check())
    return nat, ref, got


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_on_two_calls(cp):
    first = W.Workload("noalloc_gqa", 1, 8, 2, 2048, 128, 4, "zigzag", "bf16")
    second = W.Workload("noalloc_mha", 2, 4, 4, 1024, 64, 2, "contiguous", "bf16")
    for w, seed in ((first, 3), (second, 4)):  # two calls in a row, different problems
        nat, ref, got = _reference_and_noalloc(cp, w, seed)
        oracle = full_reference(w, nat)
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            # the same atomic-free kernels on the same inputs: anything short of
            # bit equality would be a scratch mix-up (stale or misplaced statistics)
            assert torch.equal(a, b), (w.name, name)
            assert rel(to_nat(a, w), oracle[name]) <= TOL["bf16"]["grad"], (w.name, name)


def test_noalloc_refuses_problems_beyond_its_scratch(cp):
    # 1 x 32 x 131072 = 4,194,304 query rows > 2,097,152
    big = cp.make_desc(1, 32, 8, 131072, 128, 8, "zigzag", "bf16")
    args = [FAKE] * 9 + [0]
    assert cp.cpattn_ring_bwd_noalloc(big, *args) == cp.ERR_UNSUPPORTED
    bad = cp.make_desc(1, 3, 2, 1024, 64, 2, "zigzag", "bf16")   # H_q % H_kv != 0
    assert cp.cpattn_ring_bwd_noalloc(bad, *args) == cp.ERR_INVALID_ARG
