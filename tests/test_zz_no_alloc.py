"""cpattn_ring_bwd_noalloc: the backward for callers that cannot allocate device
memory (engine plugins that may only use buffers handed to them, programs that
reserve all memory up front).  It must give what cpattn_ring_bwd gives with a
caller workspace, on consecutive calls that share the library's scratch, and
refuse problems larger than that scratch before enqueueing anything.

This file is collected last so that, in a run that stops at the first failure,
every other test has already run."""
import pytest
import torch

import workloads as W
from gpu_helpers import TOL, cp_mod, desc_of, dev, rel, ring_inputs

FAKE = 0x10000  # aligned, never dereferenced: the call returns before any launch


def _reference_and_noalloc(w, seed):
    cp = cp_mod()
    _, (q, k, v, do) = ring_inputs(w, seed)
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
    return ref, got


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_on_two_calls():
    tol = TOL["bf16"]["grad"]
    first = W.Workload("noalloc_gqa", 1, 8, 2, 2048, 128, 4, "zigzag", "bf16")
    second = W.Workload("noalloc_mha", 2, 4, 4, 1024, 64, 2, "contiguous", "bf16")
    for w, seed in ((first, 3), (second, 4)):  # two calls in a row, different problems
        ref, got = _reference_and_noalloc(w, seed)
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(a.float()).all(), (w.name, name)
            e = rel(a.float().cpu().numpy(), b.float().cpu().numpy())
            assert e <= tol, (w.name, name, e)


def test_noalloc_refuses_problems_beyond_its_scratch():
    cp = cp_mod()
    # 1 x 32 x 131072 = 4,194,304 query rows > 2,097,152
    big = cp.make_desc(1, 32, 8, 131072, 128, 8, "zigzag", "bf16")
    args = [FAKE] * 9 + [0]
    assert cp.cpattn_ring_bwd_noalloc(big, *args) == cp.ERR_UNSUPPORTED
    bad = cp.make_desc(1, 3, 2, 1024, 64, 2, "zigzag", "bf16")   # H_q % H_kv != 0
    assert cp.cpattn_ring_bwd_noalloc(bad, *args) == cp.ERR_INVALID_ARG
