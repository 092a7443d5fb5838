"""GPU: cpattn_partial_bwd (one ring step of the backward) against the oracle's
per-step backward, the steps accumulated in ring order against the full
backward, and the point-to-point ring driver run in one process through the
library (tutorial "上下文并行", section "朴素 Ring Attention": each step
recomputes its probabilities; pull request #181, mode "p2p": a chunk's K/V
gradient travels the ring back to its owner)."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import LSE_ABS_TOL, TOL, cp_mod, desc_of, dev, full_reference, rel, ring_inputs
from oracle import attention as OA
from oracle import layouts as OL

pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("pb_tc_T1024_cp4_zz_gqa2", 1, 4, 2, 1024, 128, 4, "zigzag", "bf16"),
    W.Workload("pb_tc_T768_cp3_contig_D64", 2, 2, 2, 768, 64, 3, "contiguous", "bf16"),
    W.Workload("pb_tc_T2048_cp2_zz_gqa4", 1, 8, 2, 2048, 128, 2, "zigzag", "bf16"),
    W.Workload("pb_simt_f32_T96_cp3_zz", 1, 2, 1, 96, 20, 3, "zigzag", "f32"),
    W.Workload("pb_simt_f32_T64_cp4", 2, 4, 2, 64, 16, 4, "contiguous", "f32"),
]


def _forward(w, lay):
    cp = cp_mod()
    ql, kl, vl, _ = lay
    d = desc_of(w)
    o = torch.empty_like(ql)
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    cp.check(cp.cpattn_ring_fwd(d, ql, kl, vl, o, lse))
    return o, lse


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_partial_bwd_steps_match_oracle_and_sum_to_the_backward(w):
    cp = cp_mod()
    nat, lay = ring_inputs(w)
    ql, kl, vl, dol = lay
    d = desc_of(w)
    o, lse = _forward(w, lay)
    q, k, v, do = (W.as_f64(x) for x in nat)
    ro, rlse = OA.attention_fwd(q, k, v, w.scale)
    rdq, rdk, rdv = OA.attention_bwd(q, k, v, do, w.scale)
    c = w.T // w.cp
    n_rep = w.H_q // w.H_kv
    pos = OL.positions(w.T, w.cp, w.layout)
    tol = TOL[w.dtype]["grad"]
    f32 = dict(dtype=torch.float32, device=dev())
    acc_dq = [torch.empty(w.B, w.H_q, c, w.D, **f32) for _ in range(w.cp)]
    acc_dk = [torch.empty(w.B, w.H_kv, c, w.D, **f32) for _ in range(w.cp)]
    acc_dv = [torch.empty(w.B, w.H_kv, c, w.D, **f32) for _ in range(w.cp)]
    # every rank's statistics, once (a workspace per rank)
    do_rows, stats = [], []
    for r in range(w.cp):
        sl_r = slice(r * c, (r + 1) * c)
        o_r, lse_r, do_r = (x[:, :, sl_r].contiguous() for x in (o, lse, dol))
        stats.append(torch.full((cp.cpattn_partial_bwd_workspace(d),), 255, dtype=torch.uint8,
                                device=dev()))
        cp.check(cp.cpattn_partial_bwd_stats(d, o_r, lse_r, do_r, stats[r]))
        do_rows.append(do_r)
    for i in range(w.cp):
        for r in range(w.cp):
            s = OL.ring_source(r, i, w.cp)
            sl_r, sl_s = slice(r * c, (r + 1) * c), slice(s * c, (s + 1) * c)
            do_r = do_rows[r]
            # the step alone (accumulate = 0) against the oracle's step
            one = [torch.full_like(t, float("nan")) for t in (acc_dq[r], acc_dk[s], acc_dv[s])]
            cp.check(cp.cpattn_partial_bwd(d, r, s, ql, kl, vl, do_r, *one, 0, stats[r]))
            qp, kp = pos[sl_r], pos[sl_s]
            sdq = np.zeros((w.B, w.H_q, c, w.D))
            sdk = np.zeros((w.B, w.H_kv, c, w.D))
            sdv = np.zeros((w.B, w.H_kv, c, w.D))
            for b in range(w.B):
                for h in range(w.H_q):
                    g = h // n_rep
                    a, bb, e = OA.partial_attention_bwd(q[b, h, qp], k[b, g, kp], v[b, g, kp],
                                                        do[b, h, qp], ro[b, h, qp], rlse[b, h, qp],
                                                        qp, kp, w.scale)
                    sdq[b, h] = a
                    sdk[b, g] += bb
                    sdv[b, g] += e
            for name, got, ref in (("dq", one[0], sdq), ("dk", one[1], sdk), ("dv", one[2], sdv)):
                g64 = got.double().cpu().numpy()
                if not ref.any():  # no visible pair: exact zeros
                    assert not g64.any(), (w.name, r, s, name)
                else:
                    assert rel(g64, ref) <= tol, (w.name, r, s, name, rel(g64, ref))
            # the ring in step order: dQ of rank r and the chunk's dK/dV accumulate
            cp.check(cp.cpattn_partial_bwd(d, r, s, ql, kl, vl, do_r, acc_dq[r], acc_dk[s],
                                           acc_dv[s], int(i > 0), stats[r]))
    cp.check(cp.cpattn_check())
    for r in range(w.cp):
        p = pos[r * c:(r + 1) * c]
        assert rel(acc_dq[r].double().cpu().numpy(), rdq[:, :, p]) <= tol, (w.name, "dq", r)
        assert rel(acc_dk[r].double().cpu().numpy(), rdk[:, :, p]) <= tol, (w.name, "dk", r)
        assert rel(acc_dv[r].double().cpu().numpy(), rdv[:, :, p]) <= tol, (w.name, "dv", r)


@pytest.mark.parametrize("w", [CASES[0], CASES[1], CASES[3]], ids=lambda w: w.name)
def test_ring_driver_emulated_on_one_gpu(w):
    """The point-to-point ring's per-rank steps (ring.py), all ranks in one process,
    every step's arithmetic in the library: forward rows and LSE, dQ rows and the
    dK/dV chunks that come home, against the oracle."""
    cp = cp_mod()
    from blockwise_online_softmax_cpattn_gb300 import ring as R
    nat, lay = ring_inputs(w)
    d = desc_of(w)
    steps = R.LibrarySteps(d, device=dev())
    qs, ks, vs, dos = (R.rank_chunks(x, w.cp) for x in lay)
    os_, lses, held_f = R.emulate_ring_forward(steps, w.cp, qs, ks, vs)
    dqs, dks, dvs, held_b = R.emulate_ring_backward(steps, w.cp, qs, ks, vs, os_, lses, dos)
    cp.check(cp.cpattn_check())
    ref = full_reference(w, nat)
    pos = OL.positions(w.T, w.cp, w.layout)
    c = w.T // w.cp
    tol = TOL[w.dtype]
    for r in range(w.cp):
        assert held_f[r] == held_b[r] == [OL.ring_source(r, i, w.cp) for i in range(w.cp)]
        p = pos[r * c:(r + 1) * c]
        assert rel(W.as_f64(os_[r]), ref["o"][:, :, p]) <= tol["o"], (w.name, "o", r)
        assert float(np.max(np.abs(lses[r].cpu().numpy() - ref["lse"][:, :, p]))) <= \
            LSE_ABS_TOL[w.dtype]
        for name, got in (("dq", dqs[r]), ("dk", dks[r]), ("dv", dvs[r])):
            assert rel(W.as_f64(got), ref[name][:, :, p]) <= tol["grad"], (w.name, name, r)


def test_ring_driver_replays_from_a_cuda_graph():
    """The emulated ring's library calls are safe to capture in a CUDA graph: a
    replay gives the eager run's results bit for bit (the kernels are deterministic)
    and so matches the oracle."""
    from blockwise_online_softmax_cpattn_gb300 import ring as R
    cp = cp_mod()
    w = CASES[0]
    nat, lay = ring_inputs(w)
    steps = R.LibrarySteps(desc_of(w), device=dev())
    chunks = [R.rank_chunks(x, w.cp) for x in lay]

    def step():
        os_, lses, _ = R.emulate_ring_forward(steps, w.cp, *chunks[:3])
        dqs, dks, dvs, _ = R.emulate_ring_backward(steps, w.cp, *chunks[:3], os_, lses, chunks[3])
        return os_ + lses + dqs + dks + dvs

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
    for x in captured:
        x.zero_()
    g.replay()
    torch.cuda.synchronize()
    cp.check(cp.cpattn_check())
    for a, b in zip(captured, eager):
        assert torch.equal(a, b)
