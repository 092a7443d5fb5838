"""GPU: the full-size workloads, in the launch configuration the benchmark times.

The oracle computes sampled outputs one by one from the definition: output rows
and dQ rows of chosen heads at chosen positions (each with all of its keys), and
dK/dV rows in bands near the end of the sequence (only the queries after them
take part).  Properties that hold at any size cover the rest: sum_j dK_j = 0 per
K/V head and sum_j dV_j = the group's sum of dO.  At the LLaMA shape the oracle
also computes one whole K/V group (its four query heads at every position), so a
slip confined to some middle tiles cannot hide between the samples.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (LSE_ABS_TOL, TOL, cp_mod, desc_of, dev, rel, ring_inputs, run_ring,
                         to_nat)
from oracle import attention as OA
from oracle import layouts as OL

pytestmark = pytest.mark.gpu


def _rows(T, seed):
    fixed = [0, 1, 127, 128, 129, 511, 512, 1023, 1024, T // 2 - 1, T // 2, T - 129, T - 128,
             T - 2, T - 1]
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([fixed, rng.integers(0, T, 17)]))


def _gather(x, slots, b, h):
    """Rows of a layout-order device tensor [B, H, T, D] at natural positions."""
    return W.as_f64(x[b, h, torch.from_numpy(slots)])


def check_sampled(w, nat, got, heads, kv_bands, rows_seed=0):
    """Compare sampled outputs of a ring run against the oracle."""
    q, k, v, do = nat
    n_rep = w.H_q // w.H_kv
    p2p = w.cp // w.a2a
    slot_of = OL.layout_slots(w.T, p2p, w.layout)
    rows = _rows(w.T, rows_seed)
    tol = TOL[w.dtype]
    for h in heads:
        g = h // n_rep
        qh, kg, vg, doh = (W.as_f64(x[0, hh]) for x, hh in ((q, h), (k, g), (v, g), (do, h)))
        ro, rl = OA.fwd_rows(qh, kg, vg, rows, w.scale)
        go = _gather(got["o"], slot_of[rows], 0, h)
        gl = W.as_f64(got["lse"][0, h, torch.from_numpy(slot_of[rows])])
        assert rel(go, ro) <= tol["o"], ("o", h)
        assert np.max(np.abs(gl - rl)) <= LSE_ABS_TOL[w.dtype], ("lse", h)
        rdq = OA.dq_rows(qh, kg, vg, doh, rows, w.scale)
        assert rel(_gather(got["dq"], slot_of[rows], 0, h), rdq) <= tol["grad"], ("dq", h)
    for g, band in kv_bands:
        qs = np.stack([W.as_f64(q[0, g * n_rep + i]) for i in range(n_rep)])
        dos = np.stack([W.as_f64(do[0, g * n_rep + i]) for i in range(n_rep)])
        rdk, rdv = OA.dkdv_rows(qs, W.as_f64(k[0, g]), W.as_f64(v[0, g]), dos, band, w.scale)
        assert rel(_gather(got["dk"], slot_of[band], 0, g), rdk) <= tol["grad"], ("dk", g)
        assert rel(_gather(got["dv"], slot_of[band], 0, g), rdv) <= tol["grad"], ("dv", g)
    # size-independent conservation laws of the backward
    dk = got["dk"].float()
    dv = got["dv"].float()
    sum_dk = dk.sum(dim=2)
    assert float(sum_dk.abs().max()) <= 1e-2 * float(dk.abs().sum(dim=2).max())
    do_dev = torch.stack([got["do_layout"][:, g * n_rep:(g + 1) * n_rep].float().sum(dim=(1, 2))
                          for g in range(w.H_kv)], dim=1)
    err = float((dv.sum(dim=2) - do_dev).abs().max())
    assert err <= 1e-2 * float(do_dev.abs().max()) + 1e-2 * float(dv.abs().sum(dim=2).max()) / 64


def check_whole_group(w, nat, got, g):
    """Every element of one K/V group against the oracle: O, LSE and dQ of its
    n_rep query heads at all T positions, and all of dK, dV of K/V head g."""
    n_rep = w.H_q // w.H_kv
    hq = slice(g * n_rep, (g + 1) * n_rep)
    q, do = (W.as_f64(x[:, hq]) for x in (nat[0], nat[3]))
    k, v = (W.as_f64(x[:, g:g + 1]) for x in (nat[1], nat[2]))
    ro, rlse = OA.attention_fwd(q, k, v, w.scale)
    rdq, rdk, rdv = OA.attention_bwd(q, k, v, do, w.scale)
    tol = TOL[w.dtype]
    assert rel(to_nat(got["o"][:, hq], w), ro) <= tol["o"], ("o", g)
    lse = to_nat(got["lse"][:, hq].unsqueeze(-1), w)[..., 0]
    assert float(np.max(np.abs(lse - rlse))) <= LSE_ABS_TOL[w.dtype], ("lse", g)
    assert rel(to_nat(got["dq"][:, hq], w), rdq) <= tol["grad"], ("dq", g)
    assert rel(to_nat(got["dk"][:, g:g + 1], w), rdk) <= tol["grad"], ("dk", g)
    assert rel(to_nat(got["dv"][:, g:g + 1], w), rdv) <= tol["grad"], ("dv", g)


def test_llama_gqa_T8192_cp8_zigzag():
    w = W.LLAMA
    nat, lay = ring_inputs(w)
    got = run_ring(w, lay)
    got["do_layout"] = lay[3]
    T = w.T
    bands = [(0, np.arange(T - 384, T)), (7, np.arange(T // 2, T // 2 + 128)),
             (3, np.arange(T - 128, T))]
    check_sampled(w, nat, got, heads=[0, 3, 13, 31], kv_bands=bands)
    # one K/V group in full (query heads 20-23, K/V head 5): every tile of every
    # work item of those heads, middle tiles included
    check_whole_group(w, nat, got, g=5)


def test_qwen3_gqa_a2a2_p2p4_zigzag():
    """a2a (2) x p2p (4): token shards -> a2a permute -> ring over 4 chunks ->
    inverse a2a permute of the output, at T = 32768."""
    cp = cp_mod()
    w = W.QWEN3
    nat = W.draw_cast(w)
    p2p = w.cp // w.a2a
    # what each of the 8 ranks holds before the all-to-all, from the oracle's map
    pos8 = OL.positions(w.T, w.cp, w.layout)
    desc = desc_of(w)
    lay = []
    for x in nat:
        H = x.shape[1]
        shards = x[0][:, torch.from_numpy(pos8)].reshape(H, w.cp, w.T // w.cp, w.D)
        shards = shards.permute(1, 2, 0, 3).contiguous().to(dev())        # [cp][T/cp][H][D]
        out = torch.empty(w.a2a, 1, H // w.a2a, w.T, w.D, dtype=x.dtype, device=dev())
        cp.check(cp.cpattn_layout(cp.A2A_FWD, desc, shards, out, H))
        want = x[:, :, torch.from_numpy(OL.positions(w.T, p2p, w.layout))]
        assert torch.equal(out.view(1, H, w.T, w.D).cpu().view(torch.int16),
                           want.contiguous().view(torch.int16))
        lay.append(out.view(1, H, w.T, w.D))
    got = run_ring(w, lay)
    got["do_layout"] = lay[3]
    # the output goes back to token shards; compare with the oracle's inverse map
    back = torch.empty(w.cp, 1, w.T // w.cp, w.H_q, w.D, dtype=torch.bfloat16, device=dev())
    cp.check(cp.cpattn_layout(cp.A2A_INV, desc, got["o"], back, w.H_q))
    want = OL.a2a_inverse(got["o"].view(w.a2a, 1, w.H_q // w.a2a, w.T, w.D).cpu()
                          .view(torch.int16).numpy(), 1, w.H_q, w.T, w.cp, w.a2a, w.layout)
    assert np.array_equal(back.cpu().view(torch.int16).numpy(), want)
    cp.check(cp.cpattn_check())
    T = w.T
    check_sampled(w, nat, got, heads=[0, 15, 16, 31],
                  kv_bands=[(0, np.arange(T - 256, T)), (3, np.arange(T - 256, T))])


@pytest.fixture(scope="module")
def long_inputs():
    w = W.LONG
    nat = W.draw_cast(w)
    return w, nat, [x.to(dev()) for x in nat]


@pytest.fixture(scope="module")
def long_reference(long_inputs):
    """Sampled oracle values, the same for every cp (the result is independent of
    how the sequence is split)."""
    w, nat, _ = long_inputs
    q, k, v, do = nat
    rows = _rows(w.T, 5)
    ref = {}
    for h in (0, 7):
        qh, kg, vg, doh = (W.as_f64(x[0, h]) for x in (q, k, v, do))
        ref[("o", h)] = OA.fwd_rows(qh, kg, vg, rows, w.scale)
        ref[("dq", h)] = OA.dq_rows(qh, kg, vg, doh, rows, w.scale)
        band = np.arange(w.T - 256, w.T)
        ref[("dkdv", h)] = OA.dkdv_rows(qh[None], kg, vg, doh[None], band, w.scale)
    return rows, ref


@pytest.mark.parametrize("cp_", [4, 8, 16, 32])
def test_long_context_T131072(long_inputs, long_reference, cp_):
    w0, nat, nat_dev = long_inputs
    w = w0.replace(cp=cp_)
    rows, ref = long_reference
    pos = torch.from_numpy(OL.positions(w.T, w.cp, w.layout)).to(dev())
    lay = [x[:, :, pos].contiguous() for x in nat_dev]
    got = run_ring(w, lay)
    slot_of = OL.layout_slots(w.T, w.cp, w.layout)
    tol = TOL[w.dtype]
    band = np.arange(w.T - 256, w.T)
    for h in (0, 7):
        ro, rl = ref[("o", h)]
        assert rel(_gather(got["o"], slot_of[rows], 0, h), ro) <= tol["o"]
        gl = W.as_f64(got["lse"][0, h, torch.from_numpy(slot_of[rows]).to(dev())])
        assert np.max(np.abs(gl - rl)) <= LSE_ABS_TOL[w.dtype]
        assert rel(_gather(got["dq"], slot_of[rows], 0, h), ref[("dq", h)]) <= tol["grad"]
        rdk, rdv = ref[("dkdv", h)]
        assert rel(_gather(got["dk"], slot_of[band], 0, h), rdk) <= tol["grad"]
        assert rel(_gather(got["dv"], slot_of[band], 0, h), rdv) <= tol["grad"]
    dk = got["dk"].float()
    assert float(dk.sum(dim=2).abs().max()) <= 1e-2 * float(dk.abs().sum(dim=2).max())
    dv_sum = got["dv"].float().sum(dim=2)
    do_sum = lay[3].float().sum(dim=2)
    assert float((dv_sum - do_sum).abs().max()) <= 2e-2 * float(do_sum.abs().max()) + 1.0
