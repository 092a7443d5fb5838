"""GPU: packed sequences (transformers pull request #50497: position ids restart
at every packed document and the mask is rebuilt for the documents) through
cpattn_ring_fwd_packed / cpattn_ring_bwd_packed, against the oracle's packed
attention.  Document boundaries fall inside tiles, on tile edges, inside zigzag
halves and between ranks; empty documents are included.  With one document per
row the packed calls give the plain ring's result up to the order of
accumulation (they visit the visible tiles in natural order, the ring in ring
order)."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import LSE_ABS_TOL, TOL, cp_mod, desc_of, dev, rel, ring_inputs, run_ring, to_nat
from oracle import attention as OA

pytestmark = pytest.mark.gpu


def _random_starts(rng, B, T, n_docs):
    rows = []
    for _ in range(B):
        cuts = np.sort(rng.integers(0, T + 1, n_docs - 1))
        rows.append(np.concatenate([[0], cuts, [T]]))
    return np.stack(rows).astype(np.int32)


CASES = [
    (W.Workload("pk_tc_T2048_cp4_zz_gqa4_B2", 2, 8, 2, 2048, 128, 4, "zigzag", "bf16"),
     np.array([[0, 300, 301, 1200, 1200, 2048], [0, 128, 1024, 1025, 1919, 2048]], np.int32)),
    (W.Workload("pk_tc_T1024_cp2_contig_D64", 1, 4, 4, 1024, 64, 2, "contiguous", "bf16"), 37),
    (W.Workload("pk_tc_T1024_cp4_zz_gqa3", 1, 3, 1, 1024, 128, 4, "zigzag", "bf16"), 5),
    # many short documents, a different cut in every row (work orders across rows)
    (W.Workload("pk_tc_T2048_cp4_contig_D64_B3", 3, 4, 2, 2048, 64, 4, "contiguous", "bf16"), 40),
    (W.Workload("pk_simt_f32_T96_cp3_zz", 2, 2, 1, 96, 20, 3, "zigzag", "f32"), 4),
    (W.Workload("pk_simt_bf16_T128_cp2_D32", 1, 2, 2, 128, 32, 2, "zigzag", "bf16"), 3),
]


def _run_packed(w, lay, starts_dev, n_docs):
    cp = cp_mod()
    ql, kl, vl, dol = lay
    desc = desc_of(w)
    ws = torch.empty(cp.cpattn_packed_workspace(desc), dtype=torch.uint8, device=dev())
    o = torch.empty_like(ql)
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev())
    cp.check(cp.cpattn_ring_fwd_packed(desc, starts_dev, n_docs, ql, kl, vl, o, lse, ws))
    dq, dk, dv = torch.empty_like(ql), torch.empty_like(kl), torch.empty_like(vl)
    cp.check(cp.cpattn_ring_bwd_packed(desc, starts_dev, n_docs, ql, kl, vl, o, lse, dol, dq, dk,
                                       dv, ws))
    cp.check(cp.cpattn_check())
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


@pytest.mark.parametrize("w,starts", CASES, ids=lambda x: getattr(x, "name", ""))
def test_packed_matches_oracle(w, starts):
    if isinstance(starts, int):
        starts = _random_starts(np.random.default_rng(w.T + starts), w.B, w.T, starts)
    n_docs = starts.shape[1] - 1
    nat, lay = ring_inputs(w)
    got = _run_packed(w, lay, torch.from_numpy(starts).to(dev()), n_docs)
    q, k, v, do = (W.as_f64(x) for x in nat)
    ro, rlse = OA.packed_attention_fwd(q, k, v, w.scale, starts)
    rdq, rdk, rdv = OA.packed_attention_bwd(q, k, v, do, w.scale, starts)
    tol = TOL[w.dtype]
    assert rel(to_nat(got["o"], w), ro) <= tol["o"]
    lse = to_nat(got["lse"].unsqueeze(-1), w)[..., 0]
    assert float(np.max(np.abs(lse - rlse))) <= LSE_ABS_TOL[w.dtype]
    for key, ref in (("dq", rdq), ("dk", rdk), ("dv", rdv)):
        assert rel(to_nat(got[key], w), ref) <= tol["grad"], key


@pytest.mark.parametrize("w", [CASES[0][0], CASES[3][0]], ids=lambda w: w.name)
def test_one_document_is_the_plain_ring(w):
    nat, lay = ring_inputs(w)
    starts = np.tile(np.array([[0, w.T]], np.int32), (w.B, 1))
    got = _run_packed(w, lay, torch.from_numpy(starts).to(dev()), 1)
    ref = run_ring(w, lay)
    # the same products over the same tiles, summed in another order
    lim = {"f32": 1e-5, "bf16": 1e-2}[w.dtype]
    for key in ("o", "dq", "dk", "dv"):
        e = rel(W.as_f64(got[key]), W.as_f64(ref[key]))
        assert e <= lim, (key, e)
    assert float((got["lse"] - ref["lse"]).abs().max()) <= LSE_ABS_TOL[w.dtype]


def test_packed_llama_T8192_eight_documents():
    """The packed benchmark's launch configuration: the LLaMA shape (B1, H_q 32 /
    H_kv 8, T 8192, D 128, cp 8 zigzag, bf16) with the seeded 8-document rows
    (documents of 20 to 4448 tokens).  The oracle computes the last K/V group in
    full (query heads 28-31 with K/V head 7); the other heads run the same tiles."""
    w = W.LLAMA
    starts = W.packed_starts(w, 8)
    nat, lay = ring_inputs(w)
    got = _run_packed(w, lay, torch.from_numpy(starts).to(dev()), 8)
    n_rep = w.H_q // w.H_kv
    tol = TOL[w.dtype]
    for g in (w.H_kv - 1,):
        hq = slice(g * n_rep, (g + 1) * n_rep)
        q, do = (W.as_f64(x[:, hq]) for x in (nat[0], nat[3]))
        k, v = (W.as_f64(x[:, g:g + 1]) for x in (nat[1], nat[2]))
        ro, rlse = OA.packed_attention_fwd(q, k, v, w.scale, starts)
        rdq, rdk, rdv = OA.packed_attention_bwd(q, k, v, do, w.scale, starts)
        assert rel(to_nat(got["o"][:, hq], w), ro) <= tol["o"], ("o", g)
        lse = to_nat(got["lse"][:, hq].unsqueeze(-1), w)[..., 0]
        assert float(np.max(np.abs(lse - rlse))) <= LSE_ABS_TOL[w.dtype], ("lse", g)
        assert rel(to_nat(got["dq"][:, hq], w), rdq) <= tol["grad"], ("dq", g)
        assert rel(to_nat(got["dk"][:, g:g + 1], w), rdk) <= tol["grad"], ("dk", g)
        assert rel(to_nat(got["dv"][:, g:g + 1], w), rdv) <= tol["grad"], ("dv", g)
