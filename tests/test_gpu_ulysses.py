"""GPU: the full Ulysses mode (pull request "Feat: Context Parallel" #181, mode table
row "a2a": an AllToAll exchanges the sequence and head dimensions, attention runs
over the whole sequence, and the output layout is restored; tutorial "上下文并行",
section "Ulysses CP").  It is the hierarchical descriptor with a2a = cp: the ring
has a single rank.  Token shards (built with the oracle's own maps) go through
cpattn_layout(A2A_FWD), the forward and backward run on H/cp heads of the whole
sequence each, and the output returns to token shards through A2A_INV.  Every
output is compared with the oracle's full attention; the permutes bit-exactly with
the oracle's index maps."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import LSE_ABS_TOL, TOL, cp_mod, desc_of, dev, rel, run_ring
from oracle import attention as OA
from oracle import layouts as OL

pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("u_tc_T2048_cp4_zz_gqa2", 1, 8, 4, 2048, 128, 4, "zigzag", "bf16", a2a=4),
    W.Workload("u_tc_T1024_cp2_contig_B2", 2, 4, 2, 1024, 64, 2, "contiguous", "bf16", a2a=2),
    W.Workload("u_simt_f32_T64_cp4_zz", 1, 4, 4, 64, 16, 4, "zigzag", "f32", a2a=4),
]


def _heads_view(x, w, H):
    """Head-sharded [a2a][B][H/a2a][T][D] -> [B][H][T][D] (natural order: p2p = 1)."""
    return x.view(w.a2a, w.B, H // w.a2a, w.T, -1).permute(1, 0, 2, 3, 4).reshape(w.B, H, w.T, -1)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_ulysses_matches_oracle(w):
    cp = cp_mod()
    assert w.a2a == w.cp
    nat = W.draw_cast(w)
    desc = desc_of(w)
    H = [w.H_q, w.H_kv, w.H_kv, w.H_q]
    head_sharded = []
    for x, h in zip(nat, H):
        shards = torch.from_numpy(OL.token_shards(x.numpy() if x.dtype == torch.float32 else
                                                  x.view(torch.int16).numpy(), w.cp, w.layout))
        if x.dtype != torch.float32:
            shards = shards.view(torch.bfloat16)
        s_dev = shards.to(dev())
        out = torch.empty(w.a2a, w.B, h // w.a2a, w.T, w.D, dtype=x.dtype, device=dev())
        cp.check(cp.cpattn_layout(cp.A2A_FWD, desc, s_dev, out, h))
        # with one ring rank the token axis is the natural order
        assert torch.equal(_heads_view(out, w, h).cpu(), x)
        head_sharded.append(out.view(w.a2a * w.B, h // w.a2a, w.T, w.D))
    got = run_ring(w, head_sharded)
    # the output returns to token shards
    back = torch.empty(w.cp, w.B, w.T // w.cp, w.H_q, w.D, dtype=nat[0].dtype, device=dev())
    cp.check(cp.cpattn_layout(cp.A2A_INV, desc, got["o"], back, w.H_q))
    o_nat = _heads_view(got["o"], w, w.H_q).cpu()
    want = OL.token_shards(o_nat.float().numpy() if o_nat.dtype == torch.float32 else
                           o_nat.view(torch.int16).numpy(), w.cp, w.layout)
    got_back = back.cpu()
    got_back = got_back.numpy() if got_back.dtype == torch.float32 else got_back.view(torch.int16).numpy()
    assert np.array_equal(got_back, want)
    cp.check(cp.cpattn_check())
    q, k, v, do = (W.as_f64(x) for x in nat)
    ro, rlse = OA.attention_fwd(q, k, v, w.scale)
    rdq, rdk, rdv = OA.attention_bwd(q, k, v, do, w.scale)
    tol = TOL[w.dtype]
    assert rel(W.as_f64(_heads_view(got["o"], w, w.H_q)), ro) <= tol["o"]
    lse = _heads_view(got["lse"].unsqueeze(-1), w, w.H_q)[..., 0]
    assert float(np.max(np.abs(W.as_f64(lse) - rlse))) <= LSE_ABS_TOL[w.dtype]
    assert rel(W.as_f64(_heads_view(got["dq"], w, w.H_q)), rdq) <= tol["grad"]
    assert rel(W.as_f64(_heads_view(got["dk"], w, w.H_kv)), rdk) <= tol["grad"]
    assert rel(W.as_f64(_heads_view(got["dv"], w, w.H_kv)), rdv) <= tol["grad"]
