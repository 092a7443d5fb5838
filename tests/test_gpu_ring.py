"""GPU: cpattn_ring_fwd / cpattn_ring_bwd against the FP64 oracle, element by
element, on seeded inputs at sizes the oracle finishes in seconds.

Covers the tiny float32 case, the GPT-2-shaped bf16 workload over cp in {2, 4} x
{contiguous, zigzag} and its q x 4 stress seed, GQA with even and odd group
sizes, cp = 1 (plain causal attention), D = 64 and 128 on the tensor-core path,
and the SIMT path on ragged shapes (T not a multiple of the tile, odd D, chunk
halves off the 128-token grid, T = 1)."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import assert_close, dev, full_reference, ring_inputs, run_ring
from oracle import layouts as OL

pytestmark = pytest.mark.gpu

CASES = [
    W.TINY,
    *W.GPT2_VARIANTS,
    W.GPT2_STRESS,
    W.GPT2_STRESS.replace(cp=4, layout="zigzag", name="gpt2_q4_cp4_zigzag"),
    W.Workload("gqa4_T1024_D128_cp4_zz", 1, 8, 2, 1024, 128, 4, "zigzag", "bf16"),
    W.Workload("gqa3_T512_D64_cp2_contig", 2, 6, 2, 512, 64, 2, "contiguous", "bf16"),
    W.Workload("gqa3_T1024_D128_cp2_zz", 1, 3, 1, 1024, 128, 2, "zigzag", "bf16"),
    W.Workload("mha_T512_D128_cp1", 1, 2, 2, 512, 128, 1, "contiguous", "bf16"),
    W.Workload("mqa_T768_D64_cp3_contig", 1, 4, 1, 768, 64, 3, "contiguous", "bf16"),
    W.Workload("gqa2_T2048_D128_cp8_zz", 1, 4, 2, 2048, 128, 8, "zigzag", "bf16"),
    # SIMT path: chunk halves off the 128-token grid, odd D, ragged sizes
    W.Workload("simt_bf16_T1152_cp3_zz", 1, 4, 2, 1152, 64, 3, "zigzag", "bf16"),
    W.Workload("simt_bf16_D96", 1, 2, 1, 256, 96, 2, "zigzag", "bf16"),
    W.Workload("simt_f32_T100_cp5_D24", 2, 3, 1, 100, 24, 5, "contiguous", "f32"),
    W.Workload("simt_f32_T512_cp4_zz", 1, 4, 2, 512, 64, 4, "zigzag", "f32"),
    W.Workload("simt_f32_T1", 1, 2, 2, 1, 8, 1, "contiguous", "f32"),
    W.Workload("simt_f32_T6_cp3_zz", 1, 2, 1, 6, 8, 3, "zigzag", "f32"),
    W.Workload("simt_f32_D128", 1, 2, 2, 96, 128, 2, "zigzag", "f32"),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_ring_fwd_bwd_matches_oracle(w):
    nat, lay = ring_inputs(w)
    got = run_ring(w, lay)
    ref = full_reference(w, nat)
    errs = assert_close(w, got, ref)
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("w", [W.GPT2_VARIANTS[3], CASES[5]], ids=lambda w: w.name)
def test_ring_is_deterministic(w):
    """No atomics anywhere: two runs give identical bits."""
    _, lay = ring_inputs(w)
    a = run_ring(w, lay)
    b = run_ring(w, lay)
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_rows_of_probabilities_sum_to_one_through_v_ones():
    """With every value row equal to 1, O must be exactly 1 up to bf16 rounding of
    P (sum of normalised probabilities), on the tensor-core path."""
    w = W.Workload("ones", 1, 4, 2, 1024, 128, 4, "zigzag", "bf16")
    nat, lay = ring_inputs(w)
    lay[2].fill_(1.0)
    got = run_ring(w, lay, bwd=False)
    o = got["o"].float().cpu().numpy()
    assert np.max(np.abs(o - 1.0)) < 1e-2


def test_running_max_jumps_after_the_first_tile():
    """Keys at natural positions [0, 256) scaled by 8: rank 1's query rows
    (positions 256-767, cp 2 zigzag) visit their own chunk first, with modest scores,
    and then rank 0's chunk, whose scores are larger by far more than 2^8 in the
    exponent.  The forward then raises the running max and forms those tiles again,
    across whole warps; the results must still match the oracle."""
    w = W.Workload("jump_T1024_D128_cp2_zz", 1, 4, 2, 1024, 128, 2, "zigzag", "bf16")
    q, k, v, do = W.draw_cast(w)
    k = k.clone()
    k[:, :, :256] *= 8  # exact in bf16
    nat = (q, k, v, do)
    pos = torch.from_numpy(OL.positions(w.T, w.cp // w.a2a, w.layout))
    lay = [x[:, :, pos].contiguous().to(dev()) for x in nat]
    got = run_ring(w, lay)
    assert_close(w, got, full_reference(w, nat))
