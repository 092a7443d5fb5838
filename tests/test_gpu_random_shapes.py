"""GPU: a seeded sweep of random problem shapes through the ring forward and
backward, against the oracle.

The fixed parity cases cover the benchmark's workloads; this sweep draws further
combinations: batch rows 1-3, 1-3 K/V heads with 1-4 query heads each, cp 1-8,
both layouts, both head dimensions of the tensor-core path and odd ones of the
SIMT path, chunk halves from one 128-token tile to three, and token counts that
do not fill whole tiles (which the SIMT path takes).  Every draw is printed in the
test id, so a failure names its shape."""
import numpy as np
import pytest

import workloads as W
from gpu_helpers import assert_close, full_reference, ring_inputs, run_ring

pytestmark = pytest.mark.gpu


def _draws(n=18, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        layout = ["contiguous", "zigzag"][rng.integers(2)]
        cp = int(rng.choice([1, 2, 3, 4, 8]))
        halves = 2 * cp if layout == "zigzag" else cp
        tensor_core = rng.random() < 0.6
        if tensor_core:
            dtype, D = "bf16", int(rng.choice([64, 128]))
            T = halves * 128 * int(rng.integers(1, 4))
        else:
            dtype = ["bf16", "f32"][rng.integers(2)]
            D = int(rng.choice([8, 20, 32, 48, 64, 100, 128]))
            T = halves * int(rng.integers(3, 40))
        if T > 3072:
            continue
        B = int(rng.integers(1, 4))
        H_kv = int(rng.integers(1, 4))
        H_q = H_kv * int(rng.integers(1, 5))
        name = f"r{len(out)}_B{B}_H{H_q}x{H_kv}_T{T}_D{D}_cp{cp}_{layout}_{dtype}"
        out.append(W.Workload(name, B, H_q, H_kv, T, D, cp, layout, dtype,
                              seed=int(rng.integers(1000))))
    return out


@pytest.mark.parametrize("w", _draws(), ids=lambda w: w.name)
def test_random_shape_matches_oracle(w):
    nat, lay = ring_inputs(w)
    got = run_ring(w, lay)
    assert_close(w, got, full_reference(w, nat))
