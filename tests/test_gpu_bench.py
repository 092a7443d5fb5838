"""GPU: bench.py as a user runs it, on small workloads (the GPT-2 shape, and the
LLaMA shape for the a2a layout), in the ring, all-gather and packed modes.  Checks
the JSON line's contract: the metric and its units, the roofline object of the
dominant kernel, the end-to-end object with its transfer byte counts, the clock
record, and a launch count that matches the per-kernel table."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "roofline", "gpu_launches", "clocks", "e2e", "kernels", "cpu_baseline"}
STEPS, WARMUP = 4, 3


def _bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", str(STEPS),
                        "--warmup", str(WARMUP), "--e2e-steps", "2", "--no-cpu-baseline", *args],
                       capture_output=True, text=True, timeout=240, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    return lines[0]


def _check_contract(out, tensor_kernel_prefix):
    assert REQUIRED <= set(out)
    assert out["unit"] == "TFLOP/s" and out["higher_is_better"] is True
    assert out["n_gpus"] == 1 and out["steps"] == STEPS and out["warmup"] == WARMUP
    assert out["value"] > 0 and out["ms_per_step"] > 0 and out["dtype"] == "bf16"
    assert out["cpu_baseline"] is None
    roof = out["roofline"]
    # the dominant kernel: a tensor-core attention kernel, or on small shapes an
    # HBM-bound one (the permutes), each against its own measured peak
    if roof["bound"] == "tensor":
        assert roof["unit"] == "TFLOP/s" and roof["kernel"].startswith(tensor_kernel_prefix)
    else:
        assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    # no kernel runs above twice the measured peak of its bound
    assert roof["frac"] < 2.0
    e2e = out["e2e"]
    assert e2e["unit"] == "TFLOP/s" and 0 < e2e["value"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    clocks = out["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clocks)
    # a dK/dV + dQ pair (the dQ kernel overlapping the end of the dK/dV kernel) is one
    # timing entry and two kernel launches
    launches = sum(k["launches"] * (2 if name.endswith("_dkdv_dq") else 1)
                   for name, k in out["kernels"].items())
    assert out["gpu_launches"] == launches > 0
    assert abs(sum(k["share"] for k in out["kernels"].values()) - 1.0) < 1e-6


def test_bench_ring_gpt2():
    out = _bench("--workload", "gpt2_small_T1024")
    _check_contract(out, "tc_")
    assert out["config"]["workload"] == "gpt2_small_T1024"
    # B4 H12 T1024 D64: q, k, v, dO in and o, dk, dv, dq (bf16) and the LSE (float32)
    # out, through one cpattn_ring_step_host call per step
    assert out["e2e"]["h2d_bytes_per_step"] == 4 * 4 * 12 * 1024 * 64 * 2
    assert out["e2e"]["d2h_bytes_per_step"] == 4 * 4 * 12 * 1024 * 64 * 2 + 4 * 12 * 1024 * 4
    assert out["e2e"]["transfers"].startswith("one cpattn_ring_step_host call")


def test_bench_allgather_gpt2():
    out = _bench("--workload", "gpt2_small_T1024", "--mode", "allgather")
    _check_contract(out, "tc_allgather_")
    assert out["config"]["mode"] == "all_gather"


def test_bench_packed_gpt2():
    out = _bench("--workload", "gpt2_small_T1024", "--packed-docs", "5")
    _check_contract(out, "tc_packed_")
    assert out["config"]["packed_docs"] == 5
    assert sum(out["config"]["doc_lengths"]) == 1024


def test_bench_a2a_ulysses():
    out = _bench("--workload", "llama_gqa_T8192_ulysses8")
    _check_contract(out, "tc_")
    assert any(name.startswith("layout_a2a") for name in out["kernels"])


def test_bench_p2p_ring_emulated_gpt2():
    """--mode p2p on one GPU: the per-step library calls of the ring across GPUs,
    all cp ranks in lockstep, replayed from a CUDA graph."""
    out = _bench("--workload", "gpt2_small_T1024_cp4_zigzag", "--mode", "p2p")
    assert REQUIRED - {"e2e"} <= set(out) and out["e2e"] is None
    assert out["unit"] == "TFLOP/s" and out["value"] > 0 and out["n_gpus"] == 1
    assert out["config"]["mode"] == "p2p" and out["config"]["graph"] is True
    names = set(out["kernels"])
    # each step's dQ kernel overlaps the end of its dK/dV kernel: timed as one unit
    assert {"tc_partial_fwd", "merge", "tc_partial_dkdv_dq"} <= names
    # cp^2 forward and backward steps per training step, over the min(steps, 5) steps
    # of the per-kernel timing pass
    assert out["kernels"]["tc_partial_fwd"]["launches"] == min(STEPS, 5) * 4 * 4
    assert out["kernels"]["tc_partial_dkdv_dq"]["launches"] == min(STEPS, 5) * 4 * 4
    assert out["roofline"]["frac"] < 2.0
