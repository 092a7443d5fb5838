"""Host-side checks of bench.py (no GPU): the reference arm's JSON contract, the
multi-rank launch (rank 0 alone prints), and the max-over-ranks reduction with
two gloo ranks on CPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
            "cpu_baseline", "e2e"}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(text):
    return [json.loads(x) for x in text.splitlines() if x.startswith("{")]


def test_reference_arm_json_contract():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--workload", "tiny_f32_T64"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    out = lines[0]
    assert REQUIRED <= set(out)
    assert out["impl"] == "reference" and out["value"] > 0 and out["unit"] == "TFLOP/s"
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["value"] == out["value"]
    assert out["config"]["workload"] == "tiny_f32_T64"


def test_reference_arm_under_two_ranks_prints_once():
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--workload", "tiny_f32_T64"],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert len(_json_lines(r.stdout)) == 1


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    got = bench.max_over_ranks(1.5 + rank, world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 2.5, 1: 2.5}


def test_tensor_peak_burst_or_sustained():
    sys.path.insert(0, ROOT)
    import bench
    pk = {"hbm_gbs": 1.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    burst, what = bench.tensor_peak(pk, "measured", 0.4)
    assert burst == 1900.0 and "burst" in what
    sus, what = bench.tensor_peak(pk, "measured", 1.5)
    assert sus == 1700.0 and "sustained" in what


def test_packed_pair_count_matches_the_document_mask():
    """The FLOP count of a packed step rests on the attended pairs: brute force
    over the oracle's document mask must give the closed form bench.py uses."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import workloads as W
    from oracle import attention as OA
    w = W.Workload("pairs_T512", 2, 3, 1, 512, 64, 2, "zigzag", "bf16")
    starts, pairs = bench.packed_documents(w, 6, seed=7)
    pos = np.arange(w.T)
    brute = sum(int(OA.packed_visible(pos, pos, starts[b]).sum()) for b in range(w.B)) * w.H_q
    assert pairs == brute
    assert starts.shape == (w.B, 7) and starts[0, 0] == 0 and starts[0, -1] == w.T
    assert np.all(np.diff(starts[0]) > 0)  # distinct cuts: no empty document


def test_permute_bytes_per_launch():
    """A step permutes q, k, v, dO and o, dk, dv, dq once each (one read, one write):
    the average launch moves the bytes of one query-sized and one K/V-sized tensor."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    w = W.LLAMA
    per_step = 2 * 2 * w.D * (4 * w.B * w.H_q * w.T + 4 * w.B * w.H_kv * w.T)
    bound, nbytes = bench.kernel_flops_or_bytes("layout_zigzag", w)
    assert bound == "hbm" and nbytes == per_step / 8


def test_hbm_roofline_arithmetic():
    sys.path.insert(0, ROOT)
    import bench
    pk = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    roof = bench.hbm_roofline("layout_zigzag", 1.0e8, 0.02, pk, "measured")
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert abs(roof["achieved"] - 5000.0) < 1e-6
    assert abs(roof["frac"] - 5000.0 / 6800.0) < 1e-12
    assert bench.hbm_roofline("x", None, 1.0, pk, "measured")["achieved"] is None


def test_source_digest_ignores_comments_only(tmp_path, monkeypatch):
    """The DRAM-traffic figures stay valid across comment edits and are voided by any
    change of the code (strings included)."""
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "blockwise_online_softmax_cpattn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = 'int f(int x) {  // doubles\n  return 2 * x;  /* one\n line */\n}\nconst char* s = "a // b";\n'
    (csrc / "k.cu").write_text(src)
    d0 = bench.source_digest()
    (csrc / "k.cu").write_text(src.replace("// doubles", "// twice x").replace("one\n line", "a\nb\nc"))
    assert bench.source_digest() == d0
    (csrc / "k.cu").write_text(src.replace("2 * x", "3 * x"))
    assert bench.source_digest() != d0
    (csrc / "k.cu").write_text(src.replace('"a // b"', '"a // c"'))
    assert bench.source_digest() != d0


def test_traffic_is_keyed_to_the_kernels_own_sources(tmp_path, monkeypatch):
    """A capture's DRAM bytes are reported while the kernel's translation unit is
    unchanged, stay valid across edits of other sources (the host-side C ABI), and
    are voided by a code change in the kernel's .cu file or a header it includes."""
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "blockwise_online_softmax_cpattn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for f, text in (("tc_fwd.cu", "int fwd() { return 1; }\n"), ("common.cuh", "#pragma once\n"),
                    ("kernels.h", "#pragma once\n"), ("api.cu", "int api() { return 2; }\n")):
        (csrc / f).write_text(text)
    digest = bench.source_digest(bench.KERNEL_SOURCES["tc_ring_fwd"])
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        f"# header\ntc_ring_fwd wl 123 {digest}\n")
    assert bench.traffic_for("tc_ring_fwd", "wl") == 123.0
    assert bench.traffic_for("tc_ring_fwd", "other") is None
    (csrc / "api.cu").write_text("int api() { return 3; }\n")
    assert bench.traffic_for("tc_ring_fwd", "wl") == 123.0
    (csrc / "common.cuh").write_text("#pragma once\nconstexpr int k = 1;\n")
    assert bench.traffic_for("tc_ring_fwd", "wl") is None


def test_traffic_of_a_unit_is_the_sum_over_its_kernels(tmp_path, monkeypatch):
    """The backward's dK/dV and dQ kernels, timed as one unit when the dQ kernel
    overlaps the end of the dK/dV kernel, report the sum of their captured DRAM
    bytes, and nothing once either capture is missing or stale."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    csrc = tmp_path / "blockwise_online_softmax_cpattn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for f, text in (("tc_bwd.cu", "int bwd() { return 1; }\n"), ("common.cuh", "#pragma once\n"),
                    ("kernels.h", "#pragma once\n")):
        (csrc / f).write_text(text)
    digest = bench.source_digest(bench.KERNEL_SOURCES["tc_bwd_dkdv"])
    path = tmp_path / "profiles" / "ncu_traffic.txt"
    path.write_text(f"tc_bwd_dkdv wl 100 {digest}\ntc_bwd_dq wl 23 {digest}\n")
    assert bench.traffic_for("tc_bwd_dkdv_dq", "wl") == 123.0
    path.write_text(f"tc_bwd_dkdv wl 100 {digest}\n")
    assert bench.traffic_for("tc_bwd_dkdv_dq", "wl") is None
    assert bench.kernel_flops_or_bytes("tc_bwd_dkdv_dq", W.LLAMA) == \
        ("tensor", 10.0 * W.LLAMA.D * W.LLAMA.attended_pairs)


def test_launch_count_counts_both_kernels_of_an_overlapped_pair():
    """The dK/dV + dQ pair is one timing entry but two kernel launches."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.kernels_in("tc_bwd_dkdv_dq") == 2
    assert bench.kernels_in("tc_partial_dkdv_dq") == 2
    assert bench.kernels_in("tc_ring_fwd") == 1 and bench.kernels_in("tc_bwd_dkdv") == 1
