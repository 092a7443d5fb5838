#!/usr/bin/env python3
"""Benchmark of causal ring attention (forward + backward) on GB300.

One step = the whole hot path over one batch of synthetic input already in HBM:
  layout permute of q, k, v, dO (natural -> zigzag layout order, one
  cpattn_layout_batch call; the all-to-all re-layout for the hierarchical a2a x p2p
  workload) -> cpattn_ring_fwd -> cpattn_ring_bwd -> inverse permute of o, dq, dk,
  dv (one call).
FLOPs counted: 4*D per attended (q, k) pair forward, 10*D backward (attended
pairs = B * H_q * T (T + 1) / 2; masked work inside diagonal tiles is not
counted).  `value` is TFLOP/s over all GPUs; L2 is flushed (256 MiB write)
before every timed step.

--impl reference times the FP64 CPU oracle (the only reference there is) on the
host cores, each step a bounded sample of the same workload.

--packed-docs N times the ring over packed sequences instead: every row holds N
documents of seeded random lengths (causal attention inside each document); the
FLOPs count the pairs the packed mask attends.

--mode hbm times the HBM-bound kernels alone, one launch at a time with L2 flushed
before each: the (O, LSE) merge at the LLaMA and Qwen3 ring-step sizes, the a2a
head<->sequence re-layout at the Qwen3 size, and the zigzag chunk copies at the
LLaMA size; GB/s of algorithmic bytes against the measured copy bandwidth.

--mode p2p times the ring of per-step library calls (cpattn_partial_fwd,
cpattn_merge, cpattn_partial_bwd) that the point-to-point ring across GPUs runs:
under torch.distributed.run with N processes, the real ring over N = cp ranks (one
per GPU, K/V exchanged by NCCL); in one process, all cp ranks of the workload in
lockstep on one GPU, replayed from a CUDA graph (the step is hundreds of small
launches).  Same FLOP count as the ring.

--mode allgather times the all-gather mode instead (pull request #181, mode table
row "all_gather"): one step = cpattn_allgather_fwd and cpattn_allgather_bwd for
every emulated rank, with the layout-order q, k, v and each rank's dO rows already
in HBM; the ranks' K/V gradient shares are summed in float32 (the mode's
ReduceScatter).  Same FLOP count as the ring.

Launch: python bench.py [--gpus N --steps K --warmup W] [--impl cpattn|reference]
        [--workload NAME]; for N > 1 under torch.distributed.run, one independent
replica of the workload per GPU (no data exchange; weak scaling).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "causal ring-attention fwd+bwd TFLOP/s and % of BF16 tensor peak (1 GB300)"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = W.LLAMA.name
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cpattn", choices=["cpattn", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.ALL))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", default="ring", choices=["ring", "allgather", "hbm", "p2p"])
    ap.add_argument("--no-graph", action="store_true",
                    help="--mode p2p on one GPU: launch the steps eagerly instead of "
                         "replaying them from a CUDA graph")
    ap.add_argument("--packed-docs", type=int, default=0,
                    help="ring mode over packed sequences: this many documents per row, "
                         "seeded random lengths (0: one sequence per row)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(pk, src_pk, timed_s):
    """The bf16 denominator for a timed region of `timed_s` seconds: the burst figure
    when the region is shorter than a second, else the sustained one (a GEMM loop
    held for seconds under the power cap), as the peaks file defines them."""
    if timed_s >= 1.0:
        return pk["bf16_tflops_sustained"], f"{src_pk} bf16 dense sustained (cuBLAS, seconds long)"
    return pk["bf16_tflops"], f"{src_pk} bf16 dense burst (cuBLAS)"


def hbm_roofline(kernel, nbytes, avg_ms, pk, src_pk):
    """Roofline object of an HBM-bound dominant kernel: algorithmic bytes per launch
    over its average launch time, against the measured copy bandwidth."""
    if nbytes is None:
        return {"bound": "hbm", "kernel": kernel, "achieved": None, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": None}
    achieved = nbytes / (avg_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
            "peak_source": f"{src_pk} copy bandwidth", "work_per_launch": nbytes,
            "avg_launch_ms": avg_ms}


def config_of(w, extra=None):
    cfg = {"workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "T": w.T, "D": w.D,
           "cp": w.cp, "a2a": w.a2a, "layout": w.layout, "causal": True, "seed": w.seed,
           "inputs": f"i.i.d. N(0,1), seeded torch CPU generator, cast to {w.dtype}",
           "flops_per_step": w.fwd_flops + w.bwd_flops}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.path = os.path.join("/tmp", f"cpattn_clocks_{os.getpid()}.csv")
        self.proc = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(1.0)  # first samples come after nvidia-smi starts up
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        mhz, mx, reasons, n_all = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                n_all += 1
                if not (t0 - 0.06 <= ts <= t1 + 0.06):
                    continue
                try:
                    mhz.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for name, val in zip(names, parts[4:8]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
def kernel_flops_or_bytes(name, w, pairs=None):
    """Algorithmic work of one launch of a library kernel on this workload (pairs:
    the attended pairs when they differ from plain causal, e.g. packed documents)."""
    pairs = w.attended_pairs if pairs is None else pairs
    elt = 2 if w.dtype == "bf16" else 4
    rows_q = w.B * w.H_q * w.T
    rows_kv = w.B * w.H_kv * w.T
    if name in ("tc_ring_fwd", "simt_ring_fwd", "tc_packed_fwd"):
        return "tensor", 4.0 * w.D * pairs
    if name in ("tc_bwd_dkdv", "simt_bwd_dkdv", "tc_packed_dkdv"):  # S, dP recomputed + dV, dK
        return "tensor", 8.0 * w.D * pairs
    if name in ("tc_bwd_dq", "simt_bwd_dq", "tc_packed_dq"):        # the dQ product only
        return "tensor", 2.0 * w.D * pairs
    # the dK/dV kernel and the dQ kernel that overlaps its end, timed as one unit
    if name in ("tc_bwd_dkdv_dq", "tc_packed_dkdv_dq"):
        return "tensor", 10.0 * w.D * pairs
    # all-gather mode: one launch covers one rank's rows (1/cp of the pairs on average)
    # one ring step (rank, chunk): 1 / cp^2 of the pairs on average
    if name == "tc_partial_fwd":
        return "tensor", 4.0 * w.D * pairs / w.cp ** 2
    if name == "tc_partial_dkdv":
        return "tensor", 8.0 * w.D * pairs / w.cp ** 2
    if name == "tc_partial_dq":
        return "tensor", 2.0 * w.D * pairs / w.cp ** 2
    if name == "tc_partial_dkdv_dq":
        return "tensor", 10.0 * w.D * pairs / w.cp ** 2
    if name == "tc_allgather_fwd":
        return "tensor", 4.0 * w.D * pairs / w.cp
    if name == "tc_allgather_dkdv":
        return "tensor", 8.0 * w.D * pairs / w.cp
    if name == "tc_allgather_dq":
        return "tensor", 2.0 * w.D * pairs / w.cp
    if name == "tc_allgather_dkdv_dq":
        return "tensor", 10.0 * w.D * pairs / w.cp
    if name == "bwd_prepass":
        return "hbm", 2.0 * rows_q * w.D * elt + 12.0 * rows_q
    if name in ("layout_zigzag_batch", "layout_a2a_batch"):
        # one launch permutes a step's four inputs (q, k, v, dO) or its four outputs
        # (o, dk, dv, dq): each read once and written once
        return "hbm", 2.0 * (2 * rows_q + 2 * rows_kv) * w.D * elt
    if name.startswith("layout"):
        # a step permutes q, k, v, dO and o, dk, dv, dq (each read once and written
        # once): the average launch moves (rows_q + rows_kv) rows each way
        return "hbm", 2.0 * (rows_q + rows_kv) * w.D * elt / 2.0
    return "hbm", None


_CODE_TOKEN = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"', re.S)


# The translation unit each kernel is compiled from: its .cu file and the headers it
# includes.  A capture stays valid while these are unchanged (other files, such as
# the host-side C ABI in api.cu, cannot change the kernel's code).
KERNEL_SOURCES = {
    "tc_ring_fwd": ("tc_fwd.cu", "common.cuh", "kernels.h"),
    "tc_bwd_dkdv": ("tc_bwd.cu", "common.cuh", "kernels.h"),
    "tc_bwd_dq": ("tc_bwd.cu", "common.cuh", "kernels.h"),
}
# units timed as one span: the sum of their kernels' traffic
KERNEL_UNITS = {"tc_bwd_dkdv_dq": ("tc_bwd_dkdv", "tc_bwd_dq")}


PAIR_NOTE = ("the dK/dV kernel and the dQ kernel launched as its programmatic dependent, "
             "which overlaps its end: one event pair around both, 10 D FLOPs per attended "
             "pair (8 D dK/dV + 2 D dQ)")


def kernels_in(entry):
    """Kernel launches behind one entry of the library's timing table: the backward's
    dK/dV + dQ pair (the dQ kernel overlapping the end of the dK/dV kernel, timed as
    one span) is two."""
    return 2 if entry.endswith("_dkdv_dq") else 1


def source_digest(files=None):
    """Hash of library sources (all of csrc/, or the given files of it) with comments,
    trailing blanks and empty lines removed, so that only a change of the code itself
    voids a capture."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "blockwise_online_softmax_cpattn_gb300", "csrc")
    for f in sorted(os.listdir(csrc) if files is None else files):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        code = _CODE_TOKEN.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
        lines = [ln.rstrip() for ln in code.splitlines()]
        h.update(f.encode() + b"\0" + "\n".join(ln for ln in lines if ln).encode() + b"\0")
    return h.hexdigest()[:16]


def traffic_for(kernel, workload):
    """dram bytes per launch from the committed ncu summary, if the sources of the
    kernel's translation unit are unchanged since the capture (for a unit of several
    kernels, the sum over them, if every one is current)."""
    if kernel in KERNEL_UNITS:
        parts = [traffic_for(k, workload) for k in KERNEL_UNITS[kernel]]
        return None if any(x is None for x in parts) else sum(parts)
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    digest = source_digest(KERNEL_SOURCES[kernel])
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload:
                return float(parts[2]) if parts[3] == digest else None
    return None


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank value over all ranks (the slowest replica sets the time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def packed_documents(w, n_docs, seed=1234):
    """Seeded document starts [B][n_docs + 1] for a packed workload (every row the same
    cut points: n_docs - 1 distinct random cuts) and the pairs the packed mask attends."""
    starts = W.packed_starts(w, n_docs, seed)
    lens = np.diff(starts[0]).astype(np.float64)
    pairs = w.B * w.H_q * float(np.sum(lens * (lens + 1) / 2))
    return starts, pairs


def run_cpattn(args, rank, world):
    import torch
    import blockwise_online_softmax_cpattn_gb300 as cp

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.ALL[args.workload]
    stream = torch.cuda.current_stream()
    desc = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype, a2a=w.a2a)
    dt = W.torch_dtype(w)
    nat_host = [x.pin_memory() for x in W.draw_cast(w)]             # natural order
    q, k, v, do = [x.to(dev) for x in nat_host]
    H = [w.H_q, w.H_kv, w.H_kv, w.H_q]
    if w.a2a > 1:
        # inputs as the cp ranks' token shards [cp][B][T/cp][H][D]: prepared once,
        # outside the timed region (zigzag over cp, then rank-major transpose)
        d_cp = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype)
        shards = []
        for x, h in zip((q, k, v, do), H):
            y = torch.empty_like(x)
            cp.check(cp.cpattn_layout(cp.ZIGZAG_FWD, d_cp, x, y, h))
            shards.append(y.view(w.B, h, w.cp, w.T // w.cp, w.D).permute(2, 0, 3, 1, 4)
                          .contiguous())
        src = shards
        fwd_perm, inv_perm = cp.A2A_FWD, cp.A2A_INV
    else:
        src = [q, k, v, do]
        fwd_perm, inv_perm = cp.ZIGZAG_FWD, cp.ZIGZAG_INV
    lay = [torch.empty(w.B, h, w.T, w.D, dtype=dt, device=dev) for h in H]
    o = torch.empty_like(lay[0])
    lse = torch.empty(w.B, w.H_q, w.T, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(lay[0]), torch.empty_like(lay[1]), torch.empty_like(lay[2])
    outs = [torch.empty_like(s) for s in (src[0], src[1], src[2], src[0])]  # o, dk, dv, dq
    packed = args.packed_docs > 0
    if packed:
        if w.a2a != 1:
            raise SystemExit("--packed-docs takes a plain ring workload (a2a = 1)")
        starts_np, doc_pairs = packed_documents(w, args.packed_docs)
        starts = torch.from_numpy(starts_np).to(dev)
        ws = torch.empty(cp.cpattn_packed_workspace(desc), dtype=torch.uint8, device=dev)
    else:
        ws = torch.empty(cp.cpattn_ring_bwd_workspace(desc), dtype=torch.uint8, device=dev)

    def ring_fwd(q_, k_, v_, o_, lse_, d=desc):
        if packed:
            return cp.cpattn_ring_fwd_packed(d, starts, args.packed_docs, q_, k_, v_, o_, lse_, ws)
        return cp.cpattn_ring_fwd(d, q_, k_, v_, o_, lse_)

    def ring_bwd(q_, k_, v_, o_, lse_, do_, dq_, dk_, dv_, d=desc):
        if packed:
            return cp.cpattn_ring_bwd_packed(d, starts, args.packed_docs, q_, k_, v_, o_, lse_,
                                             do_, dq_, dk_, dv_, ws)
        return cp.cpattn_ring_bwd(d, q_, k_, v_, o_, lse_, do_, dq_, dk_, dv_, ws)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    H_out = [w.H_q, w.H_kv, w.H_kv, w.H_q]  # o, dk, dv, dq

    def step():
        cp.check(cp.cpattn_layout_batch(fwd_perm, desc, src, lay, H))
        cp.check(ring_fwd(lay[0], lay[1], lay[2], o, lse))
        cp.check(ring_bwd(lay[0], lay[1], lay[2], o, lse, lay[3], dq, dk, dv))
        cp.check(cp.cpattn_layout_batch(inv_perm, desc, [o, dk, dv, dq], outs, H_out))

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    cp.check(cp.cpattn_check())

    # ---- device-resident timed region
    sampler = ClockSampler(local)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    clocks = sampler.stop(t0, t1)
    cp.check(cp.cpattn_check())
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, dev)
    # 14 D FLOPs per attended pair (4 D forward, 10 D backward)
    flops = 14.0 * w.D * doc_pairs if packed else w.fwd_flops + w.bwd_flops
    value = world * flops / (ms * 1e-3) / 1e12

    # ---- per-kernel durations (events on the launch stream, same steps)
    cp.cpattn_timing_reset()
    cp.cpattn_timing_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        step()
    cp.check(cp.cpattn_timing_collect())
    cp.cpattn_timing_enable(False)
    table = cp.cpattn_timing_table()
    cp.cpattn_timing_reset()
    launches_per_step = sum(n * kernels_in(k) for k, (_, n) in table.items()) / args.steps
    kernels = {name: {"avg_ms": tot / n, "launches": n, "share": tot / sum(t for t, _ in table.values())}
               for name, (tot, n) in table.items()}
    dom = max(table, key=lambda n: table[n][0])
    pk, src_pk = peaks()
    bound, work = kernel_flops_or_bytes(dom, w, doc_pairs if packed else None)
    avg_ms = table[dom][0] / table[dom][1]
    peak, peak_what = tensor_peak(pk, src_pk, t1 - t0)
    if bound == "tensor":
        achieved = work / (avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_what,
                "work_per_launch": work, "avg_launch_ms": avg_ms}
        if kernels_in(dom) == 2:
            roof["unit_of"] = PAIR_NOTE
    else:
        roof = hbm_roofline(dom, work, avg_ms, pk, src_pk)
    traffic = None if packed else traffic_for(dom, w.name)
    roof["traffic"] = traffic

    # ---- end to end through the C ABI with host buffers
    host_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in outs]
    # the host holds what the library takes: natural-order tensors for the ring, the
    # ranks' token shards for the a2a layout (prepared once, here)
    up_host = nat_host if w.a2a == 1 else [x.cpu().pin_memory() for x in src]
    h2d = sum(x.numel() * x.element_size() for x in up_host)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_e2e)]
    side_in, side_out = torch.cuda.Stream(), torch.cuda.Stream()
    e_do, e_o = torch.cuda.Event(), torch.cuda.Event()

    def e2e_step_overlapped(a_ev):
        # One step through host buffers with the transfers a caller can overlap, all
        # between the step's two events: dO uploads on a side stream while the
        # forward runs, o downloads on another while the backward runs; q, k, v are
        # uploaded and dq, dk, dv downloaded on the step's own stream.
        side_in.wait_event(a_ev)
        side_out.wait_event(a_ev)
        with torch.cuda.stream(side_in):
            src[3].copy_(up_host[3], non_blocking=True)
            e_do.record(side_in)
        for dst_, hsrc in zip(src[:3], up_host[:3]):
            dst_.copy_(hsrc, non_blocking=True)
        cp.check(cp.cpattn_layout_batch(fwd_perm, desc, src[:3], lay[:3], H[:3]))
        cp.check(ring_fwd(lay[0], lay[1], lay[2], o, lse))
        cp.check(cp.cpattn_layout(inv_perm, desc, o, outs[0], w.H_q))
        e_o.record(stream)
        side_out.wait_event(e_o)
        with torch.cuda.stream(side_out):
            host_out[0].copy_(outs[0], non_blocking=True)
        stream.wait_event(e_do)
        cp.check(cp.cpattn_layout(fwd_perm, desc, src[3], lay[3], H[3]))
        cp.check(ring_bwd(lay[0], lay[1], lay[2], o, lse, lay[3], dq, dk, dv))
        cp.check(cp.cpattn_layout_batch(inv_perm, desc, [dk, dv, dq], outs[1:], H_out[1:]))
        for hdst, dsrc in zip(host_out[1:], outs[1:]):
            hdst.copy_(dsrc, non_blocking=True)
        stream.wait_stream(side_out)  # o's download is part of the step

    # The plain ring (not packed): one cpattn_ring_step_host call per step, the
    # library's own overlap of the transfers with the compute (independent halves of
    # the problem, two copy streams); its host outputs are natural order, as outs.
    host_step = not packed and w.a2a == 1
    if host_step:
        ws_step = torch.empty(cp.cpattn_ring_step_host_workspace(desc), dtype=torch.uint8,
                              device=dev)
        h_lse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        d2h += h_lse.numel() * 4

    def e2e_step_library(a_ev):
        cp.check(cp.cpattn_ring_step_host(desc, *up_host, host_out[0], h_lse, host_out[3],
                                          host_out[1], host_out[2], ws_step))

    e2e_step = e2e_step_library if host_step else e2e_step_overlapped
    # untimed first calls: the library creates its copy streams on the first one
    for _ in range(max(1, min(3, args.warmup))):
        a_w = torch.cuda.Event()
        a_w.record(stream)
        e2e_step(a_w)
    torch.cuda.synchronize()
    for a, b in ev2:
        flush.zero_()
        a.record(stream)
        e2e_step(a)
        b.record(stream)
    torch.cuda.synchronize()
    cp.check(cp.cpattn_check())
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev2), world, dev)
    # the end-to-end outputs are the device step's, bit for bit (the same calls on the
    # same inputs; in halves, independent problems with the same per-tile arithmetic)
    e2e_out = [x.clone() for x in host_out]
    step()
    torch.cuda.synchronize()
    if not all(torch.equal(a_, b_.cpu()) for a_, b_ in zip(e2e_out, outs)):
        raise RuntimeError("end-to-end outputs differ from the device-resident step's")
    if host_step:
        d_lse = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, 1, w.cp, w.layout, "f32")
        lse_nat = torch.empty_like(lse)
        cp.check(cp.cpattn_layout(inv_perm, d_lse, lse, lse_nat, w.H_q))
        if not torch.equal(h_lse, lse_nat.cpu()):
            raise RuntimeError("end-to-end LSE differs from the device-resident step's")
    e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "transfers": ("one cpattn_ring_step_host call per step on pinned host buffers: the "
                         "library runs the problem as independent groups (forward quarters, "
                         "backward halves) and overlaps their uploads and downloads with "
                         "other groups' compute on its own copy streams, all inside each "
                         "step's events"
                         if host_step else
                         "pinned host buffers (the ranks' token shards for the a2a layout); dO "
                         "upload overlaps the forward and o download overlaps the backward on "
                         "side streams inside each step's events")}

    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
           "config": config_of(w, {
               "parallelism": "replicas" if world > 1 else "single GPU, cp ranks emulated in-kernel",
               "l2": "flushed before every timed step (256 MiB device write, outside the events)",
               "step": ("a2a permute" if w.a2a > 1 else "zigzag permute")
               + " q,k,v,dO -> ring fwd -> ring bwd -> inverse permute o,dq,dk,dv",
               "pct_of_bf16_peak": value / world / peak,
               "peak_source": peak_what,
               **({"packed_docs": args.packed_docs,
                   "doc_lengths": [int(x) for x in np.diff(starts_np[0])],
                   "attended_pairs": doc_pairs, "flops_per_step": 14.0 * w.D * doc_pairs}
                  if packed else {})}),
           "roofline": roof, "gpu_launches": int(round(launches_per_step * args.steps)),
           "clocks": clocks, "e2e": e2e, "kernels": kernels}
    return out


def run_allgather(args, rank, world):
    """The all-gather mode: every emulated rank's forward and backward per step."""
    import torch
    import blockwise_online_softmax_cpattn_gb300 as cp

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.ALL[args.workload]
    if w.a2a != 1:
        raise SystemExit("--mode allgather takes a plain ring workload (a2a = 1)")
    stream = torch.cuda.current_stream()
    desc = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype)
    dt = W.torch_dtype(w)
    c = w.T // w.cp
    nat = W.draw_cast(w)
    # inputs as the ranks hold them: the gathered q, k, v in layout order, and each
    # rank's own dO rows; prepared once, outside the timed region
    H = [w.H_q, w.H_kv, w.H_kv, w.H_q]
    lay = []
    for x, h in zip(nat, H):
        y = torch.empty(w.B, h, w.T, w.D, dtype=dt, device=dev)
        cp.check(cp.cpattn_layout(cp.ZIGZAG_FWD, desc, x.to(dev), y, h))
        lay.append(y)
    ql, kl, vl, dol = lay
    do_r = [dol[:, :, r * c:(r + 1) * c].contiguous() for r in range(w.cp)]
    o_r = [torch.empty(w.B, w.H_q, c, w.D, dtype=dt, device=dev) for _ in range(w.cp)]
    lse_r = [torch.empty(w.B, w.H_q, c, dtype=torch.float32, device=dev) for _ in range(w.cp)]
    dq_r = [torch.empty_like(o) for o in o_r]
    dk_sum = torch.empty(w.B, w.H_kv, w.T, w.D, dtype=torch.float32, device=dev)
    dv_sum = torch.empty_like(dk_sum)
    ws = torch.empty(cp.cpattn_allgather_bwd_workspace(desc), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        for r in range(w.cp):
            cp.check(cp.cpattn_allgather_fwd(desc, r, ql, kl, vl, o_r[r], lse_r[r]))
        for r in range(w.cp):
            cp.check(cp.cpattn_allgather_bwd(desc, r, ql, kl, vl, o_r[r], lse_r[r], do_r[r],
                                             dq_r[r], dk_sum, dv_sum, r > 0, ws))

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    cp.check(cp.cpattn_check())
    sampler = ClockSampler(local)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    clocks = sampler.stop(t0, t1)
    cp.check(cp.cpattn_check())
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, dev)
    flops = w.fwd_flops + w.bwd_flops
    value = world * flops / (ms * 1e-3) / 1e12

    cp.cpattn_timing_reset()
    cp.cpattn_timing_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        step()
    cp.check(cp.cpattn_timing_collect())
    cp.cpattn_timing_enable(False)
    table = cp.cpattn_timing_table()
    cp.cpattn_timing_reset()
    launches_per_step = sum(n * kernels_in(k) for k, (_, n) in table.items()) / args.steps
    kernels = {name: {"avg_ms": tot / n, "launches": n, "share": tot / sum(t for t, _ in table.values())}
               for name, (tot, n) in table.items()}
    dom = max(table, key=lambda n: table[n][0])
    pk, src_pk = peaks()
    bound, work = kernel_flops_or_bytes(dom, w)
    avg_ms = table[dom][0] / table[dom][1]
    peak, peak_what = tensor_peak(pk, src_pk, t1 - t0)
    if bound == "tensor":
        achieved = work / (avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_what,
                "work_per_launch": work, "avg_launch_ms": avg_ms,
                "note": "work per launch is the average over the ranks (pairs / cp)"}
        if kernels_in(dom) == 2:
            roof["unit_of"] = PAIR_NOTE
    else:
        roof = hbm_roofline(dom, work, avg_ms, pk, src_pk)
    roof["traffic"] = None

    # end to end: the ranks' inputs uploaded from pinned host memory and their
    # outputs (o, dq rows, float32 dK/dV sums) read back, inside each step's events
    h_in = [x.cpu().pin_memory() for x in (ql, kl, vl)] + [x.cpu().pin_memory() for x in do_r]
    d_in = [ql, kl, vl] + do_r
    d_out = o_r + dq_r + [dk_sum, dv_sum]
    h_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in d_out]
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = sum(x.numel() * x.element_size() for x in h_out)
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_e2e)]
    side_in, side_out = torch.cuda.Stream(), torch.cuda.Stream()
    e_do = torch.cuda.Event()
    e_o = [torch.cuda.Event() for _ in range(w.cp)]
    e_dq = [torch.cuda.Event() for _ in range(w.cp)]
    h_o, h_dq, h_sums = h_out[:w.cp], h_out[w.cp:2 * w.cp], h_out[2 * w.cp:]

    def e2e_step(a_ev):
        # q, k, v upload on the step's stream; the ranks' dO uploads on a side stream
        # while the forwards run; each rank's o downloads behind its forward and its
        # dQ rows behind its backward on another side stream; the float32 K/V gradient
        # sums download after the last backward.  All between the step's two events.
        side_in.wait_event(a_ev)
        side_out.wait_event(a_ev)
        with torch.cuda.stream(side_in):
            for d_, h_ in zip(d_in[3:], h_in[3:]):
                d_.copy_(h_, non_blocking=True)
            e_do.record(side_in)
        for d_, h_ in zip(d_in[:3], h_in[:3]):
            d_.copy_(h_, non_blocking=True)
        for r in range(w.cp):
            cp.check(cp.cpattn_allgather_fwd(desc, r, ql, kl, vl, o_r[r], lse_r[r]))
            e_o[r].record(stream)
            side_out.wait_event(e_o[r])
            with torch.cuda.stream(side_out):
                h_o[r].copy_(o_r[r], non_blocking=True)
        stream.wait_event(e_do)
        for r in range(w.cp):
            cp.check(cp.cpattn_allgather_bwd(desc, r, ql, kl, vl, o_r[r], lse_r[r], do_r[r],
                                             dq_r[r], dk_sum, dv_sum, r > 0, ws))
            e_dq[r].record(stream)
            side_out.wait_event(e_dq[r])
            with torch.cuda.stream(side_out):
                h_dq[r].copy_(dq_r[r], non_blocking=True)
        for h_, d_ in zip(h_sums, (dk_sum, dv_sum)):
            h_.copy_(d_, non_blocking=True)
        stream.wait_stream(side_out)  # every download is part of the step

    for _ in range(max(1, min(3, args.warmup))):  # untimed first calls
        a_w = torch.cuda.Event()
        a_w.record(stream)
        e2e_step(a_w)
    torch.cuda.synchronize()
    for a, b in ev2:
        flush.zero_()
        a.record(stream)
        e2e_step(a)
        b.record(stream)
    torch.cuda.synchronize()
    cp.check(cp.cpattn_check())
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev2), world, dev)
    # the end-to-end outputs are the device-resident step's, bit for bit
    e2e_out = [x.clone() for x in h_out]
    step()
    torch.cuda.synchronize()
    if not all(torch.equal(a_, b_.cpu()) for a_, b_ in zip(e2e_out, d_out)):
        raise RuntimeError("end-to-end outputs differ from the device-resident step's")
    e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "transfers": "pinned host buffers; the ranks' dO uploads overlap the forwards, "
                        "each rank's o and dQ rows download behind its own launch, on side "
                        "streams inside each step's events"}
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": config_of(w, {
                "mode": "all_gather",
                "parallelism": "replicas" if world > 1 else "single GPU, cp ranks emulated",
                "l2": "flushed before every timed step (256 MiB device write, outside the events)",
                "step": "for every rank: cpattn_allgather_fwd, then for every rank: "
                        "cpattn_allgather_bwd (K/V gradient shares summed in float32)",
                "pct_of_bf16_peak": value / world / peak, "peak_source": peak_what}),
            "roofline": roof, "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clocks, "e2e": e2e, "kernels": kernels}


def run_p2p(args, rank, world):
    """The point-to-point ring of per-step library calls: the real ring over the
    world's ranks (world = cp), or all cp ranks emulated in lockstep on one GPU."""
    import torch
    import blockwise_online_softmax_cpattn_gb300 as cp
    from blockwise_online_softmax_cpattn_gb300 import ring as R

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.ALL[args.workload]
    if w.a2a != 1:
        raise SystemExit("--mode p2p takes a plain ring workload (a2a = 1)")
    if world > 1:
        w = w.replace(cp=world)  # one rank per GPU
    stream = torch.cuda.current_stream()
    desc = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype)
    nat = W.draw_cast(w)
    H = [w.H_q, w.H_kv, w.H_kv, w.H_q]
    lay = []
    for x, h in zip(nat, H):  # layout order, prepared outside the timed region
        y = torch.empty(w.B, h, w.T, w.D, dtype=x.dtype, device=dev)
        cp.check(cp.cpattn_layout(cp.ZIGZAG_FWD, desc, x.to(dev), y, h))
        lay.append(y)
    chunks = [R.rank_chunks(x, w.cp) for x in lay]  # [tensor][rank]
    steps = R.LibrarySteps(desc, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    if world > 1:
        exch = R.DistExchange()
        mine = [c[rank] for c in chunks]

        def step():
            o, lse, _ = R.ring_forward(steps, exch, mine[0], mine[1], mine[2])
            return R.ring_backward(steps, exch, mine[0], mine[1], mine[2], o, lse, mine[3])[:3]
    else:
        def step():
            os_, lses, _ = R.emulate_ring_forward(steps, w.cp, *chunks[:3])
            return R.emulate_ring_backward(steps, w.cp, *chunks[:3], os_, lses, chunks[3])[:3]

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    cp.check(cp.cpattn_check())
    graph = None
    if world == 1 and not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()

    def run_once():
        if graph is not None:
            graph.replay()
        else:
            step()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        run_once()
        b.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    clocks = sampler.stop(t0, t1)
    cp.check(cp.cpattn_check())
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, dev)
    flops = w.fwd_flops + w.bwd_flops
    value = flops / (ms * 1e-3) / 1e12   # the ranks share one problem: no world factor
    # per-kernel durations (eager launches of the same steps, events on the stream)
    cp.cpattn_timing_reset()
    cp.cpattn_timing_enable(True)
    for _ in range(min(args.steps, 5)):
        flush.zero_()
        step()
    cp.check(cp.cpattn_timing_collect())
    cp.cpattn_timing_enable(False)
    table = cp.cpattn_timing_table()
    cp.cpattn_timing_reset()
    n_timed = min(args.steps, 5)
    launches_per_step = sum(n * kernels_in(k) for k, (_, n) in table.items()) / n_timed
    total = sum(t for t, _ in table.values())
    kernels = {name: {"avg_ms": tot / n, "launches": n, "share": tot / total}
               for name, (tot, n) in table.items()}
    dom = max(table, key=lambda n: table[n][0])
    pk, src_pk = peaks()
    peak, peak_what = tensor_peak(pk, src_pk, t1 - t0)
    bound, work = kernel_flops_or_bytes(dom, w)
    avg_ms = table[dom][0] / table[dom][1]
    if bound == "tensor":
        achieved = work / (avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_what,
                "work_per_launch": work, "avg_launch_ms": avg_ms,
                "note": "work per launch is the average over the cp^2 (rank, chunk) steps",
                "traffic": None}
        if kernels_in(dom) == 2:
            roof["unit_of"] = PAIR_NOTE
    else:
        roof = hbm_roofline(dom, work, avg_ms, pk, src_pk)
        roof["traffic"] = None
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": config_of(w, {
                "mode": "p2p",
                "parallelism": (f"ring over {world} GPUs, K/V exchanged by NCCL point to point"
                                if world > 1 else
                                f"the {w.cp} ranks of the ring emulated in lockstep on one GPU"),
                "graph": graph is not None,
                "l2": "flushed before every timed step (256 MiB device write, outside the events)",
                "step": "per rank and step: cpattn_partial_fwd + cpattn_merge, then "
                        "cpattn_partial_bwd with the chunk's float32 dK/dV travelling the ring",
                "pct_of_bf16_peak": value / peak, "peak_source": peak_what}),
            "roofline": roof, "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clocks, "e2e": None,
            "e2e_note": "not measured in this mode: the inputs are the ranks' chunks, "
                        "already resident", "kernels": kernels}


def run_hbm(args):
    """The HBM-bound kernels alone: each launch timed with CUDA events on its stream,
    L2 flushed (256 MiB write) before every launch, outside the events."""
    import torch
    import blockwise_online_softmax_cpattn_gb300 as cp

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    g = torch.Generator(device="cpu").manual_seed(5)
    pk, src_pk = peaks()
    reps = max(5, min(args.steps, 50))

    def timed(fn):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        cp.check(cp.cpattn_check())
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    out = {}

    def record(name, nbytes, ms, what):
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"bytes": nbytes, "ms": ms, "gbs": gbs, "frac": gbs / pk["hbm_gbs"],
                     "what": what}

    # (O, LSE) merge of one ring step's partials: B * H_q * c rows of D floats
    for label, w in (("llama", W.LLAMA), ("qwen3", W.QWEN3)):
        rows = w.B * w.a2a * (w.H_q // w.a2a) * (w.T // (w.cp // w.a2a))
        o_a, o_b = (torch.randn(rows, w.D, generator=g).to(dev) for _ in range(2))
        l_a, l_b = (torch.randn(rows, generator=g).to(dev) for _ in range(2))
        o_o, l_o = torch.empty_like(o_a), torch.empty_like(l_a)
        ms = timed(lambda: cp.check(cp.cpattn_merge(rows, w.D, o_a, l_a, o_b, l_b, o_o, l_o)))
        record(f"merge_{label}", rows * (3 * 4 * w.D + 12), ms,
               f"cpattn_merge, {rows} rows x D {w.D} (one ring step of {w.name}): "
               "two (O, LSE) read, one written, float32")
        del o_a, o_b, o_o
    # a2a re-layout of the Qwen3 workload (a2a 2 x p2p 4): q-sized and k-sized
    w = W.QWEN3
    d = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype, a2a=w.a2a)
    for h, tag in ((w.H_q, "q"), (w.H_kv, "kv")):
        x = torch.randn(w.B * w.T * h * w.D, generator=g).to(torch.bfloat16).to(dev)
        y = torch.empty_like(x)
        n = x.numel() * 2
        record(f"a2a_fwd_{tag}", 2 * n,
               timed(lambda: cp.check(cp.cpattn_layout(cp.A2A_FWD, d, x, y, h))),
               f"cpattn_layout A2A_FWD of the {tag} tensor of {w.name} ({h} heads, "
               f"{n / 1e6:.1f} MB): one read, one write")
        record(f"a2a_inv_{tag}", 2 * n,
               timed(lambda: cp.check(cp.cpattn_layout(cp.A2A_INV, d, y, x, h))),
               f"cpattn_layout A2A_INV of the {tag} tensor of {w.name}: one read, one write")
        del x, y
    # zigzag chunk copies of the LLaMA workload
    w = W.LLAMA
    d = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype)
    for h, tag in ((w.H_q, "q"), (w.H_kv, "kv")):
        x = torch.randn(w.B, h, w.T, w.D, generator=g).to(torch.bfloat16).to(dev)
        y = torch.empty_like(x)
        n = x.numel() * 2
        record(f"zigzag_fwd_{tag}", 2 * n,
               timed(lambda: cp.check(cp.cpattn_layout(cp.ZIGZAG_FWD, d, x, y, h))),
               f"cpattn_layout ZIGZAG_FWD of the {tag} tensor of {w.name} ({n / 1e6:.1f} MB)")
        del x, y
    # the batched permutes a step launches: the four tensors q, k, v, dO in one call
    for label, w, perm, tag in ((("zigzag_batch_llama", W.LLAMA, cp.ZIGZAG_FWD, "zigzag"),
                                 ("a2a_batch_ulysses", W.ULYSSES, cp.A2A_FWD, "a2a"))):
        d = cp.make_desc(w.B, w.H_q, w.H_kv, w.T, w.D, w.cp, w.layout, w.dtype, a2a=w.a2a)
        heads = [w.H_q, w.H_kv, w.H_kv, w.H_q]
        xs = [torch.randn(w.B * h * w.T * w.D, generator=g).to(torch.bfloat16).to(dev)
              for h in heads]
        ys = [torch.empty_like(x) for x in xs]
        n = sum(x.numel() * 2 for x in xs)
        record(label, 2 * n,
               timed(lambda: cp.check(cp.cpattn_layout_batch(perm, d, xs, ys, heads))),
               f"cpattn_layout_batch of the {tag} permutes of a {w.name} step's q, k, v, dO "
               f"({n / 1e6:.1f} MB) in one launch")
        del xs, ys
    return {"metric": "HBM-bound kernels: GB/s of algorithmic bytes per launch", "unit": "GB/s",
            "n_gpus": 1, "higher_is_better": True, "data": "synthetic",
            "peak": pk["hbm_gbs"], "peak_source": f"{src_pk} copy bandwidth",
            "l2": "flushed before every launch (256 MiB device write, outside the events)",
            "reps": reps, "kernels": out}


# ---------------------------------------------------------------------------
# the oracle (CPU) legs
# ---------------------------------------------------------------------------
def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [x.get("num_threads") for x in threadpool_info() if x.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def oracle_head(w, nat, h, T_sample=None):
    """Time the oracle's forward + backward of query head h (and its K/V head),
    on the first T_sample tokens (a causal prefix is a self-contained problem)."""
    from oracle import attention as OA
    Ts = w.T if T_sample is None else T_sample
    g = h // (w.H_q // w.H_kv)
    q, k, v, do = (W.as_f64(x[:1, hh:hh + 1, :Ts]) for x, hh in
                   ((nat[0], h), (nat[1], g), (nat[2], g), (nat[3], h)))
    t0 = time.perf_counter()
    OA.attention_fwd(q, k, v, w.scale)
    OA.attention_bwd(q, k, v, do, w.scale)
    dt = time.perf_counter() - t0
    flops = 14.0 * w.D * Ts * (Ts + 1) / 2
    return flops, dt


def cpu_baseline(w):
    nat = W.draw_cast(w)
    flops, dt, n = 0.0, 0.0, 0
    for h in range(w.H_q):
        f, t = oracle_head(w, nat, h)
        flops += f
        dt += t
        n += 1
        if dt > 10.0:
            break
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{n} of {w.H_q} query heads (with their K/V heads), full T={w.T}, "
                      f"fwd+bwd in float64 numpy, {dt:.1f} s",
            "seconds": dt}


def run_reference(args):
    w = W.ALL[args.workload]
    nat = W.draw_cast(w)
    Ts = min(w.T, 1024)
    for i in range(args.warmup):
        oracle_head(w, nat, i % w.H_q, Ts)
    flops, dt = 0.0, 0.0
    for i in range(args.steps):
        f, t = oracle_head(w, nat, i % w.H_q, Ts)
        flops += f
        dt += t
    value = flops / dt / 1e12
    ms = dt / args.steps * 1e3
    sample = (f"per step: the first {Ts} tokens of one query head (cycling over the {w.H_q} heads) "
              f"with its K/V head, fwd+bwd in float64 numpy")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, {"sample": sample}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if args.mode == "hbm":
        if rank == 0:
            print(json.dumps(run_hbm(args)))
        return
    if args.mode == "p2p":
        out = run_p2p(args, rank, world)
    elif args.mode == "allgather":
        out = run_allgather(args, rank, world)
    else:
        out = run_cpattn(args, rank, world)
    if rank == 0:
        w = W.ALL[args.workload]
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(w)
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
