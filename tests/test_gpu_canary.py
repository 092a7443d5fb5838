"""GPU: no entry point writes outside the buffers it is given, and each writes all
of its outputs.

compute-sanitizer is closed on this machine, so out-of-bounds stores are caught with
guard regions instead.  Every output (and workspace) of every entry point lives
inside a larger allocation: 64 KiB of canary bytes before it and after it.  The
output itself is filled with 0xFF bytes, a NaN in float32 and in bfloat16, before
the call.  After the call the host checks that every canary byte is unchanged and
that no output element is still NaN (every element was written).  Shapes are
small but span several 128-token tiles, ragged chunk halves, grouped queries,
both head dimensions of the tensor-core path and the float32 path."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import cp_mod, desc_of, dev, ring_inputs

pytestmark = pytest.mark.gpu

GUARD = 64 * 1024
CANARY = 0xA5


class Guarded:
    """A tensor placed between two canary regions of one device allocation."""

    def __init__(self, shape, dtype):
        elt = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape)) * elt
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), CANARY, dtype=torch.uint8,
                              device=dev())
        self.raw[GUARD:GUARD + self.nbytes] = 0xFF
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def guards_intact(self):
        r = self.raw.cpu()
        return bool((r[:GUARD] == CANARY).all() and (r[GUARD + self.nbytes:] == CANARY).all())

    def all_written(self):
        return not bool(torch.isnan(self.t.float()).any())


def guarded_like(x, shape=None, dtype=None):
    return Guarded(tuple(x.shape) if shape is None else shape, x.dtype if dtype is None else dtype)


def check_all(bufs, written=()):
    for name, g in bufs.items():
        assert g.guards_intact(), f"{name}: a canary byte changed"
    for name in written:
        assert bufs[name].all_written(), f"{name}: some element was never written"


RING = [
    W.Workload("cn_tc_T1024_cp4_zz_gqa2", 2, 4, 2, 1024, 128, 4, "zigzag", "bf16"),
    W.Workload("cn_tc_T768_cp3_contig_D64", 1, 3, 3, 768, 64, 3, "contiguous", "bf16"),
    W.Workload("cn_simt_f32_T96_cp3_zz", 1, 2, 1, 96, 20, 3, "zigzag", "f32"),
    W.Workload("cn_simt_bf16_T128_cp2_D32", 1, 2, 2, 128, 32, 2, "zigzag", "bf16"),
]


@pytest.mark.parametrize("w", RING, ids=lambda w: w.name)
def test_ring_and_partial_stay_in_bounds(w):
    cp = cp_mod()
    _, (q, k, v, do) = ring_inputs(w)
    d = desc_of(w)
    B, H, T, D, c = w.B, w.H_q, w.T, w.D, w.T // w.cp
    f32 = torch.float32
    b = {"o": guarded_like(q), "lse": Guarded((B, H, T), f32), "dq": guarded_like(q),
         "dk": guarded_like(k), "dv": guarded_like(v),
         "ws": Guarded((cp.cpattn_ring_bwd_workspace(d),), torch.uint8),
         "o_part": Guarded((B, H, c, D), f32), "lse_part": Guarded((B, H, c), f32),
         "o_m": Guarded((B, H, c, D), f32), "lse_m": Guarded((B, H, c), f32),
         "dq_part": Guarded((B, H, c, D), f32), "dk_part": Guarded((B, w.H_kv, c, D), f32),
         "dv_part": Guarded((B, w.H_kv, c, D), f32),
         "ws_part": Guarded((cp.cpattn_partial_bwd_workspace(d),), torch.uint8)}
    cp.check(cp.cpattn_ring_fwd(d, q, k, v, b["o"].t, b["lse"].t))
    cp.check(cp.cpattn_ring_bwd(d, q, k, v, b["o"].t, b["lse"].t, do, b["dq"].t, b["dk"].t,
                                b["dv"].t, b["ws"].t))
    r = w.cp - 1
    cp.check(cp.cpattn_partial_fwd(d, r, r, q, k, v, b["o_part"].t, b["lse_part"].t))
    # the merge of the diagonal step with itself (out of place): lse + ln 2, same o
    cp.check(cp.cpattn_merge(B * H * c, D, b["o_part"].t, b["lse_part"].t, b["o_part"].t,
                             b["lse_part"].t, b["o_m"].t, b["lse_m"].t))
    # one backward ring step: the last rank's rows against chunk 0
    sl = slice(r * c, (r + 1) * c)
    o_r, lse_r, do_r = (x[:, :, sl].contiguous() for x in (b["o"].t, b["lse"].t, do))
    cp.check(cp.cpattn_partial_bwd_stats(d, o_r, lse_r, do_r, b["ws_part"].t))
    cp.check(cp.cpattn_partial_bwd(d, r, 0, q, k, v, do_r, b["dq_part"].t, b["dk_part"].t,
                                   b["dv_part"].t, 0, b["ws_part"].t))
    cp.check(cp.cpattn_check())
    check_all(b, written=("o", "lse", "dq", "dk", "dv", "o_part", "lse_part", "o_m", "lse_m",
                          "dq_part", "dk_part", "dv_part"))


@pytest.mark.parametrize("w", [RING[0], RING[2]], ids=lambda w: w.name)
def test_allgather_stays_in_bounds(w):
    cp = cp_mod()
    _, (q, k, v, do) = ring_inputs(w)
    d = desc_of(w)
    B, H, T, D, c = w.B, w.H_q, w.T, w.D, w.T // w.cp
    f32 = torch.float32
    b = {"dk_sum": Guarded((B, w.H_kv, T, D), f32), "dv_sum": Guarded((B, w.H_kv, T, D), f32),
         "ws": Guarded((cp.cpattn_allgather_bwd_workspace(d),), torch.uint8)}
    for r in range(w.cp):
        b[f"o{r}"] = Guarded((B, H, c, D), q.dtype)
        b[f"lse{r}"] = Guarded((B, H, c), f32)
        b[f"dq{r}"] = Guarded((B, H, c, D), q.dtype)
        cp.check(cp.cpattn_allgather_fwd(d, r, q, k, v, b[f"o{r}"].t, b[f"lse{r}"].t))
        do_r = do[:, :, r * c:(r + 1) * c].contiguous()
        cp.check(cp.cpattn_allgather_bwd(d, r, q, k, v, b[f"o{r}"].t, b[f"lse{r}"].t, do_r,
                                         b[f"dq{r}"].t, b["dk_sum"].t, b["dv_sum"].t, r > 0,
                                         b["ws"].t))
    cp.check(cp.cpattn_check())
    check_all(b, written=[n for n in b if n != "ws"])


@pytest.mark.parametrize("w", [RING[0], RING[1], RING[2]], ids=lambda w: w.name)
def test_packed_stays_in_bounds(w):
    cp = cp_mod()
    _, (q, k, v, do) = ring_inputs(w)
    d = desc_of(w)
    B, H, T = w.B, w.H_q, w.T
    rng = np.random.default_rng(T)
    starts = np.stack([np.concatenate([[0], np.sort(rng.integers(0, T + 1, 4)), [T]])
                       for _ in range(B)]).astype(np.int32)
    st = torch.from_numpy(starts).to(dev())
    b = {"o": guarded_like(q), "lse": Guarded((B, H, T), torch.float32), "dq": guarded_like(q),
         "dk": guarded_like(k), "dv": guarded_like(v),
         "ws": Guarded((cp.cpattn_packed_workspace(d),), torch.uint8)}
    cp.check(cp.cpattn_ring_fwd_packed(d, st, 5, q, k, v, b["o"].t, b["lse"].t, b["ws"].t))
    cp.check(cp.cpattn_ring_bwd_packed(d, st, 5, q, k, v, b["o"].t, b["lse"].t, do, b["dq"].t,
                                       b["dk"].t, b["dv"].t, b["ws"].t))
    cp.check(cp.cpattn_check())
    check_all(b, written=("o", "lse", "dq", "dk", "dv"))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_layouts_stay_in_bounds(dtype):
    cp = cp_mod()
    B, H, T, D, cp_, a2a = 2, 4, 256, 48, 4, 2
    dt = "bf16" if dtype == torch.bfloat16 else "f32"
    x = torch.randn(B, H, T, D, generator=torch.Generator().manual_seed(3)).to(dtype).to(dev())
    dz = cp.make_desc(B, H, H, T, D, cp_, "zigzag", dt)
    da = cp.make_desc(B, H, H, T, D, cp_, "zigzag", dt, a2a=a2a)
    b = {"zz": guarded_like(x), "inv": guarded_like(x),
         "a2a": Guarded((a2a, B, H // a2a, T, D), dtype), "a2a_inv": guarded_like(x)}
    cp.check(cp.cpattn_layout(cp.ZIGZAG_FWD, dz, x, b["zz"].t, H))
    cp.check(cp.cpattn_layout(cp.ZIGZAG_INV, dz, b["zz"].t, b["inv"].t, H))
    # x read as token shards [cp][B][T/cp][H][D] (same bytes)
    cp.check(cp.cpattn_layout(cp.A2A_FWD, da, x, b["a2a"].t, H))
    cp.check(cp.cpattn_layout(cp.A2A_INV, da, b["a2a"].t, b["a2a_inv"].t, H))
    cp.check(cp.cpattn_check())
    check_all(b, written=tuple(b))
    assert torch.equal(b["inv"].t, x) and torch.equal(b["a2a_inv"].t, x)
