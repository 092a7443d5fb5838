"""GPU: layout permutes (bit-exact against the oracle's index maps) and the
(O, LSE) merge kernel (against the oracle's merge)."""
import numpy as np
import pytest
import torch

from gpu_helpers import cp_mod, dev, rel
from oracle import attention as OA
from oracle import layouts as OL

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,T,D,cp_,layout", [
    (2, 3, 64, 16, 4, "zigzag"), (1, 4, 1024, 128, 8, "zigzag"), (2, 2, 96, 24, 3, "contiguous"),
    (1, 2, 40, 5, 2, "zigzag"), (4, 12, 1024, 64, 4, "zigzag")])
def test_zigzag_permute_bit_exact(dtype, B, H, T, D, cp_, layout):
    cp = cp_mod()
    g = torch.Generator().manual_seed(7)
    x = torch.randn(B, H, T, D, generator=g).to(dtype)
    d = cp.make_desc(B, H, H, T, D, cp_, layout, "bf16" if dtype == torch.bfloat16 else "f32")
    xs = x.to(dev())
    y = torch.empty_like(xs)
    cp.check(cp.cpattn_layout(cp.ZIGZAG_FWD, d, xs, y, H))
    want = x[:, :, torch.from_numpy(OL.positions(T, cp_, layout))]
    assert torch.equal(_bits(y.cpu()), _bits(want.contiguous()))
    z = torch.empty_like(xs)
    cp.check(cp.cpattn_layout(cp.ZIGZAG_INV, d, y, z, H))
    assert torch.equal(_bits(z.cpu()), _bits(x))
    cp.check(cp.cpattn_check())


@pytest.mark.parametrize("kind", ["fwd", "inv"])
@pytest.mark.parametrize("dtype,layout,B,Hq,Hkv,T,D,cp_", [
    (torch.bfloat16, "zigzag", 1, 32, 8, 8192, 128, 8),     # the LLaMA step's four tensors
    (torch.bfloat16, "contiguous", 2, 4, 2, 1024, 64, 4),
    (torch.float32, "zigzag", 2, 3, 1, 96, 20, 3),
    (torch.float32, "zigzag", 2, 3, 1, 96, 6, 3),           # 24-byte rows: per-tensor launches
    (torch.float32, "zigzag", 1, 4, 4, 256, 16, 2)])
def test_layout_batch_equals_single_permutes(kind, dtype, layout, B, Hq, Hkv, T, D, cp_):
    """cpattn_layout_batch over a step's q, k, v, dO equals cpattn_layout on each,
    bit for bit, and so the oracle's index map."""
    cp = cp_mod()
    g = torch.Generator().manual_seed(13)
    dt = "bf16" if dtype == torch.bfloat16 else "f32"
    heads = [Hq, Hkv, Hkv, Hq]
    xs = [torch.randn(B, h, T, D, generator=g).to(dtype) for h in heads]
    d = cp.make_desc(B, Hq, Hkv, T, D, cp_, layout, dt)
    perm = cp.ZIGZAG_FWD if kind == "fwd" else cp.ZIGZAG_INV
    src = [x.to(dev()) for x in xs]
    got = [torch.empty_like(x) for x in src]
    cp.check(cp.cpattn_layout_batch(perm, d, src, got, heads))
    for x, y, h in zip(src, got, heads):
        one = torch.empty_like(x)
        cp.check(cp.cpattn_layout(perm, d, x, one, h))
        assert torch.equal(_bits(y), _bits(one))
    pos = OL.positions(T, cp_, layout)
    idx = torch.from_numpy(pos if kind == "fwd" else OL.layout_slots(T, cp_, layout))
    for x, y in zip(xs, got):
        assert torch.equal(_bits(y.cpu()), _bits(x[:, :, idx].contiguous()))
    cp.check(cp.cpattn_check())


@pytest.mark.parametrize("B,Hq,Hkv,T,D,cp_,a2a,dtype", [
    (1, 32, 8, 8192, 128, 8, 8, torch.bfloat16),   # the full-Ulysses step's four tensors
    (2, 8, 4, 1024, 64, 4, 2, torch.bfloat16),
    (1, 8, 2, 512, 128, 4, 2, torch.float32),      # 512-byte rows
    (1, 6, 3, 96, 24, 6, 3, torch.float32)])       # 96-byte rows: per-tensor launches
def test_a2a_layout_batch_equals_single_permutes(B, Hq, Hkv, T, D, cp_, a2a, dtype):
    """cpattn_layout_batch of the all-to-all re-layout (one launch of row gathers)
    equals cpattn_layout on each tensor, bit for bit, both ways."""
    cp = cp_mod()
    g = torch.Generator().manual_seed(17)
    dt = "bf16" if dtype == torch.bfloat16 else "f32"
    heads = [Hq, Hkv, Hkv, Hq]
    d = cp.make_desc(B, Hq, Hkv, T, D, cp_, "zigzag", dt, a2a=a2a)
    shards = [torch.randn(B * T * h * D, generator=g).to(dtype).to(dev()) for h in heads]
    got = [torch.empty_like(x) for x in shards]
    cp.check(cp.cpattn_layout_batch(cp.A2A_FWD, d, shards, got, heads))
    for x, y, h in zip(shards, got, heads):
        one = torch.empty_like(x)
        cp.check(cp.cpattn_layout(cp.A2A_FWD, d, x, one, h))
        assert torch.equal(_bits(y), _bits(one))
    back = [torch.empty_like(x) for x in shards]
    cp.check(cp.cpattn_layout_batch(cp.A2A_INV, d, got, back, heads))
    for x, y in zip(shards, back):
        assert torch.equal(_bits(y), _bits(x))
    cp.check(cp.cpattn_check())


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("B,H,T,D,cp_,a2a", [(1, 8, 256, 64, 8, 2), (2, 4, 128, 32, 4, 2),
                                             (1, 6, 96, 16, 6, 3), (1, 32, 32768, 128, 8, 2),
                                             (1, 4, 32768, 128, 8, 2)])
def test_a2a_permute_bit_exact(layout, B, H, T, D, cp_, a2a):
    cp = cp_mod()
    g = torch.Generator().manual_seed(11)
    nat = torch.randn(B, H, T, D, generator=g).to(torch.bfloat16)
    src = torch.from_numpy(OL.token_shards(nat.view(torch.int16).numpy(), cp_, layout))
    idx = torch.from_numpy(OL.a2a_source_rows(B, H, T, cp_, a2a, layout).reshape(-1))
    want = src.reshape(-1, D)[idx].reshape(a2a, B, H // a2a, T, D)
    d = cp.make_desc(B, H, H, T, D, cp_, layout, "bf16", a2a=a2a)
    s_dev = src.view(torch.bfloat16).to(dev())
    out = torch.empty(a2a, B, H // a2a, T, D, dtype=torch.bfloat16, device=dev())
    cp.check(cp.cpattn_layout(cp.A2A_FWD, d, s_dev, out, H))
    assert torch.equal(out.cpu().view(torch.int16), want)
    back = torch.empty_like(s_dev)
    cp.check(cp.cpattn_layout(cp.A2A_INV, d, out, back, H))
    assert torch.equal(back.cpu().view(torch.int16), src)
    cp.check(cp.cpattn_check())


def _partials(rows, D, seed):
    rng = np.random.default_rng(seed)
    oa = rng.standard_normal((rows, D)).astype(np.float32)
    ob = rng.standard_normal((rows, D)).astype(np.float32)
    la = (rng.standard_normal(rows) * 4).astype(np.float32)
    lb = (rng.standard_normal(rows) * 4).astype(np.float32)
    la[::7] = -np.inf
    oa[::7] = 0
    lb[::5] = -np.inf
    ob[::5] = 0
    if rows > 4:
        lb[3] = la[3] = -np.inf
        oa[3] = ob[3] = 0
        la[4] = lb[4] = 80.0   # equal large logits
    return oa, la, ob, lb


@pytest.mark.parametrize("rows,D", [(1000, 128), (77, 64), (33, 5), (1, 16), (32 * 1024, 128)])
def test_merge_matches_oracle(rows, D):
    cp = cp_mod()
    oa, la, ob, lb = _partials(rows, D, rows + D)
    ro, rl = OA.merge(oa.astype(np.float64), la, ob.astype(np.float64), lb)
    t = [torch.from_numpy(a).to(dev()) for a in (oa, la, ob, lb)]
    oo = torch.empty_like(t[0])
    lo = torch.empty_like(t[1])
    cp.check(cp.cpattn_merge(rows, D, t[0], t[1], t[2], t[3], oo, lo))
    o = oo.cpu().numpy()
    lse = lo.cpu().numpy()
    assert np.array_equal(np.isinf(lse), np.isinf(rl)) and not np.isnan(lse).any()
    fin = np.isfinite(rl)
    if fin.any():
        assert np.max(np.abs(lse[fin] - rl[fin])) <= 1e-5 * max(1.0, np.max(np.abs(rl[fin])))
    assert rel(o, ro) <= 1e-5
    if rows > 4:
        assert np.all(o[3] == 0) and lse[3] == -np.inf
    # in place (out aliases a) gives the same bits
    cp.check(cp.cpattn_merge(rows, D, t[0], t[1], t[2], t[3], t[0], t[1]))
    assert torch.equal(t[0].cpu(), oo.cpu()) and torch.equal(t[1].cpu(), lo.cpu())
    cp.check(cp.cpattn_check())
