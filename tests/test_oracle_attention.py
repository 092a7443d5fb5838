"""Pins of the FP64 oracle's attention, backward and merge (CPU only).

Each pin ties the oracle to something other than itself: a library routine on
the case it covers (torch's scaled_dot_product_attention and autograd in float64),
closed forms, invariances of softmax, conservation laws of the backward, central
finite differences, and the order invariance of the merge that the tutorial
"上下文并行" (section "朴素 Ring Attention") states.
"""
import numpy as np
import pytest
import torch

from conftest import rel_err
from oracle import attention as A
from oracle import layouts as L


def _rand(rng, B, Hq, Hkv, T, D, qs=1.0):
    q = rng.standard_normal((B, Hq, T, D)) * qs
    k = rng.standard_normal((B, Hkv, T, D))
    v = rng.standard_normal((B, Hkv, T, D))
    do = rng.standard_normal((B, Hq, T, D))
    return q, k, v, do


def _torch_reference(q, k, v, do, scale):
    """float64 torch SDPA (is_causal) with explicit head repeat, plus autograd."""
    n_rep = q.shape[1] // k.shape[1]
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    kr = tk.repeat_interleave(n_rep, dim=1)
    vr = tv.repeat_interleave(n_rep, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(tq, kr, vr, is_causal=True,
                                                         scale=scale)
    (o * torch.tensor(do)).sum().backward()
    T = q.shape[2]
    s = scale * tq.detach() @ kr.detach().transpose(-1, -2)
    s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return (o.detach().numpy(), lse.numpy(), tq.grad.numpy(), tk.grad.numpy(),
            tv.grad.numpy())


@pytest.mark.parametrize("B,Hq,Hkv,T,D", [(2, 4, 4, 37, 8), (1, 6, 2, 50, 16), (1, 4, 1, 33, 5)])
def test_matches_torch_sdpa_and_autograd(rng, B, Hq, Hkv, T, D):
    q, k, v, do = _rand(rng, B, Hq, Hkv, T, D)
    scale = 1 / np.sqrt(D)
    o, lse = A.attention_fwd(q, k, v, scale, rows_per_block=16)
    dq, dk, dv = A.attention_bwd(q, k, v, do, scale, rows_per_block=16)
    ro, rlse, rdq, rdk, rdv = _torch_reference(q, k, v, do, scale)
    assert rel_err(o, ro) < 1e-13
    assert rel_err(lse, rlse) < 1e-13
    assert rel_err(dq, rdq) < 1e-12
    assert rel_err(dk, rdk) < 1e-12
    assert rel_err(dv, rdv) < 1e-12


def test_large_logits_stay_finite(rng):
    """Safe softmax: logits of size ~1e3 neither overflow nor lose the result."""
    q, k, v, do = _rand(rng, 1, 2, 2, 40, 8, qs=300.0)
    scale = 1 / np.sqrt(8)
    o, lse = A.attention_fwd(q, k, v, scale)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    ro, rlse, *_ = _torch_reference(q, k, v, do, scale)
    assert rel_err(o, ro) < 1e-12
    assert rel_err(lse, rlse) < 1e-12


def test_zero_queries_give_prefix_mean(rng):
    """q = 0 => S = 0 => O_i = mean(v_0..v_i), LSE_i = ln(i+1)."""
    _, k, v, _ = _rand(rng, 1, 3, 3, 29, 7)
    q = np.zeros((1, 3, 29, 7))
    o, lse = A.attention_fwd(q, k, v, 0.5)
    n = np.arange(1, 30)
    prefix_mean = np.cumsum(v, axis=2) / n[None, None, :, None]
    assert np.max(np.abs(o - prefix_mean)) < 1e-13
    assert np.max(np.abs(lse - np.log(n)[None, None, :])) < 1e-13


def test_single_token(rng):
    """T = 1 => O = v_0 and LSE = S_00."""
    q, k, v, _ = _rand(rng, 2, 2, 1, 1, 6)
    o, lse = A.attention_fwd(q, k, v, 0.3)
    assert np.array_equal(o, np.repeat(v, 2, axis=1))
    s00 = 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], np.repeat(k, 2, axis=1)[:, :, 0])
    assert np.max(np.abs(lse[:, :, 0] - s00)) < 1e-14


def test_shift_invariances(rng):
    """Adding one vector to every key leaves O unchanged (a per-row constant in S);
    adding one vector to every value shifts O by it."""
    q, k, v, _ = _rand(rng, 1, 4, 2, 31, 8)
    scale = 0.4
    o, lse = A.attention_fwd(q, k, v, scale)
    ck = rng.standard_normal((1, 2, 1, 8))
    o2, lse2 = A.attention_fwd(q, k + ck, v, scale)
    assert np.max(np.abs(o2 - o)) < 1e-12
    shift = scale * np.einsum("bhtd,bhd->bht", q, np.repeat(ck, 2, axis=1)[:, :, 0])
    assert np.max(np.abs(lse2 - (lse + shift))) < 1e-12
    cv = rng.standard_normal((1, 2, 1, 8))
    o3, _ = A.attention_fwd(q, k, v + cv, scale)
    assert np.max(np.abs(o3 - (o + np.repeat(cv, 2, axis=1)))) < 1e-12


def test_probability_rows_sum_to_one(rng):
    S = rng.standard_normal((20, 20)) * 5
    vis = A.causal_visible(np.arange(20), np.arange(20))
    P, m, l = A.safe_softmax_rows(S, vis)
    assert np.max(np.abs(P.sum(axis=1) - 1)) < 1e-14
    assert np.all(P[~vis] == 0)
    assert np.all(P <= 1.0)


def test_backward_conservation_laws(rng):
    """sum_j dS_ij = 0 per row => sum_j dK_j = 0 per kv head;
    dV sums the probabilities' columns => sum_j dV_j = sum over the group's dO."""
    q, k, v, do = _rand(rng, 2, 6, 2, 45, 8)
    dq, dk, dv = A.attention_bwd(q, k, v, do, 0.35)
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-11
    do_group = do.reshape(2, 2, 3, 45, 8).sum(axis=(2, 3))
    assert np.max(np.abs(dv.sum(axis=2) - do_group)) < 1e-11


def test_finite_differences(rng):
    """Central differences of L = sum(dO * O) agree with the analytic gradients."""
    q, k, v, do = _rand(rng, 1, 2, 1, 6, 3)
    scale = 0.7
    dq, dk, dv = A.attention_bwd(q, k, v, do, scale)

    def loss(q_, k_, v_):
        return float(np.sum(do * A.attention_fwd(q_, k_, v_, scale)[0]))

    eps = 1e-5
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args_p = [q, k, v]; args_p[which] = xp
            args_m = [q, k, v]; args_m[which] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        assert rel_err(g, num) < 1e-8, which


def test_row_blocking_is_exact(rng):
    q, k, v, do = _rand(rng, 1, 2, 2, 70, 8)
    a = A.attention_fwd(q, k, v, 0.3, rows_per_block=70)
    b = A.attention_fwd(q, k, v, 0.3, rows_per_block=9)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    ga = A.attention_bwd(q, k, v, do, 0.3, rows_per_block=70)
    gb = A.attention_bwd(q, k, v, do, 0.3, rows_per_block=13)
    for x, y in zip(ga, gb):
        assert rel_err(x, y) < 1e-14


def test_sampled_rows_match_full(rng):
    q, k, v, do = _rand(rng, 1, 4, 2, 64, 8)
    scale = 0.35
    o, lse = A.attention_fwd(q, k, v, scale)
    dq, dk, dv = A.attention_bwd(q, k, v, do, scale)
    rows = np.array([0, 5, 31, 63])
    ro, rl = A.fwd_rows(q[0, 3], k[0, 1], v[0, 1], rows, scale)
    assert rel_err(ro, o[0, 3, rows]) < 1e-14 and rel_err(rl, lse[0, 3, rows]) < 1e-14
    rdq = A.dq_rows(q[0, 2], k[0, 1], v[0, 1], do[0, 2], rows, scale)
    assert rel_err(rdq, dq[0, 2, rows]) < 1e-13
    kv_rows = np.array([40, 41, 60, 63])
    rdk, rdv = A.dkdv_rows(q[0, 2:4], k[0, 1], v[0, 1], do[0, 2:4], kv_rows, scale,
                           rows_per_block=7)
    assert rel_err(rdk, dk[0, 1, kv_rows]) < 1e-13
    assert rel_err(rdv, dv[0, 1, kv_rows]) < 1e-13


# ---------------------------------------------------------------- merge ----

def _partials(rng, n=9, D=5):
    os_ = [rng.standard_normal((n, D)) for _ in range(3)]
    ls = [rng.standard_normal(n) * 3 for _ in range(3)]
    ls[2][:3] = -np.inf
    os_[2][:3] = 0.0
    return os_, ls


def test_merge_commutative_associative_identity(rng):
    (oa, ob, oc), (la, lb, lc) = _partials(rng)
    m1 = A.merge(oa, la, ob, lb)
    m2 = A.merge(ob, lb, oa, la)
    assert np.max(np.abs(m1[0] - m2[0])) < 1e-14 and np.max(np.abs(m1[1] - m2[1])) < 1e-14
    x = A.merge(*A.merge(oa, la, ob, lb), oc, lc)
    y = A.merge(oa, la, *A.merge(ob, lb, oc, lc))
    assert rel_err(x[0], y[0]) < 1e-14 and rel_err(x[1], y[1]) < 1e-14
    empty_o = np.zeros_like(oa)
    empty_l = np.full_like(la, -np.inf)
    e = A.merge(oa, la, empty_o, empty_l)
    assert np.array_equal(e[0], oa) and np.array_equal(e[1], la)
    z = A.merge(empty_o, empty_l, empty_o, empty_l)
    assert np.all(z[0] == 0) and np.all(z[1] == -np.inf)


def test_merge_of_two_halves_is_attention_over_union(rng):
    """Splitting the keys in two sets and merging equals attention over all keys."""
    q = rng.standard_normal((12, 6)); k = rng.standard_normal((30, 6)); v = rng.standard_normal((30, 6))
    qp = np.arange(18, 30); kp = np.arange(30)
    full = A.partial_attention(q, k, v, qp, kp, 0.4)
    a = A.partial_attention(q, k[:11], v[:11], qp, kp[:11], 0.4)
    b = A.partial_attention(q, k[11:], v[11:], qp, kp[11:], 0.4)
    m = A.merge(*a, *b)
    assert rel_err(m[0], full[0]) < 1e-14 and rel_err(m[1], full[1]) < 1e-14


@pytest.mark.parametrize("layout,cp,T", [("contiguous", 4, 64), ("zigzag", 4, 64),
                                         ("zigzag", 2, 48), ("contiguous", 3, 45),
                                         ("zigzag", 8, 64)])
def test_ring_merge_equals_full_attention_any_order(rng, layout, cp, T):
    """Merging each rank's per-step partials in ring order gives full causal
    attention, and so does any shuffled step order."""
    q, k, v, _ = _rand(rng, 1, 2, 1, T, 8)
    scale = 0.35
    o_full, lse_full = A.attention_fwd(q, k, v, scale)
    c = T // cp
    pos = L.positions(T, cp, layout)
    for h in range(2):
        for r in range(cp):
            qs = pos[r * c:(r + 1) * c]
            for order in (list(range(cp)), list(rng.permutation(cp))):
                acc_o = np.zeros((c, 8)); acc_l = np.full(c, -np.inf)
                for i in order:
                    s = L.ring_source(r, i, cp)
                    ks = pos[s * c:(s + 1) * c]
                    po, pl = A.partial_attention(q[0, h, qs], k[0, 0, ks], v[0, 0, ks], qs, ks, scale)
                    acc_o, acc_l = A.merge(acc_o, acc_l, po, pl)
                assert rel_err(acc_o, o_full[0, h, qs]) < 1e-13
                assert np.max(np.abs(acc_l - lse_full[0, h, qs])) < 1e-12


@pytest.mark.parametrize("layout,cp,T", [("zigzag", 4, 48), ("contiguous", 3, 45),
                                         ("zigzag", 2, 20), ("contiguous", 4, 64)])
def test_partial_backward_steps_sum_to_the_full_backward(rng, layout, cp, T):
    """The per-step contributions of the ring backward (whole-forward statistics,
    one K/V chunk at a time): over the chunks a rank's queries meet they add up to
    the rank's dQ, and over the ranks a chunk meets (and the query heads of its
    group) to the chunk's dK and dV -- the backward pinned above."""
    q, k, v, do = _rand(rng, 1, 4, 2, T, 6)
    scale = 0.4
    o, lse = A.attention_fwd(q, k, v, scale)
    dq, dk, dv = A.attention_bwd(q, k, v, do, scale)
    c = T // cp
    pos = L.positions(T, cp, layout)
    gq, gk, gv = np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dv)
    for h in range(4):
        g = h // 2
        for r in range(cp):
            qs = pos[r * c:(r + 1) * c]
            for i in range(cp):
                s = L.ring_source(r, i, cp)
                ks = pos[s * c:(s + 1) * c]
                a, b, e = A.partial_attention_bwd(q[0, h, qs], k[0, g, ks], v[0, g, ks],
                                                  do[0, h, qs], o[0, h, qs], lse[0, h, qs], qs,
                                                  ks, scale)
                gq[0, h, qs] += a
                gk[0, g, ks] += b
                gv[0, g, ks] += e
    assert rel_err(gq, dq) < 1e-12 and rel_err(gk, dk) < 1e-12 and rel_err(gv, dv) < 1e-12


def test_partial_backward_of_one_chunk_is_the_backward(rng):
    """With a single chunk (cp = 1) the step is the whole backward of the head."""
    q, k, v, do = _rand(rng, 1, 1, 1, 30, 5)
    o, lse = A.attention_fwd(q, k, v, 0.5)
    dq, dk, dv = A.attention_bwd(q, k, v, do, 0.5)
    pos = np.arange(30)
    a, b, e = A.partial_attention_bwd(q[0, 0], k[0, 0], v[0, 0], do[0, 0], o[0, 0], lse[0, 0],
                                      pos, pos, 0.5)
    assert rel_err(a, dq[0, 0]) < 1e-13 and rel_err(b, dk[0, 0]) < 1e-13
    assert rel_err(e, dv[0, 0]) < 1e-13


def test_partial_backward_of_a_hidden_chunk_is_zero(rng):
    """Queries that see none of the chunk's keys contribute nothing."""
    q, k, v, do = _rand(rng, 1, 1, 1, 8, 3)
    o = rng.standard_normal((8, 3))
    a, b, e = A.partial_attention_bwd(q[0, 0], k[0, 0], v[0, 0], do[0, 0], o, np.zeros(8),
                                      np.arange(8), np.arange(8, 16), 1.0)
    assert not a.any() and not b.any() and not e.any()


def test_empty_partial_is_merge_identity(rng):
    """A query set that sees none of the keys yields (0, -inf)."""
    q = rng.standard_normal((4, 3)); k = rng.standard_normal((5, 3)); v = rng.standard_normal((5, 3))
    o, l = A.partial_attention(q, k, v, np.arange(4), np.arange(10, 15), 1.0)
    assert np.all(o == 0) and np.all(l == -np.inf)


# ---------------------------------------------------------------------------
# All-gather mode (pull request #181, mode table row "all_gather": local queries
# over the gathered K/V, K/V gradients summed over ranks by a ReduceScatter).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("layout,cp,T", [("zigzag", 4, 32), ("contiguous", 2, 24),
                                         ("zigzag", 2, 20)])
def test_allgather_rows_match_torch(rng, layout, cp, T):
    """Every rank's rows equal the library's full causal attention at its positions,
    its dQ rows the autograd dQ there, and the ranks' K/V gradients add up to the
    autograd dK/dV (the ReduceScatter sum)."""
    q, k, v, do = _rand(rng, 1, 4, 2, T, 8)
    scale = 0.4
    ro, rlse, rdq, rdk, rdv = _torch_reference(q, k, v, do, scale)
    dk_sum = np.zeros_like(k)
    dv_sum = np.zeros_like(v)
    for r in range(cp):
        pos = L.rank_positions(T, cp, layout, r)
        o, lse = A.allgather_fwd(q, k, v, scale, pos)
        assert rel_err(o, ro[:, :, pos]) < 1e-13
        assert rel_err(lse, rlse[:, :, pos]) < 1e-13
        dq, dk, dv = A.allgather_bwd(q, k, v, do, scale, pos)
        assert rel_err(dq, rdq[:, :, pos]) < 1e-12
        dk_sum += dk
        dv_sum += dv
    assert rel_err(dk_sum, rdk) < 1e-12
    assert rel_err(dv_sum, rdv) < 1e-12


def test_allgather_rank_share_finite_differences(rng):
    """A rank's K/V gradient is the gradient of its own rows' share of the loss,
    L_r = sum over its rows i of dO_i . O_i (central differences)."""
    T, cp, layout = 8, 2, "zigzag"
    q, k, v, do = _rand(rng, 1, 2, 1, T, 3)
    scale = 0.6
    pos = L.rank_positions(T, cp, layout, 1)
    _, dk, dv = A.allgather_bwd(q, k, v, do, scale, pos)

    def loss(k_, v_):
        o, _ = A.attention_fwd(q, k_, v_, scale)
        return float(np.sum(do[:, :, pos] * o[:, :, pos]))

    eps = 1e-5
    for x, g, which in ((k, dk, 0), (v, dv, 1)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args_p = [k, v]; args_p[which] = xp
            args_m = [k, v]; args_m[which] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        assert rel_err(g, num) < 1e-8, which
    # keys after the rank's last query position get nothing from it
    later = np.arange(T) > pos.max()
    assert np.all(dk[:, :, later] == 0) and np.all(dv[:, :, later] == 0)


# ---------------------------------------------------------------------------
# Packed sequences (position restart at every document)
# ---------------------------------------------------------------------------

def test_packed_equals_documents_alone(rng):
    """Each document of a packed row is attended exactly as if it were a sequence
    of its own (positions restarting at 0); the backward likewise."""
    T, D = 40, 6
    q, k, v, do = _rand(rng, 2, 4, 2, T, D)
    starts = np.array([[0, 7, 7, 23, 40], [0, 1, 19, 33, 40]])   # one empty document
    scale = 0.5
    o, lse = A.packed_attention_fwd(q, k, v, scale, starts)
    dq, dk, dv = A.packed_attention_bwd(q, k, v, do, scale, starts)
    for b in range(2):
        for d in range(starts.shape[1] - 1):
            s0, s1 = starts[b, d], starts[b, d + 1]
            if s1 == s0:
                continue
            sl = slice(s0, s1)
            ro, rl = A.attention_fwd(q[b:b + 1, :, sl], k[b:b + 1, :, sl], v[b:b + 1, :, sl], scale)
            rq, rk, rv = A.attention_bwd(q[b:b + 1, :, sl], k[b:b + 1, :, sl], v[b:b + 1, :, sl],
                                         do[b:b + 1, :, sl], scale)
            assert rel_err(o[b:b + 1, :, sl], ro) < 1e-13
            assert rel_err(lse[b:b + 1, :, sl], rl) < 1e-13
            assert rel_err(dq[b:b + 1, :, sl], rq) < 1e-12
            assert rel_err(dk[b:b + 1, :, sl], rk) < 1e-12
            assert rel_err(dv[b:b + 1, :, sl], rv) < 1e-12


def test_packed_matches_torch_masked_sdpa(rng):
    """The library routine with the packed boolean mask, plus autograd."""
    T, D = 33, 5
    q, k, v, do = _rand(rng, 1, 4, 1, T, D)
    starts = np.array([[0, 10, 11, 33]])
    scale = 0.45
    o, lse = A.packed_attention_fwd(q, k, v, scale, starts)
    dq, dk, dv = A.packed_attention_bwd(q, k, v, do, scale, starts)
    pos = np.arange(T)
    doc = np.searchsorted(starts[0], pos, side="right") - 1
    mask = torch.tensor((pos[None, :] <= pos[:, None]) & (doc[None, :] == doc[:, None]))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kr, vr = tk.repeat_interleave(4, dim=1), tv.repeat_interleave(4, dim=1)
    to = torch.nn.functional.scaled_dot_product_attention(tq, kr, vr, attn_mask=mask, scale=scale)
    (to * torch.tensor(do)).sum().backward()
    s_ = (scale * tq.detach() @ kr.detach().transpose(-1, -2)).masked_fill(~mask, float("-inf"))
    assert rel_err(o, to.detach().numpy()) < 1e-13
    assert rel_err(lse, torch.logsumexp(s_, dim=-1).numpy()) < 1e-13
    assert rel_err(dq, tq.grad.numpy()) < 1e-12
    assert rel_err(dk, tk.grad.numpy()) < 1e-12
    assert rel_err(dv, tv.grad.numpy()) < 1e-12


def test_packed_single_document_is_causal(rng):
    q, k, v, do = _rand(rng, 1, 2, 2, 24, 4)
    starts = np.array([[0, 24]])
    o, lse = A.packed_attention_fwd(q, k, v, 0.3, starts)
    ro, rl = A.attention_fwd(q, k, v, 0.3)
    assert rel_err(o, ro) < 1e-14 and rel_err(lse, rl) < 1e-14
    g = A.packed_attention_bwd(q, k, v, do, 0.3, starts)
    r = A.attention_bwd(q, k, v, do, 0.3)
    for a_, b_ in zip(g, r):
        assert rel_err(a_, b_) < 1e-13
