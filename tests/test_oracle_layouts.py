"""Pins of the oracle's token-to-rank maps (CPU only, integer work, exact)."""
import numpy as np
import pytest

from conftest import read_golden
from oracle import layouts as L
from workloads import Workload


def test_zigzag_assignment_matches_the_page():
    rows = read_golden("zigzag_assignment_cp4.txt")
    cp = int(rows[0][1])
    T = 2 * cp * 5          # any chunk length: 5 tokens per chunk here
    h = T // (2 * cp)
    for r, first, second in ((int(a), int(b), int(c)) for a, b, c in rows[1:]):
        held = L.rank_positions(T, cp, "zigzag", r)
        assert np.array_equal(held[:h], np.arange(first * h, (first + 1) * h))
        assert np.array_equal(held[h:], np.arange(second * h, (second + 1) * h))
    assert L.zigzag_rank_chunks(cp) == [(0, 7), (1, 6), (2, 5), (3, 4)]


@pytest.mark.parametrize("layout,cp,T", [("contiguous", 4, 64), ("zigzag", 4, 64),
                                         ("zigzag", 8, 1024), ("zigzag", 1, 6),
                                         ("contiguous", 1, 5)])
def test_layout_is_a_permutation_and_round_trips(rng, layout, cp, T):
    pos = L.positions(T, cp, layout)
    assert np.array_equal(np.sort(pos), np.arange(T))
    x = rng.standard_normal((2, 3, T, 4))
    assert np.array_equal(L.to_natural(L.to_layout(x, cp, layout), cp, layout), x)
    assert np.array_equal(L.to_layout(L.to_natural(x, cp, layout), cp, layout), x)


def test_zigzag_needs_even_chunks():
    with pytest.raises(ValueError):
        L.positions(60, 8, "zigzag")


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_ring_schedule_visits_every_chunk_once(cp):
    for r in range(cp):
        seen = [L.ring_source(r, i, cp) for i in range(cp)]
        assert sorted(seen) == list(range(cp)) and seen[0] == r
        # what rank r holds at step i+1 is what rank r-1 held at step i (send to next)
        for i in range(cp - 1):
            assert L.ring_source(r, i + 1, cp) == L.ring_source((r - 1) % cp, i, cp)


@pytest.mark.parametrize("T,cp", [(64, 4), (128, 8), (48, 2), (1024, 4)])
def test_attended_pair_counts_closed_forms(T, cp):
    """Brute-force pair counts per (rank, step) against their closed forms.

    contiguous: own chunk c(c+1)/2, an earlier chunk c^2, a later one 0;
    zigzag: own chunk c(c+1)/2 and exactly c^2/2 at every other step, for every
    rank, which is the balance the tutorial's section "Zig-Zag Ring Attention"
    is after.  Both sum to T(T+1)/2.
    """
    c = T // cp
    con = L.attended_pairs(T, cp, "contiguous")
    zz = L.attended_pairs(T, cp, "zigzag")
    for r in range(cp):
        for i in range(cp):
            s = L.ring_source(r, i, cp)
            want = c * (c + 1) // 2 if s == r else (c * c if s < r else 0)
            assert con[r, i] == want
            assert zz[r, i] == (c * (c + 1) // 2 if i == 0 else c * c // 2)
    assert con.sum() == zz.sum() == T * (T + 1) // 2
    if (T, cp) == (64, 4):
        assert zz.tolist() == [[136, 128, 128, 128]] * 4
        assert con[0].tolist() == [136, 0, 0, 0] and con[3].tolist() == [136, 256, 256, 256]


@pytest.mark.parametrize("T,cp", [(64, 4), (96, 4), (128, 8), (40, 2)])
def test_zigzag_exclusion_rule_matches_the_page(T, cp):
    rule = {cond: excl for cond, excl in read_golden("zigzag_exclusion_rule.txt")}
    got = L.zigzag_unused_halves(T, cp)
    for (r, i), (q_head, q_tail, kv_head, kv_tail, partial) in got.items():
        if i == 0:
            cond = "i==0"
        elif i <= r:
            cond = "i<=rank"
        else:
            cond = "i>rank"
        expect = rule[cond]
        assert (q_head, q_tail, kv_head, kv_tail) == (
            expect == "q_first_half", False, False, expect == "kv_second_half"), (r, i)
        # the steps other than i = 0 need no mask inside the used halves
        assert partial == (i == 0), (r, i)


def test_chunk_pair_flops_match_the_page():
    """4*d*c^2 FLOPs for a fully visible chunk pair; the workload accounting
    (4*d per attended pair) reproduces it through the brute-force pair count."""
    for c, d, flops in ((int(a), int(b), int(f)) for a, b, f in read_golden("chunk_pair_flops.txt")):
        T, cp = 2 * c, 2
        pairs = L.attended_pairs(T, cp, "contiguous")
        assert pairs[1, 1] == c * c           # rank 1 at step 1 holds the earlier chunk
        assert 4 * d * pairs[1, 1] == flops
        w = Workload("x", 1, 1, 1, T, d, cp, "contiguous", "bf16")
        assert w.fwd_flops == 4 * d * pairs.sum()


# ------------------------------------------------------------------ a2a ----

@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("B,H,T,cp,a2a", [(1, 8, 64, 8, 2), (2, 4, 32, 4, 2), (1, 6, 48, 6, 3),
                                          (1, 4, 16, 2, 2), (1, 4, 32, 4, 1),
                                          # full Ulysses (a2a = cp, p2p = 1)
                                          (1, 8, 64, 4, 4), (2, 8, 64, 8, 8)])
def test_a2a_round_trip_and_structure(rng, B, H, T, cp, a2a, layout):
    D = 3
    nat = rng.standard_normal((B, H, T, D))
    src = L.token_shards(nat, cp, layout)
    dst = L.a2a_forward(src, B, H, T, cp, a2a, layout)
    assert np.array_equal(L.a2a_inverse(dst, B, H, T, cp, a2a, layout), src)
    p2p = cp // a2a
    Hs = H // a2a
    # slice j holds heads [j*Hs, (j+1)*Hs) of every token, token axis in the
    # layout order of a zigzag ring over p2p ranks
    for j in range(a2a):
        want = L.to_layout(nat[:, j * Hs:(j + 1) * Hs], p2p, layout)
        assert np.array_equal(dst[j], want)
    # p2p rank k's slots hold exactly the tokens of a2a group k's cp ranks
    groups, rings = L.a2a_groups(cp, a2a)
    c_p = T // p2p
    dst_pos = L.positions(T, p2p, layout)
    for k, grp in enumerate(groups):
        held = np.concatenate([L.rank_positions(T, cp, layout, r) for r in grp])
        assert np.array_equal(np.sort(dst_pos[k * c_p:(k + 1) * c_p]), np.sort(held))
    assert all(len(r_) == p2p for r_ in rings)


def test_a2a_index_is_a_bijection():
    idx = L.a2a_source_rows(2, 8, 64, 8, 2)
    flat = np.sort(idx.reshape(-1))
    assert np.array_equal(flat, np.arange(2 * 8 * 64))
