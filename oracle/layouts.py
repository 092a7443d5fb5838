"""Token-to-rank maps of context parallelism, in plain numpy (integer work).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Layout order" is the token axis as the emulated ranks hold it: rank r owns the
slots [r*c, (r+1)*c) with c = T / cp.  ``positions(...)[t]`` is the natural
(global) position of the token stored in layout slot t.

* contiguous (pull request "Feat: Context Parallel" #181, the default layout):
  rank r holds the r-th contiguous slice of length c.
* zigzag (tutorial "上下文并行", section "Zig-Zag Ring Attention"): the sequence is
  cut into 2*cp chunks of length c/2 numbered 0..2cp-1; rank r holds chunk r and
  chunk 2cp-1-r, in that order (cp = 4: [0,7], [1,6], [2,5], [3,4]).
* ring schedule (tutorial, section "朴素 Ring Attention": each step a rank sends
  its K/V to the next rank and receives from the previous one): at step i rank r
  holds the K/V chunk of rank (r - i) mod cp.
* all-to-all re-layout of the hierarchical mode (pull request #181, mode
  "a2a+p2p"; tutorial, section "Ulysses CP"): the cp ranks are split into a2a
  groups of ``a2a`` consecutive ranks; inside a group an all-to-all turns each
  rank's token shard (all heads) into a head shard (H / a2a contiguous heads) of
  all the group's tokens; the ring then runs over the cp / a2a groups.
"""
from __future__ import annotations

import numpy as np


def chunk_len(T: int, cp: int) -> int:
    if T % cp:
        raise ValueError("T must be divisible by cp")
    return T // cp


def zigzag_rank_chunks(cp: int):
    """Pairs (head chunk, tail chunk) held by each rank, chunks of length T/(2cp)."""
    return [(r, 2 * cp - 1 - r) for r in range(cp)]


def positions(T: int, cp: int, layout: str) -> np.ndarray:
    """Natural position of the token in each layout slot (a permutation of 0..T-1)."""
    if layout == "contiguous":
        chunk_len(T, cp)
        return np.arange(T)
    if layout != "zigzag":
        raise ValueError(layout)
    if T % (2 * cp):
        raise ValueError("zigzag needs T divisible by 2*cp")
    h = T // (2 * cp)
    out = []
    for head, tail in zigzag_rank_chunks(cp):
        out.append(np.arange(head * h, (head + 1) * h))
        out.append(np.arange(tail * h, (tail + 1) * h))
    return np.concatenate(out)


def layout_slots(T: int, cp: int, layout: str) -> np.ndarray:
    """Inverse map: layout slot of each natural position."""
    pos = positions(T, cp, layout)
    inv = np.empty_like(pos)
    inv[pos] = np.arange(T)
    return inv


def to_layout(x_natural, cp: int, layout: str, axis: int = 2):
    """Gather a natural-order tensor into layout order along ``axis``."""
    T = x_natural.shape[axis]
    return np.take(x_natural, positions(T, cp, layout), axis=axis)


def to_natural(x_layout, cp: int, layout: str, axis: int = 2):
    """Gather a layout-order tensor back into natural order along ``axis``."""
    T = x_layout.shape[axis]
    return np.take(x_layout, layout_slots(T, cp, layout), axis=axis)


def rank_positions(T: int, cp: int, layout: str, r: int) -> np.ndarray:
    c = chunk_len(T, cp)
    return positions(T, cp, layout)[r * c:(r + 1) * c]


def ring_source(r: int, i: int, cp: int) -> int:
    """Rank whose K/V chunk rank r holds at ring step i."""
    return (r - i) % cp


def attended_pairs(T: int, cp: int, layout: str) -> np.ndarray:
    """Brute force: visible (q, k) pairs per [rank, step] for one head."""
    out = np.zeros((cp, cp), dtype=np.int64)
    for r in range(cp):
        qp = rank_positions(T, cp, layout, r)
        for i in range(cp):
            kp = rank_positions(T, cp, layout, ring_source(r, i, cp))
            out[r, i] = int(np.sum(kp[None, :] <= qp[:, None]))
    return out


def zigzag_unused_halves(T: int, cp: int):
    """Brute force of the zigzag per-step exclusion rule.

    For each (rank r, step i) returns (q_head_unused, q_tail_unused,
    kv_head_unused, kv_tail_unused, partially_masked): a half is "unused" when
    none of its tokens takes part in a visible pair of that step, and
    partially_masked says whether any pair inside the used halves is hidden.
    """
    h = T // (2 * cp)
    res = {}
    for r in range(cp):
        qp = rank_positions(T, cp, "zigzag", r)
        for i in range(cp):
            kp = rank_positions(T, cp, "zigzag", ring_source(r, i, cp))
            vis = kp[None, :] <= qp[:, None]
            q_used = vis.any(axis=1)
            k_used = vis.any(axis=0)
            used = vis[np.ix_(q_used, k_used)]
            res[(r, i)] = (not q_used[:h].any(), not q_used[h:].any(),
                           not k_used[:h].any(), not k_used[h:].any(),
                           bool(used.size and not used.all()))
    return res


# ----------------------------------------------------------------------------
# all-to-all (Ulysses) re-layout of the hierarchical a2a x p2p mode
# ----------------------------------------------------------------------------

def a2a_groups(cp: int, a2a: int):
    """a2a groups of consecutive ranks, and the p2p rings across them."""
    if cp % a2a:
        raise ValueError("a2a must divide cp")
    p2p = cp // a2a
    groups = [list(range(a2a * k, a2a * (k + 1))) for k in range(p2p)]
    rings = [[a2a * k + j for k in range(p2p)] for j in range(a2a)]
    return groups, rings


def a2a_source_rows(B: int, H: int, T: int, cp: int, a2a: int,
                    layout: str = "zigzag") -> np.ndarray:
    """Flat source row of every destination row of the a2a re-layout.

    Source (token-sharded, what each of the cp ranks holds before the
    all-to-all): [cp][B][T/cp][H] rows of D values, rank r's T/cp tokens being its
    share over cp in ``layout`` (zigzag: chunks r and 2cp-1-r of length T/(2cp)).
    Destination (head-sharded, after the all-to-all): [a2a][B][H/a2a][T] rows,
    where slice j holds heads [j*H/a2a, (j+1)*H/a2a) and its token axis is the
    layout order of a ring over p2p = cp/a2a ranks in the same ``layout``: p2p
    rank k (a2a group k) owns slots [k*T/p2p, (k+1)*T/p2p) (zigzag: the p2p
    chunks k and 2*p2p-1-k of length T/(2*p2p)).
    Returns an int64 array of shape [a2a, B, H/a2a, T].
    """
    if H % a2a:
        raise ValueError("heads must be divisible by a2a")
    p2p = cp // a2a
    Hs = H // a2a
    c_src = T // cp
    # natural position -> (source rank, slot within rank)
    src_rank = np.empty(T, dtype=np.int64)
    src_slot = np.empty(T, dtype=np.int64)
    for r in range(cp):
        pos_r = rank_positions(T, cp, layout, r)
        src_rank[pos_r] = r
        src_slot[pos_r] = np.arange(c_src)
    dst_pos = positions(T, p2p, layout)        # natural position of each dst slot
    out = np.empty((a2a, B, Hs, T), dtype=np.int64)
    for j in range(a2a):
        for b in range(B):
            for hh in range(Hs):
                hglob = j * Hs + hh
                r = src_rank[dst_pos]
                s = src_slot[dst_pos]
                out[j, b, hh] = ((r * B + b) * c_src + s) * H + hglob
    return out


def a2a_forward(src, B, H, T, cp, a2a, layout="zigzag"):
    """Apply the re-layout to a source array of shape [cp, B, T/cp, H, D]."""
    D = src.shape[-1]
    flat = src.reshape(-1, D)
    idx = a2a_source_rows(B, H, T, cp, a2a, layout)
    return flat[idx.reshape(-1)].reshape(a2a, B, H // a2a, T, D)


def a2a_inverse(dst, B, H, T, cp, a2a, layout="zigzag"):
    """Undo the re-layout: [a2a, B, H/a2a, T, D] -> [cp, B, T/cp, H, D]."""
    D = dst.shape[-1]
    idx = a2a_source_rows(B, H, T, cp, a2a, layout).reshape(-1)
    out = np.empty((cp * B * (T // cp) * H, D), dtype=dst.dtype)
    out[idx] = dst.reshape(-1, D)
    return out.reshape(cp, B, T // cp, H, D)


def token_shards(x_natural_bhtd, cp, layout="zigzag"):
    """Natural [B, H, T, D] -> the cp ranks' token shards [cp, B, T/cp, H, D]."""
    B, H, T, D = x_natural_bhtd.shape
    c = T // cp
    out = np.empty((cp, B, c, H, D), dtype=x_natural_bhtd.dtype)
    for r in range(cp):
        pos_r = rank_positions(T, cp, layout, r)
        out[r] = np.transpose(x_natural_bhtd[:, :, pos_r, :], (0, 2, 1, 3))
    return out
