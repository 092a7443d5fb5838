"""Plain FP64 causal attention, its analytic backward, and the (O, LSE) merge.

TEST INFRASTRUCTURE ONLY (see the package docstring).

All arrays are numpy float64 in NATURAL token order:
  q, o, dO : [B, H_q, T, D]      k, v : [B, H_kv, T, D]      lse : [B, H_q, T]
Query head h reads key/value head g = h // n_rep with n_rep = H_q // H_kv: the
grouped-query view reshapes the H_q heads as (H_q / n_rep, n_rep) with the n_rep
copies innermost, and its backward sums over that innermost axis (pull request
"Feat: Context Parallel" #181, review thread on ``RepeatKVHeads``).

Definitions used (tutorial "上下文并行", section "朴素 Ring Attention"):
  S_ij = scale * q_i . k_j                           (scale = 1/sqrt(d) by default)
  causal: key j is visible to query i iff j <= i      (section "Zig-Zag Ring
          Attention": token i sees [1, i]); hidden entries contribute exactly 0
  m_i  = max over visible j of S_ij                   (safe softmax: subtract the max)
  P_ij = exp(S_ij - m_i) / sum_j' exp(S_ij' - m_i)
  O_i  = sum_j P_ij v_j,   LSE_i = m_i + ln(sum_j exp(S_ij - m_i))
Backward (softmax calculus; the pull request recomputes P in the backward):
  Delta_i = dO_i . O_i,  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - Delta_i)
  dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i
with dK, dV summed over the n_rep query heads of a group.

Rows are processed in blocks of whole rows; every row is computed from the
definition above with a two-pass max/sum over all of its keys.  Nothing here uses
an online (running) softmax except ``merge``, which is the merge rule itself.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _group(H_q: int, H_kv: int) -> int:
    if H_q % H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    return H_q // H_kv


def scores(q_rows, k_all, scale):
    """S = scale * Q K^T for a block of query rows against all keys."""
    return scale * (q_rows @ k_all.T)


def causal_visible(q_pos, k_pos):
    """Boolean [len(q_pos), len(k_pos)]: key visible iff its position <= the query's."""
    return np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]


def safe_softmax_rows(S, visible):
    """Row-wise safe softmax over the visible entries.

    Returns (P, m, l) with P_ij = exp(S_ij - m_i) / l_i on visible entries and
    exactly 0 elsewhere; m_i = row max, l_i = sum_j exp(S_ij - m_i).  A row with
    no visible entry gets P = 0, m = -inf, l = 0.
    """
    Sm = np.where(visible, S, NEG_INF)
    m = Sm.max(axis=1)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    E = np.where(visible, np.exp(Sm - m_safe[:, None]), 0.0)
    l = E.sum(axis=1)
    P = np.zeros_like(E)
    P[has] = E[has] / l[has, None]
    return P, m, l


def _row_blocks(T, rows_per_block):
    for r0 in range(0, T, rows_per_block):
        yield r0, min(T, r0 + rows_per_block)


def attention_fwd(q, k, v, scale, rows_per_block=1024):
    """Causal attention forward in natural order.  Returns (O, LSE)."""
    B, H_q, T, D = q.shape
    n_rep = _group(H_q, k.shape[1])
    o = np.empty_like(q)
    lse = np.empty((B, H_q, T))
    pos = np.arange(T)
    for b in range(B):
        for h in range(H_q):
            g = h // n_rep
            for r0, r1 in _row_blocks(T, rows_per_block):
                S = scores(q[b, h, r0:r1], k[b, g], scale)
                P, m, l = safe_softmax_rows(S, causal_visible(pos[r0:r1], pos))
                o[b, h, r0:r1] = P @ v[b, g]
                lse[b, h, r0:r1] = m + np.log(l)
    return o, lse


def attention_bwd(q, k, v, do, scale, rows_per_block=1024):
    """Analytic backward of causal attention in natural order.

    The probabilities and the output are recomputed from the definition (no
    saved statistics are consumed).  Returns (dQ, dK, dV).
    """
    B, H_q, T, D = q.shape
    n_rep = _group(H_q, k.shape[1])
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    pos = np.arange(T)
    for b in range(B):
        for h in range(H_q):
            g = h // n_rep
            for r0, r1 in _row_blocks(T, rows_per_block):
                S = scores(q[b, h, r0:r1], k[b, g], scale)
                P, _, _ = safe_softmax_rows(S, causal_visible(pos[r0:r1], pos))
                O = P @ v[b, g]
                dO = do[b, h, r0:r1]
                delta = np.sum(dO * O, axis=1)
                dP = dO @ v[b, g].T
                dS = P * (dP - delta[:, None])
                dq[b, h, r0:r1] = scale * (dS @ k[b, g])
                dk[b, g] += scale * (dS.T @ q[b, h, r0:r1])
                dv[b, g] += P.T @ dO
    return dq, dk, dv


def partial_attention(q_rows, k_rows, v_rows, q_pos, k_pos, scale):
    """Attention of a set of query rows over one set of key/value rows.

    This is one ring step's partial result (tutorial, section "朴素 Ring
    Attention": partial_i = Softmax(Q_i K^T / sqrt(d)) V over the K/V block held
    at that step), with the causal mask taken from GLOBAL positions.
    q_rows [n, D], k_rows/v_rows [m, D].  Returns (O [n, D], LSE [n]); a row with
    no visible key gets O = 0 and LSE = -inf (the identity of ``merge``).
    """
    S = scores(q_rows, k_rows, scale)
    P, m, l = safe_softmax_rows(S, causal_visible(q_pos, k_pos))
    o = P @ v_rows
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)
    return o, lse


def partial_attention_bwd(q_rows, k_rows, v_rows, do_rows, o_rows, lse_rows, q_pos, k_pos,
                          scale):
    """One ring step's gradient contributions: a set of query rows against one set
    of key/value rows.

    The backward of the tutorial's section "朴素 Ring Attention" recomputes each
    step's probabilities; the pull request's "p2p" mode sends each K/V chunk's
    gradient around the ring with the chunk.  Per step that is the analytic
    softmax backward restricted to the keys held at the step, with the WHOLE
    forward's statistics: P_ij = exp(S_ij - LSE_i) for visible pairs (global
    positions) and 0 otherwise, Delta_i = dO_i . O_i with the whole forward's
    output, dP_ij = dO_i . v_j, dS_ij = P_ij (dP_ij - Delta_i).
    q_rows, do_rows, o_rows [n, D], lse_rows [n], k_rows, v_rows [m, D].
    Returns (dq [n, D], dk [m, D], dv [m, D]): the block's contribution to the
    rows' dQ, and the rows' contribution to the keys' dK and dV.  Over a
    partition of the keys the dq contributions add up to the rows' dQ; over a
    partition of the queries the dk, dv contributions add up to the keys' dK, dV.
    """
    S = scores(q_rows, k_rows, scale)
    vis = causal_visible(q_pos, k_pos)
    P = np.where(vis, np.exp(np.where(vis, S, 0.0) - np.asarray(lse_rows)[:, None]), 0.0)
    delta = np.sum(do_rows * o_rows, axis=1)
    dP = do_rows @ v_rows.T
    dS = P * (dP - delta[:, None])
    return scale * (dS @ k_rows), scale * (dS.T @ q_rows), P.T @ do_rows


def merge(o_a, lse_a, o_b, lse_b):
    """Merge two normalised partial results over disjoint key sets.

    LSE = ln(e^LSE_a + e^LSE_b) and O = e^(LSE_a - LSE) O_a + e^(LSE_b - LSE) O_b,
    evaluated in the max-shifted form; merging with an empty partial
    (LSE = -inf) returns the other operand, and two empty partials give (0, -inf).
    This is the running-max/running-sum update of the tutorial's section
    "朴素 Ring Attention" (the order of the K/V blocks does not matter as long as
    the current O, max and sum are carried) written for (O, LSE) pairs.
    """
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    m = np.maximum(lse_a, lse_b)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    wa = np.where(finite, np.exp(lse_a - m_safe), 0.0)
    wb = np.where(finite, np.exp(lse_b - m_safe), 0.0)
    s = wa + wb
    s_safe = np.where(finite, s, 1.0)
    with np.errstate(divide="ignore"):
        lse = np.where(finite, m_safe + np.log(s_safe), NEG_INF)
    o = (wa / s_safe)[..., None] * o_a + (wb / s_safe)[..., None] * o_b
    o = np.where(finite[..., None], o, 0.0)
    return o, lse


# ----------------------------------------------------------------------------
# Sampled rows for problems too large to compute whole on the host.
# Every value is still the plain definition for that row (all of its keys).
# ----------------------------------------------------------------------------

def fwd_rows(q_h, k_g, v_g, rows, scale):
    """(O, LSE) of the given natural-order query rows of one head.

    q_h [T, D] (one query head), k_g/v_g [T, D] (its key/value head).
    """
    rows = np.asarray(rows)
    T = k_g.shape[0]
    S = scores(q_h[rows], k_g, scale)
    P, m, l = safe_softmax_rows(S, causal_visible(rows, np.arange(T)))
    return P @ v_g, m + np.log(l)


def dq_rows(q_h, k_g, v_g, do_h, rows, scale):
    """dQ of the given natural-order query rows of one head (definition above)."""
    rows = np.asarray(rows)
    T = k_g.shape[0]
    S = scores(q_h[rows], k_g, scale)
    P, _, _ = safe_softmax_rows(S, causal_visible(rows, np.arange(T)))
    O = P @ v_g
    dO = do_h[rows]
    delta = np.sum(dO * O, axis=1)
    dS = P * (dO @ v_g.T - delta[:, None])
    return scale * (dS @ k_g)


def dkdv_rows(q_heads, k_g, v_g, do_heads, kv_rows, scale, rows_per_block=512):
    """dK and dV of the given natural-order key rows of one key/value head.

    q_heads/do_heads [n_rep, T, D] are the query heads of the group.  Only query
    rows i >= min(kv_rows) can see these keys, so only those rows are formed (in
    full, with all of their keys).
    """
    kv_rows = np.asarray(kv_rows)
    T = k_g.shape[0]
    j0 = int(kv_rows.min())
    dk = np.zeros((len(kv_rows), k_g.shape[1]))
    dv = np.zeros_like(dk)
    pos = np.arange(T)
    for h in range(q_heads.shape[0]):
        for r0, r1 in _row_blocks(T - j0, rows_per_block):
            rows = pos[j0 + r0:j0 + r1]
            S = scores(q_heads[h, rows], k_g, scale)
            P, _, _ = safe_softmax_rows(S, causal_visible(rows, pos))
            O = P @ v_g
            dO = do_heads[h, rows]
            delta = np.sum(dO * O, axis=1)
            dS = P * (dO @ v_g.T - delta[:, None])
            dk += scale * (dS[:, kv_rows].T @ q_heads[h, rows])
            dv += P[:, kv_rows].T @ dO
    return dk, dv


# ----------------------------------------------------------------------------
# All-gather mode (pull request "Feat: Context Parallel" #181, mode table row
# "all_gather": every rank gathers the whole sequence's K/V and runs attention of
# its own query chunk over it; the backward sums the K/V gradients of all ranks
# with a ReduceScatter.  Tutorial "上下文并行", section "Zig-Zag Ring Attention 的
# 通信与计算重叠", bullet "all-gather": one all-gather gives every GPU the complete
# K/V at once).  A rank's result is the definition above restricted to its query
# rows; its K/V gradient is the part of the sums over i that runs over its rows.
# ----------------------------------------------------------------------------

def allgather_fwd(q, k, v, scale, q_pos):
    """(O, LSE) of the query rows at natural positions ``q_pos`` over all keys.

    q [B, H_q, T, D], k/v [B, H_kv, T, D] in natural order; ``q_pos`` lists the
    rank's query positions (in the order its rows are stored).  Returns
    O [B, H_q, n, D] and LSE [B, H_q, n] with n = len(q_pos).
    """
    q_pos = np.asarray(q_pos)
    B, H_q, T, D = q.shape
    n_rep = _group(H_q, k.shape[1])
    o = np.empty((B, H_q, len(q_pos), D))
    lse = np.empty((B, H_q, len(q_pos)))
    pos = np.arange(T)
    for b in range(B):
        for h in range(H_q):
            g = h // n_rep
            S = scores(q[b, h, q_pos], k[b, g], scale)
            P, m, l = safe_softmax_rows(S, causal_visible(q_pos, pos))
            o[b, h] = P @ v[b, g]
            lse[b, h] = m + np.log(l)
    return o, lse


def allgather_bwd(q, k, v, do, scale, q_pos):
    """One rank's backward in all-gather mode.

    ``q_pos`` are the rank's query positions (natural order indices) and
    ``do`` [B, H_q, T, D] the upstream gradient in natural order (only the rows
    at ``q_pos`` are read).  Returns (dQ [B, H_q, n, D] of the rank's rows,
    dK_part, dV_part [B, H_kv, T, D]): the K/V gradient sums of the definition
    with i running over the rank's rows only, which the ReduceScatter adds up over
    the ranks.
    """
    q_pos = np.asarray(q_pos)
    B, H_q, T, D = q.shape
    n_rep = _group(H_q, k.shape[1])
    dq = np.zeros((B, H_q, len(q_pos), D))
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    pos = np.arange(T)
    for b in range(B):
        for h in range(H_q):
            g = h // n_rep
            S = scores(q[b, h, q_pos], k[b, g], scale)
            P, _, _ = safe_softmax_rows(S, causal_visible(q_pos, pos))
            O = P @ v[b, g]
            dO = do[b, h, q_pos]
            delta = np.sum(dO * O, axis=1)
            dS = P * (dO @ v[b, g].T - delta[:, None])
            dq[b, h] = scale * (dS @ k[b, g])
            dk[b, g] += scale * (dS.T @ q[b, h, q_pos])
            dv[b, g] += P.T @ dO
    return dq, dk, dv


# ----------------------------------------------------------------------------
# Packed sequences (transformers pull request #50497, the packed variant of the
# context-parallel tests: position_ids restart mid-sequence, and the mask has to
# be rebuilt for the packed documents; InfiniTrain pull request #181 lists packed /
# variable-length sequences as not covered).  Every batch row holds n_docs
# documents back to back, document d at natural positions [starts[b, d],
# starts[b, d + 1]); a token attends to the keys of its own document at or before
# it: causal attention with the position restarting at every document.
# ----------------------------------------------------------------------------

def doc_of(starts_row, pos):
    """Document index of each natural position (starts_row: [n_docs + 1])."""
    return np.searchsorted(np.asarray(starts_row), np.asarray(pos), side="right") - 1


def packed_visible(q_pos, k_pos, starts_row):
    """Boolean [len(q_pos), len(k_pos)]: causal and in the same document."""
    dq = doc_of(starts_row, q_pos)
    dk = doc_of(starts_row, k_pos)
    return causal_visible(q_pos, k_pos) & (dk[None, :] == dq[:, None])


def packed_attention_fwd(q, k, v, scale, starts):
    """Forward of packed causal attention in natural order; starts [B, n_docs + 1]."""
    B, H_q, T, D = q.shape
    n_rep = _group(H_q, k.shape[1])
    o = np.empty_like(q)
    lse = np.empty((B, H_q, T))
    pos = np.arange(T)
    for b in range(B):
        vis = packed_visible(pos, pos, starts[b])
        for h in range(H_q):
            g = h // n_rep
            P, m, l = safe_softmax_rows(scores(q[b, h], k[b, g], scale), vis)
            o[b, h] = P @ v[b, g]
            lse[b, h] = m + np.log(l)
    return o, lse


def packed_attention_bwd(q, k, v, do, scale, starts):
    """Analytic backward of packed causal attention (definition as above, with the
    packed mask).  Returns (dQ, dK, dV)."""
    B, H_q, T, D = q.shape
    n_rep = _group(H_q, k.shape[1])
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    pos = np.arange(T)
    for b in range(B):
        vis = packed_visible(pos, pos, starts[b])
        for h in range(H_q):
            g = h // n_rep
            P, _, _ = safe_softmax_rows(scores(q[b, h], k[b, g], scale), vis)
            O = P @ v[b, g]
            delta = np.sum(do[b, h] * O, axis=1)
            dS = P * (do[b, h] @ v[b, g].T - delta[:, None])
            dq[b, h] = scale * (dS @ k[b, g])
            dk[b, g] += scale * (dS.T @ q[b, h])
            dv[b, g] += P.T @ do[b, h]
    return dq, dk, dv
