"""Unshared full-sequence causal attention -- the plain definition, float64.

Source: the openjev-sglang article (jdon.com), sections on the radix cache and
on counting the N+1 prefills (the shared prefix is computed once, each branch
prefill reuses its KV and computes only the suffix), and the LLM2Jev "shared
prefix" page, section on reusing SGLang's radix cache (a branch continues from
the cached prefix; the result is that of processing the full input).  Reuse
changes where work happens, not what is computed, so the oracle recomputes
every branch's whole token sequence on its own:

    s_ij  = q_i . k_j / sqrt(d)            for keys j <= i (causal), else -inf
    p_ij  = exp(s_ij - max_j s_ij)
    o_i   = sum_j p_ij v_j / sum_j p_ij
    lse_i = max_j s_ij + ln sum_j p_ij     (natural log)

Readings where the pages are silent: scale 1/sqrt(d); grouped-query attention
with contiguous groups (query head h reads KV head h // (Hq / Hkv)); no
positional encoding inside the layer (q and k are given post-rotary).

Parity: pinned by a brute-force scalar loop, by the library scaled-dot-product
attention in float64, and by closed forms (single key, equal keys, prefix-free
sequence) in ``tests/test_oracle_attention.py``.
"""
from __future__ import annotations

import math

import numpy as np


def to64(t) -> np.ndarray:
    """bf16/fp32 torch tensor (or array) -> float64 numpy, exactly."""
    if hasattr(t, "detach"):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """q [L, Hq, d], k/v [L, Hkv, d] (float64) -> out [L, Hq, d], lse [L, Hq]."""
    L, Hq, d = q.shape
    Hkv = k.shape[1]
    assert Hq % Hkv == 0
    group = Hq // Hkv
    scale = 1.0 / math.sqrt(d)
    out = np.empty((L, Hq, d))
    lse = np.empty((L, Hq))
    future = np.triu(np.ones((L, L), dtype=bool), 1)
    for hq in range(Hq):
        g = hq // group
        s = (q[:, hq, :] @ k[:, g, :].T) * scale
        s[future] = -np.inf
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        out[:, hq, :] = (p @ v[:, g, :]) / l
        lse[:, hq] = m[:, 0] + np.log(l[:, 0])
    return out, lse


def attention_at(q_row: np.ndarray, k: np.ndarray, v: np.ndarray):
    """One query position against keys k/v [n, Hkv, d] (all visible).

    q_row [Hq, d] -> out [Hq, d], lse [Hq].  Used for sampled rows of large
    workloads: the row's visible keys are exactly its branch's first n tokens.
    """
    Hq, d = q_row.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    scale = 1.0 / math.sqrt(d)
    out = np.empty((Hq, d))
    lse = np.empty(Hq)
    for hq in range(Hq):
        g = hq // group
        s = (k[:, g, :] @ q_row[hq]) * scale
        m = s.max()
        p = np.exp(s - m)
        l = p.sum()
        out[hq] = (p @ v[:, g, :]) / l
        lse[hq] = m + math.log(l)
    return out, lse


def branch_rows(plan, b: int) -> np.ndarray:
    """Node-token rows of branch b's full sequence, in token order."""
    rows = []
    for sid in plan.paths[b]:
        s = plan.segments[sid]
        rows.append(np.arange(s.node_start, s.node_start + s.length))
    return np.concatenate(rows)


def reference_attention(plan, q, k, v, branches=None):
    """Recomputes each branch's full sequence without sharing.

    Returns (out [T, Hq, d], lse [T, Hq], max_disagreement) in node-token
    layout.  Rows shared by several branches are produced by each of them;
    ``max_disagreement`` is the largest difference between those copies (it is
    zero up to float64 rounding, since a shared row sees the same keys in every
    branch).  Rows of branches not listed stay NaN.
    """
    q64, k64, v64 = to64(q), to64(k), to64(v)
    T, Hq, d = q64.shape
    out = np.full((T, Hq, d), np.nan)
    lse = np.full((T, Hq), np.nan)
    worst = 0.0
    for b in (range(len(plan.paths)) if branches is None else branches):
        rows = branch_rows(plan, b)
        o, l = causal_attention(q64[rows], k64[rows], v64[rows])
        seen = ~np.isnan(lse[rows, 0])
        if seen.any():
            worst = max(worst, float(np.abs(out[rows][seen] - o[seen]).max()))
        out[rows] = o
        lse[rows] = l
    return out, lse, worst


def branch_suffix_attention(plan, q, k, v, b: int):
    """The rows of branch b's own last segment (its suffix), each attending
    causally over the branch's whole sequence: the last rows of
    ``causal_attention`` on that sequence, computed for those rows only (the
    other rows of the sequence are not needed, so a large workload's every
    suffix row stays affordable).  The query heads of one KV head are stacked
    into one matrix product per KV head; each score still is q.k / sqrt(d).

    Returns (node rows [S], out [S, Hq, d], lse [S, Hq]).
    """
    rows = branch_rows(plan, b)
    leaf = plan.segments[plan.paths[b][-1]]
    S = leaf.length
    L = len(rows)
    P = L - S
    qs = to64(q[rows[P:]])                    # [S, Hq, d]
    kk, vv = to64(k[rows]), to64(v[rows])     # [L, Hkv, d]
    _, Hq, d = qs.shape
    Hkv = kk.shape[1]
    group = Hq // Hkv
    scale = 1.0 / math.sqrt(d)
    # query i of the suffix sits at position P + i and sees keys 0 .. P + i
    future = np.arange(L)[None, :] > (P + np.arange(S))[:, None]          # [S, L]
    future = np.repeat(future, group, axis=0)                              # [S * group, L]
    out = np.empty((S, Hq, d))
    lse = np.empty((S, Hq))
    for g in range(Hkv):
        qg = qs[:, g * group:(g + 1) * group, :].reshape(S * group, d)
        sc = (qg @ kk[:, g, :].T) * scale
        sc[future] = -np.inf
        m = sc.max(axis=1, keepdims=True)
        p = np.exp(sc - m)
        l = p.sum(axis=1, keepdims=True)
        out[:, g * group:(g + 1) * group, :] = ((p @ vv[:, g, :]) / l).reshape(S, group, d)
        lse[:, g * group:(g + 1) * group] = (m[:, 0] + np.log(l[:, 0])).reshape(S, group)
    return rows[P:], out, lse


def sampled_attention(plan, q, k, v, rows):
    """Output rows for selected node-token rows (any size of workload).

    Row r belongs to a segment; the row is evaluated in the sequence of the
    segment's first member branch: keys are that branch's tokens up to and
    including r.
    """
    q_, k_, v_ = q, k, v
    seg_of_row = {}
    starts = np.array([s.node_start for s in plan.segments])
    res_o = []
    res_l = []
    for r in rows:
        sid = int(np.searchsorted(starts, r, side="right") - 1)
        if sid not in seg_of_row:
            b = plan.segments[sid].members[0]
            seg_of_row[sid] = branch_rows(plan, b)
        brow = seg_of_row[sid]
        pos = int(np.nonzero(brow == r)[0][0])
        keys = brow[:pos + 1]
        o, l = attention_at(to64(q_[r]), to64(k_[keys]), to64(v_[keys]))
        res_o.append(o)
        res_l.append(l)
    return np.stack(res_o), np.stack(res_l)
