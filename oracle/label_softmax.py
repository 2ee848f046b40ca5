"""Stable softmax over each branch's label logprobs, and the argmax label.

Source: the openjev-sglang article (jdon.com), request-flow step 5 and the
worked refund example in the prefill-only section: the label logprobs that
come back (yes -0.3, no -1.5) are renormalised with a numerically stable
softmax into P(yes) = 0.77, P(no) = 0.23.

    p_j = exp(lp_j - max lp) / sum_i exp(lp_i - max lp)

argmax: the label with the largest probability; on exact ties, the lowest
label index (reading: the pages do not say; this is the usual convention).

Parity: pinned by the printed worked example (tests/golden), by sum-to-one,
by scipy.special.softmax and by tie handling.
"""
from __future__ import annotations

import numpy as np


def label_softmax(lp, label_off):
    lp = np.asarray(lp, dtype=np.float64)
    label_off = np.asarray(label_off)
    probs = np.empty_like(lp)
    N = len(label_off) - 1
    argmax = np.empty(N, dtype=np.int32)
    for n in range(N):
        a, b = int(label_off[n]), int(label_off[n + 1])
        x = lp[a:b]
        m = x.max()
        e = np.exp(x - m)
        probs[a:b] = e / e.sum()
        argmax[n] = int(np.argmax(x))  # first index among equal maxima
    return probs, argmax


def top2_margin(probs, label_off):
    """Per branch: largest minus second-largest probability (inf if one label)."""
    probs = np.asarray(probs)
    out = []
    for n in range(len(label_off) - 1):
        x = np.sort(probs[label_off[n]:label_off[n + 1]])[::-1]
        out.append(x[0] - x[1] if len(x) > 1 else np.inf)
    return np.array(out)
