"""Final-position label log-probabilities -- the plain definition, float64.

Source: the openjev-sglang article (jdon.com), section on what prefill-only
means: the engine runs one forward pass with at most one new token (which is
discarded), and returns the log-probabilities of the requested label token ids
at the last prompt position.  A log-probability is the log-softmax of the
logits over the whole vocabulary:

    logits[n, :] = W h_n
    lse[n]       = ln sum_v exp(logits[n, v])
    lp[n, j]     = logits[n, id_j] - lse[n]

The matmul is a library primitive (numpy, float64), evaluated over slices of
the vocabulary only to bound memory (each logit is an independent dot
product; no arithmetic changes).  The log-sum-exp subtracts the row maximum
before exponentiating, the textbook stable form.

Readings: duplicate label ids inside one branch are allowed and read out
independently; label sets are given as CSR (offsets, ids).

Parity: pinned in ``tests/test_oracle_readout.py`` by W = 0 (lp = -ln V), by
torch.logsumexp / scipy log_softmax in float64, by the shift invariance of
log-softmax and by a dominant label (lp -> 0).
"""
from __future__ import annotations

import numpy as np

from .attention import to64


def full_logits(h, W, branches=None, chunk: int = 8192) -> np.ndarray:
    h64 = to64(h)
    if branches is not None:
        h64 = h64[np.asarray(branches)]
    V = W.shape[0]
    logits = np.empty((h64.shape[0], V))
    for v0 in range(0, V, chunk):
        v1 = min(V, v0 + chunk)
        logits[:, v0:v1] = h64 @ to64(W[v0:v1]).T
    return logits


def log_sum_exp(logits: np.ndarray) -> np.ndarray:
    m = logits.max(axis=1)
    return m + np.log(np.exp(logits - m[:, None]).sum(axis=1))


def label_logprobs(h, W, label_off, label_ids, branches=None):
    """Returns (lp per label [sum k] or for the selected branches, lse [N])."""
    label_off = np.asarray(label_off)
    label_ids = np.asarray(label_ids)
    N = len(label_off) - 1
    sel = list(range(N)) if branches is None else list(branches)
    logits = full_logits(h, W, sel)
    lse = log_sum_exp(logits)
    lp = []
    for i, n in enumerate(sel):
        ids = label_ids[label_off[n]:label_off[n + 1]]
        lp.append(logits[i, ids] - lse[i])
    lp = np.concatenate(lp) if lp else np.zeros(0)
    return lp, lse
