"""Multi-token option scoring and label-prior calibration -- plain float64.

Test infrastructure: only tests, the smoke check and the benchmark's CPU legs
use this module.

Source: the openjev-multimodal "performance" page, section on next steps,
names label-prior calibration and multi-token option scoring as planned work
that changes the probabilities and needs its own evaluation.  The pages give
no formula for either; the readings taken (each listed in the design notes):

* Option score.  An option of m tokens t_1 .. t_m is scored by its joint
  log-probability under the model, the chain rule

      score = sum_i log softmax(W h_i)[t_i]

  where h_i is the hidden state at the position before t_i (the last prompt
  position for t_1, the position of t_{i-1} for the others).  Each term is
  the prefill-only readout of the openjev-sglang article (full-vocabulary
  log-softmax at one position, gathered at one token id), so a one-token
  option scores exactly its single-token label log-probability.  No length
  normalisation: the score is the probability of the option's whole string.
* Calibration.  A per-option prior log-probability pi_o (for instance the
  same readout on a content-free input) is subtracted before the
  renormalisation, p_o proportional to exp(score_o - pi_o): the diagonal form
  of contextual calibration (Zhao et al., "Calibrate before use", 2021).
* Renormalisation over a question's options: the stable softmax of the
  label softmax (openjev-sglang article, request-flow step 5); argmax is the
  lowest index among equal maxima.

Parity: pinned in ``tests/test_oracle_options.py`` by the printed worked
example reached through one-token options, by exact normalisation of the
chain rule over every string of a toy model, by closed forms of the
calibration and by brute force against scipy's log_softmax.
"""
from __future__ import annotations

import numpy as np

from . import readout as R


def row_logprobs(h_rows, W, tokens):
    """Log-probability of tokens[r] under the full-vocabulary softmax of
    W h_rows[r], one token per row (the readout with one label per row)."""
    n = len(tokens)
    off = np.arange(n + 1, dtype=np.int64)
    lp, _ = R.label_logprobs(h_rows, W, off, np.asarray(tokens))
    return lp


def option_scores(row_lp, opt_off):
    """score_o = sum of the row log-probabilities of option o's tokens
    (rows opt_off[o] .. opt_off[o+1]-1)."""
    row_lp = np.asarray(row_lp, dtype=np.float64)
    opt_off = np.asarray(opt_off)
    return np.array([row_lp[opt_off[o]:opt_off[o + 1]].sum() for o in range(len(opt_off) - 1)])


def option_softmax(row_lp, opt_off, q_off, prior=None):
    """Returns (scores [n_opts], probs [n_opts], argmax [n_questions]).

    scores: uncalibrated joint log-probabilities; probs: per question q
    (options q_off[q] .. q_off[q+1]-1), the stable softmax of scores - prior
    (prior = 0 when None); argmax: index within the question of the largest
    calibrated score, lowest on ties."""
    scores = option_scores(row_lp, opt_off)
    x = scores - (0.0 if prior is None else np.asarray(prior, dtype=np.float64))
    q_off = np.asarray(q_off)
    probs = np.empty_like(x)
    argmax = np.empty(len(q_off) - 1, dtype=np.int32)
    for q in range(len(q_off) - 1):
        a, b = int(q_off[q]), int(q_off[q + 1])
        z = x[a:b]
        m = z.max()
        e = np.exp(z - m)
        probs[a:b] = e / e.sum()
        argmax[q] = int(np.argmax(z))
    return scores, probs, argmax


def option_readout(h_rows, W, opt_off, opt_tokens, q_off, prior=None):
    """The whole path from hidden states: row log-probabilities, then
    option_softmax.  Returns (row_lp, scores, probs, argmax)."""
    lp = row_logprobs(h_rows, W, opt_tokens)
    scores, probs, argmax = option_softmax(lp, opt_off, q_off, prior)
    return lp, scores, probs, argmax
