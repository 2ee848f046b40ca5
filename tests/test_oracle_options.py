"""Pins of multi-token option scoring and label-prior calibration
(oracle/options.py): the pages' worked example, exact normalisation of the
chain rule, closed forms and brute force.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import log_softmax

from oracle import label_softmax as LS
from oracle import options as OP

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_one_token_options_are_the_label_softmax():
    """openjev-sglang article, prefill-only section: yes -0.3 / no -1.5 gives
    0.77 / 0.23; one-token options without a prior reach it unchanged."""
    g = golden("label_softmax_worked_example.json")
    lp = np.array(g["logprobs"])
    scores, probs, am = OP.option_softmax(lp, [0, 1, 2], [0, 2])
    assert np.array_equal(scores, lp)
    assert [round(p, g["printed_decimals"]) for p in probs] == g["printed_probs"]
    assert am[0] == g["printed_argmax"]
    p2, a2 = LS.label_softmax(lp, [0, 2])
    assert np.allclose(probs, p2, rtol=0, atol=1e-15) and am[0] == a2[0]


def toy_model(V, H, seed):
    """A toy language model: the hidden state at a position is the embedding
    of the token there (h = E[token]), the next-token distribution is
    softmax(W h)."""
    rng = np.random.default_rng(seed)
    E = rng.normal(size=(V, H))
    W = rng.normal(size=(V, H)) * 0.7
    return E, W


@pytest.mark.parametrize("m", [1, 2, 3])
def test_chain_rule_normalises_over_every_string(m):
    """Scoring every string of m tokens after a fixed prompt gives joint
    probabilities that sum to 1 exactly (the chain rule over the model's
    conditionals): a dropped term, a logit in place of a log-softmax, a mean
    in place of the sum, or a token scored at the wrong position breaks it."""
    V, H = 5, 4
    E, W = toy_model(V, H, seed=m)
    last_prompt_token = 3
    strings = list(itertools.product(range(V), repeat=m))
    rows, toks, opt_off = [], [], [0]
    for s in strings:
        prev = last_prompt_token
        for t in s:
            rows.append(E[prev])
            toks.append(t)
            prev = t
        opt_off.append(len(toks))
    lp = OP.row_logprobs(np.array(rows), W, toks)  # float64 arrays: no rounding
    scores = OP.option_scores(lp, opt_off)
    assert abs(np.exp(scores).sum() - 1.0) < 1e-12
    # the renormalised distribution over all strings is then the joint itself
    _, probs, _ = OP.option_softmax(lp, opt_off, [0, len(strings)])
    assert np.allclose(probs, np.exp(scores), rtol=0, atol=1e-13)


def test_row_logprobs_brute_force():
    """Each row term against scipy's log_softmax of the full logit row."""
    rng = np.random.default_rng(7)
    V, H, n = 37, 6, 11
    h = rng.normal(size=(n, H))
    W = rng.normal(size=(V, H))
    toks = rng.integers(0, V, n)
    lp = OP.row_logprobs(h, W, toks)
    want = log_softmax(h @ W.T, axis=1)[np.arange(n), toks]
    assert np.allclose(lp, want, rtol=0, atol=1e-12)
    # bf16 inputs as the GPU path sees them: the same after exact upcast
    hb = torch.tensor(h).bfloat16()
    Wb = torch.tensor(W).bfloat16()
    lpb = OP.row_logprobs(hb, Wb, toks)
    wantb = log_softmax(hb.double().numpy() @ Wb.double().numpy().T, axis=1)[np.arange(n), toks]
    assert np.allclose(lpb, wantb, rtol=0, atol=1e-12)


def test_calibration_closed_forms():
    """Contextual calibration (diagonal): a prior equal to the scores gives
    the uniform distribution; a prior constant over a question's options
    changes nothing; with two options p_0 = 1 / (1 + exp((s1 - pi1) - (s0 - pi0)))."""
    rng = np.random.default_rng(3)
    row = rng.normal(size=9) - 4
    opt_off = [0, 2, 3, 6, 7, 9]  # 5 options of 2, 1, 3, 1, 2 tokens
    q_off = [0, 3, 5]             # questions of 3 and 2 options
    s, _, _ = OP.option_softmax(row, opt_off, q_off)
    _, pu, _ = OP.option_softmax(row, opt_off, q_off, prior=s)
    assert np.allclose(pu, [1 / 3] * 3 + [1 / 2] * 2, rtol=0, atol=1e-15)
    _, p0, a0 = OP.option_softmax(row, opt_off, q_off)
    _, pc, ac = OP.option_softmax(row, opt_off, q_off, prior=[2.5, 2.5, 2.5, -1.0, -1.0])
    assert np.allclose(p0, pc, rtol=0, atol=1e-14) and np.array_equal(a0, ac)
    prior = rng.normal(size=5)
    _, p, am = OP.option_softmax(row, opt_off, q_off, prior=prior)
    want = 1.0 / (1.0 + math.exp((s[4] - prior[4]) - (s[3] - prior[3])))
    assert abs(p[3] - want) < 1e-14
    assert am[1] == (0 if want >= 0.5 else 1)


def test_calibration_can_flip_the_choice():
    """A prior that favours an option as much as its score does removes its
    advantage: the calibrated argmax moves to the other option."""
    row = np.array([-0.3, -1.5])
    _, p, am = OP.option_softmax(row, [0, 1, 2], [0, 2], prior=[-0.1, -2.0])
    assert am[0] == 1 and p[1] > 0.5


def test_ties_take_the_lowest_index():
    _, p, am = OP.option_softmax([-1.0, -0.5, -0.5, -1.0], [0, 2, 3, 4], [0, 3])
    # scores: -1.5, -0.5, -1.0 -> option 1
    assert am[0] == 1
    _, p, am = OP.option_softmax([-1.0, -1.0], [0, 1, 2], [0, 2])
    assert am[0] == 0 and np.allclose(p, [0.5, 0.5], rtol=0, atol=1e-15)
