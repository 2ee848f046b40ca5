"""Pins for the LM-head readout oracle."""
import json
import math
import os

import numpy as np
import scipy.special
import torch

from oracle import readout as R
from oracle import label_softmax as LS
from oracle import postprocess as PP

from conftest import GOLDEN


def _rand(n, H, V, seed=0):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(n, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) * 0.02).to(torch.bfloat16)
    return h, W


def test_zero_head_gives_uniform_logprob():
    V = 1000
    h, _ = _rand(3, 16, V)
    W = torch.zeros(V, 16, dtype=torch.bfloat16)
    off = np.array([0, 2, 4, 6])
    ids = np.array([0, 999, 5, 5, 17, 3])
    lp, lse = R.label_logprobs(h, W, off, ids)
    assert np.allclose(lp, -math.log(V), rtol=0, atol=1e-13)
    assert np.allclose(lse, math.log(V), atol=1e-13)


def test_matches_library_logsumexp_and_log_softmax():
    h, W = _rand(4, 64, 3001, seed=1)
    off = np.array([0, 2, 5, 6, 9])
    ids = np.array([1, 2, 3000, 0, 7, 11, 12, 13, 2999])
    lp, lse = R.label_logprobs(h, W, off, ids)
    logits = h.double() @ W.double().T
    ref_lse = torch.logsumexp(logits, dim=1).numpy()
    assert np.abs(lse - ref_lse).max() < 1e-12
    ls = scipy.special.log_softmax(logits.numpy(), axis=1)
    ref = np.concatenate([ls[n, ids[off[n]:off[n + 1]]] for n in range(4)])
    assert np.abs(lp - ref).max() < 1e-12


def test_shift_invariance():
    """Adding one constant to every logit (an extra hidden unit fixed at 1
    whose weight is the constant for all rows) leaves the logprobs unchanged
    and moves lse by the constant."""
    h, W = _rand(2, 32, 500, seed=2)
    off = np.array([0, 3, 5])
    ids = np.array([4, 8, 15, 16, 23])
    lp0, lse0 = R.label_logprobs(h, W, off, ids)
    c = 0.75  # exactly representable in bf16
    h1 = torch.cat([h, torch.ones(2, 1, dtype=torch.bfloat16)], 1)
    W1 = torch.cat([W, torch.full((500, 1), c, dtype=torch.bfloat16)], 1)
    lp1, lse1 = R.label_logprobs(h1, W1, off, ids)
    assert np.abs(lp1 - lp0).max() < 1e-12
    assert np.abs(lse1 - lse0 - c).max() < 1e-12


def test_dominant_label_logprob_tends_to_zero():
    V, H = 300, 8
    h = torch.zeros(1, H, dtype=torch.bfloat16)
    h[0, 0] = 1.0
    W = torch.zeros(V, H, dtype=torch.bfloat16)
    W[42, 0] = 64.0
    lp, _ = R.label_logprobs(h, W, np.array([0, 2]), np.array([42, 0]))
    # lp = -ln(1 + (V-1) e^-64) for the dominant id, -64 - that for the other
    assert abs(lp[0] - (-math.log1p((V - 1) * math.exp(-64.0)))) < 1e-15
    assert abs(lp[1] - (-64.0 + lp[0])) < 1e-12


def test_branch_subset_matches_full():
    h, W = _rand(5, 32, 700, seed=3)
    off = np.array([0, 2, 4, 6, 8, 10])
    ids = np.arange(10) * 7
    lp, lse = R.label_logprobs(h, W, off, ids)
    lp2, lse2 = R.label_logprobs(h, W, off, ids, branches=[1, 3])
    assert np.allclose(lp2, np.concatenate([lp[2:4], lp[6:8]]), atol=1e-14)
    assert np.allclose(lse2, lse[[1, 3]], atol=1e-14)


# ---- label softmax ----------------------------------------------------------

def test_worked_example_from_page():
    g = json.load(open(os.path.join(GOLDEN, "label_softmax_worked_example.json")))
    probs, am = LS.label_softmax(g["logprobs"], [0, 2])
    assert list(np.round(probs, g["printed_decimals"])) == g["printed_probs"]
    assert am[0] == g["printed_argmax"]
    # exact value: 1 / (1 + e^-1.2)
    assert abs(probs[0] - 1.0 / (1.0 + math.exp(-1.2))) < 1e-15


def test_softmax_sums_to_one_and_matches_scipy():
    rng = np.random.default_rng(5)
    off = np.array([0, 2, 66, 70, 73])
    lp = -np.abs(rng.standard_normal(73)) * 10 - 3
    probs, am = LS.label_softmax(lp, off)
    for n in range(4):
        a, b = off[n], off[n + 1]
        assert abs(probs[a:b].sum() - 1.0) < 1e-12
        assert np.abs(probs[a:b] - scipy.special.softmax(lp[a:b])).max() < 1e-15
        assert am[n] == int(np.argmax(lp[a:b]))


def test_argmax_ties_take_lowest_index():
    probs, am = LS.label_softmax([-1.0, -0.5, -0.5, -2.0], [0, 4])
    assert am[0] == 1
    assert abs(probs[1] - probs[2]) == 0.0


def test_softmax_large_magnitudes_stable():
    probs, _ = LS.label_softmax([-1000.0, -1001.0], [0, 2])
    assert abs(probs[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


# ---- post-processing (question types, confidence) --------------------------

def test_confidence_examples_from_page():
    g = json.load(open(os.path.join(GOLDEN, "confidence_example.json")))
    c0 = g["cases"][0]
    assert round(PP.entropy(c0["p"]), 3) == c0["printed_entropy"]
    assert round(math.log(len(c0["p"])), 3) == c0["printed_ln_k"]
    assert round(PP.confidence(c0["p"]), c0["decimals"]) == c0["printed_confidence"]
    for c in g["cases"][1:]:
        assert abs(PP.confidence(c["p"]) - c["printed_confidence"]) < 10 ** -c["decimals"]


def test_score_example_from_page():
    g = json.load(open(os.path.join(GOLDEN, "score_example.json")))
    assert abs(PP.score_value(g["p"]) - g["printed_score"]) < 1e-15
    assert PP.choice_value(g["p"])[0] == 1
    assert PP.noul_value([0.77, 0.23]) == 0.77
