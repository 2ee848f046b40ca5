"""Pins of the question-type decision (oracle/postprocess.py): the pages'
printed examples, closed forms and invariants.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

from oracle import postprocess as PP

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _csr(groups):
    off = np.concatenate([[0], np.cumsum([len(g) for g in groups])]).astype(np.int32)
    return np.concatenate([np.asarray(g, float) for g in groups]), off


def test_label_decide_refund_example():
    """openjev-sglang article, prefill-only section: yes -0.3 / no -1.5 gives
    P(yes) 0.77, the noul value."""
    g = golden("label_softmax_worked_example.json")
    lp, off = _csr([g["logprobs"]])
    probs, am, val, conf = PP.label_decide(lp, off, [PP.NOUL])
    assert round(val[0], g["printed_decimals"]) == g["printed_probs"][0]
    assert am[0] == g["printed_argmax"]


def test_label_decide_confidence_and_score_examples():
    """The confidence example [0.9, 0.05, 0.05] -> 0.641 and the score
    example [0.2, 0.6, 0.2] -> 1.0, reached from log-probabilities shifted by
    an arbitrary constant (the softmax removes it)."""
    c = golden("confidence_example.json")["cases"][0]
    s = golden("score_example.json")
    lp, off = _csr([np.log(c["p"]) - 2.5, np.log(s["p"]) + 7.0])
    probs, am, val, conf = PP.label_decide(lp, off, [PP.CHOICE, PP.SCORE])
    assert round(conf[0], c["decimals"]) == c["printed_confidence"]
    assert abs(val[0] - 0.9) < 1e-12 and am[0] == 0
    assert abs(val[1] - s["printed_score"]) < 1e-12
    assert am[1] == 1


@pytest.mark.parametrize("K", [2, 3, 7, 64])
def test_uniform_and_one_hot_closed_forms(K):
    # uniform: confidence 0, score (K - 1) / 2, choice value 1 / K, argmax 0
    lp, off = _csr([np.zeros(K)] * 3)
    _, am, val, conf = PP.label_decide(lp, off, [PP.NOUL, PP.CHOICE, PP.SCORE])
    assert np.allclose(conf, 0.0, atol=1e-12)
    assert abs(val[0] - 1 / K) < 1e-12 and abs(val[1] - 1 / K) < 1e-12
    assert abs(val[2] - (K - 1) / 2) < 1e-12
    assert (am == 0).all()
    # one-hot at i: confidence 1, score i
    for i in (0, K // 2, K - 1):
        x = np.full(K, -1e4)
        x[i] = 0.0
        lp, off = _csr([x])
        _, am, val, conf = PP.label_decide(lp, off, [PP.SCORE])
        assert abs(conf[0] - 1.0) < 1e-12 and abs(val[0] - i) < 1e-9 and am[0] == i


def test_two_option_confidence_symmetric_and_monotone():
    ps = np.linspace(0.5, 1.0, 11)
    c = [PP.confidence([p, 1 - p]) for p in ps]
    assert all(abs(PP.confidence([1 - p, p]) - x) < 1e-12 for p, x in zip(ps, c))
    assert all(b > a for a, b in zip(c, c[1:]))
    assert abs(c[0]) < 1e-12 and abs(c[-1] - 1) < 1e-12


def test_score_is_linear_in_the_distribution():
    rng = np.random.default_rng(3)
    p, q = rng.dirichlet(np.ones(9)), rng.dirichlet(np.ones(9))
    t = 0.3
    assert abs(PP.score_value(t * p + (1 - t) * q)
               - (t * PP.score_value(p) + (1 - t) * PP.score_value(q))) < 1e-12


def test_candidate_decide_department_and_severity():
    """LLM2Jev page's example request: department (choice over shipping,
    billing, returns) and severity (score over levels 0..2), each option a
    yes/no branch.  P(yes) proportional to the printed distributions of the
    openjev-sglang article gives back its printed confidence and score."""
    c = golden("confidence_example.json")["cases"][0]
    s = golden("score_example.json")
    y = np.concatenate([0.4 * np.asarray(c["p"]), 0.9 * np.asarray(s["p"])])
    # each candidate branch has labels (yes, no): probs [yes, 1 - yes]
    probs = np.stack([y, 1 - y], 1).ravel()
    label_off = np.arange(0, 2 * len(y) + 1, 2)
    cand_off = np.array([0, 3, 6])
    dist, am, val, conf = PP.candidate_decide(probs, label_off, cand_off, [PP.CHOICE, PP.SCORE])
    assert np.allclose(dist[:3], c["p"], atol=1e-12) and np.allclose(dist[3:], s["p"], atol=1e-12)
    assert round(conf[0], c["decimals"]) == c["printed_confidence"]
    assert am[0] == 0 and abs(val[0] - 0.9) < 1e-12
    assert abs(val[1] - s["printed_score"]) < 1e-12 and am[1] == 1


def test_candidate_decide_scale_invariance_and_noul():
    rng = np.random.default_rng(7)
    y = rng.uniform(0.05, 0.95, 12)
    label_off = np.arange(0, 13, 1)  # one label per branch suffices here
    cand_off = np.array([0, 5, 11, 12])
    qt = [PP.SCORE, PP.CHOICE, PP.NOUL]
    d1, a1, v1, c1 = PP.candidate_decide(y, label_off, cand_off, qt)
    y2 = y.copy()
    y2[:11] *= 0.37  # scaling a choice / score question's P(yes) changes nothing
    d2, a2, v2, c2 = PP.candidate_decide(y2, label_off, cand_off, qt)
    assert np.allclose(d1[:11], d2[:11]) and (a1 == a2).all()
    assert np.allclose(v1[:2], v2[:2]) and np.allclose(c1[:2], c2[:2])
    for q in range(2):
        assert abs(d1[cand_off[q]:cand_off[q + 1]].sum() - 1) < 1e-12
    # noul: the branch's own P(yes) and the two-option confidence
    assert v1[2] == y[11] and abs(c1[2] - PP.confidence([y[11], 1 - y[11]])) < 1e-15
    with pytest.raises(ValueError):
        PP.candidate_decide(y, label_off, np.array([0, 2]), [PP.NOUL])


def test_planted_mistakes_fail_a_pin():
    """Plausible slips (score counted from 1, log base 2, P(yes) read from the
    second label) each break one of the printed examples."""
    s = golden("score_example.json")
    p = np.asarray(s["p"])
    assert abs(float(((np.arange(3) + 1) * p).sum()) - s["printed_score"]) > 0.5
    c = golden("confidence_example.json")["cases"][0]
    h2 = -(np.asarray(c["p"]) * np.log2(c["p"])).sum()
    assert round(1 - h2 / math.log(3), 3) != c["printed_confidence"]
    g = golden("label_softmax_worked_example.json")
    lp, off = _csr([g["logprobs"]])
    probs, _, _, _ = PP.label_decide(lp, off, [PP.NOUL])
    assert round(probs[1], 2) != g["printed_probs"][0]
