"""Question-type readouts and the confidence value.

Source: the openjev-sglang article (jdon.com):
* section on the confidence value: confidence = 1 - H(P) / ln K, with H the
  Shannon entropy in nats and K the number of options (worked example
  [0.9, 0.05, 0.05] -> about 0.641; uniform -> 0; one-hot -> 1);
* section on the three question types: a yes/no ("noul") question returns
  P(yes); a choice returns the argmax and the full distribution; a score
  returns the expectation sum_i i * P_i with i counted from 0 (worked example
  [0.2, 0.6, 0.2] -> 1.0).

The batched forms follow the two layouts on the pages:
* label_decide: one question per branch, its options the branch's labels
  (openjev-sglang article: a single-token label per option, softmax over the
  returned log-probabilities, then the question type);
* candidate_decide: one question per group of yes/no candidate branches
  (LLM2Jev page, on why the same material is computed many times: every
  choice option and score level is its own yes/no input; section on outputs:
  the final answers are read after normalisation).

Readings: 0 * ln 0 is taken as 0 (the one-hot case is printed as 1); the
"yes" label is the first label of a branch; a choice question's scalar value
is the chosen option's probability; candidate groups normalise P(yes) by its
sum over the question (the LLM2Jev page prints no formula).

This module is test infrastructure: only tests, the smoke check and the
benchmark's CPU baseline call it.

Parity: pinned by the printed examples (tests/golden: 0.641, 1.0, 0.77),
closed forms (score of a one-hot and of a uniform distribution, confidence 0
for uniform and 1 for one-hot at every K, symmetry of the two-option
confidence) and invariants (scale invariance of the candidate assembly).
"""
from __future__ import annotations

import math

import numpy as np


def entropy(p) -> float:
    p = np.asarray(p, dtype=np.float64)
    nz = p[p > 0]
    return float(-(nz * np.log(nz)).sum())


def confidence(p) -> float:
    K = len(p)
    return 1.0 - entropy(p) / math.log(K)


def score_value(p) -> float:
    p = np.asarray(p, dtype=np.float64)
    return float((np.arange(len(p)) * p).sum())


def noul_value(p) -> float:
    return float(p[0])


def choice_value(p):
    p = np.asarray(p, dtype=np.float64)
    return int(np.argmax(p)), p.copy()


# Question-type codes shared by the batched functions below.
NOUL, CHOICE, SCORE = 0, 1, 2


def _decide_one(p, qtype):
    """value and confidence of one distribution under a question type.

    noul: value = probability of the first label ("yes");
    choice: value = probability of the chosen (argmax) option (reading: the
    article returns the argmax and the distribution; the scalar slot carries
    the chosen option's probability);
    score: value = sum_i i * P_i, i from 0.
    """
    p = np.asarray(p, dtype=np.float64)
    if qtype == NOUL:
        v = noul_value(p)
    elif qtype == CHOICE:
        v = float(p[choice_value(p)[0]])
    elif qtype == SCORE:
        v = score_value(p)
    else:
        raise ValueError(qtype)
    return v, confidence(p)


def label_decide(lp, label_off, qtype):
    """One question per branch, its options being the branch's labels
    (openjev-sglang layout): label softmax, argmax, then the question type's
    value and the confidence over the K labels.

    Returns probs [sum k], argmax [N], value [N], confidence [N] (float64)."""
    from oracle.label_softmax import label_softmax

    probs, am = label_softmax(lp, label_off)
    N = len(label_off) - 1
    value = np.empty(N)
    conf = np.empty(N)
    for n in range(N):
        p = probs[label_off[n]:label_off[n + 1]]
        value[n], conf[n] = _decide_one(p, int(qtype[n]))
    return probs, am, value, conf


def candidate_decide(probs, label_off, cand_off, qtype):
    """One question per group of candidate branches (LLM2Jev layout: every
    choice option or score level is its own yes/no branch).

    Reading (the page says the final answers are normalised but prints no
    formula): y_c = the candidate branch's probability of its first label
    ("yes"); a choice or score question's distribution over its K >= 2
    candidates is y_c / sum y; a noul question has one candidate, its value is
    y and its confidence is taken over (y, 1 - y).

    Returns dist [n_candidates], argmax [Q] (candidate index within the
    question, lowest on ties), value [Q], confidence [Q] (float64)."""
    probs = np.asarray(probs, dtype=np.float64)
    Q = len(cand_off) - 1
    dist = np.empty(int(cand_off[-1]))
    am = np.empty(Q, dtype=np.int32)
    value = np.empty(Q)
    conf = np.empty(Q)
    for q in range(Q):
        a, b = int(cand_off[q]), int(cand_off[q + 1])
        y = np.array([probs[label_off[c]] for c in range(a, b)])
        if qtype[q] == NOUL:
            if b - a != 1:
                raise ValueError("a noul question has one candidate")
            dist[a] = y[0]
            am[q] = 0
            value[q], conf[q] = y[0], confidence([y[0], 1.0 - y[0]])
            continue
        d = y / y.sum()
        dist[a:b] = d
        am[q] = int(np.argmax(y))
        value[q], conf[q] = _decide_one(d, int(qtype[q]))
    return dist, am, value, conf
