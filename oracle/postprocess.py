"""Question-type readouts and the confidence value.

Source: the openjev-sglang article (jdon.com):
* section on the confidence value: confidence = 1 - H(P) / ln K, with H the
  Shannon entropy in nats and K the number of options (worked example
  [0.9, 0.05, 0.05] -> about 0.641; uniform -> 0; one-hot -> 1);
* section on the three question types: a yes/no ("noul") question returns
  P(yes); a choice returns the argmax and the full distribution; a score
  returns the expectation sum_i i * P_i with i counted from 0 (worked example
  [0.2, 0.6, 0.2] -> 1.0).

Reading: 0 * ln 0 is taken as 0 (the one-hot case is printed as 1); for a
yes/no question the "yes" label is the first label of the branch.

Parity: pinned by the three printed examples (tests/golden).
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
