"""Continuous batching across requests: the admission rule, plainly.

Test infrastructure: only tests, the smoke check and the benchmark's CPU legs
use this module.

Source: the openjev-multimodal "performance" page, section on next steps,
plans continuous batching across requests to raise throughput; the SGLang-JAX
blog translation (section on reducing scheduling overhead) describes the
host preparing the next batch while the device computes the current one.
Neither gives an admission rule; the readings (listed in the design notes):

* A request's size is its node tokens: the number of distinct prefixes of its
  branches, i.e. the positions of its token trie, what its plan computes cold
  (taken here from the staging oracle's plan of the request alone).
* Requests wait first-in first-out.  A batch takes them from the head, in
  submission order, while its node tokens stay within ``max_tokens`` and its
  request count within ``max_requests``; the head request always goes in.
* Request i of a batch is request id i of the batch's plan, so the batch's
  node rows are its requests' rows one after the other.

Parity: pinned in ``tests/test_oracle_batching.py`` by brute-force counting of
distinct prefixes, by closed forms (equal requests, a budget below one
request) and by invariants of the rule (every request once, in order, within
the limits, and no batch that could have taken the next request).
"""
from __future__ import annotations

import numpy as np

from . import staging as S


def node_tokens(tok_offsets, tokens) -> int:
    """Node tokens of one request: its cold plan's node rows."""
    off = np.asarray(tok_offsets, dtype=np.int64)
    n = len(off) - 1
    plan = S.build_plan(np.zeros(n, dtype=np.int32), off, np.asarray(tokens, dtype=np.int32))
    return int(plan.node_tokens)


def form_batches(sizes, max_tokens: int, max_requests: int):
    """The batches (lists of request ids) that the rule forms from a queue of
    requests of the given node-token sizes, all submitted before the first
    batch forms."""
    batches = []
    i, n = 0, len(sizes)
    while i < n:
        batch = [i]
        total = int(sizes[i])
        j = i + 1
        while j < n and len(batch) < max_requests and total + int(sizes[j]) <= max_tokens:
            total += int(sizes[j])
            batch.append(j)
            j += 1
        batches.append(batch)
        i = j
    return batches


def batch_offsets(batch, sizes, n_branches):
    """Branch and node-row offsets of a batch's requests within its plan."""
    boff = np.concatenate([[0], np.cumsum([n_branches[r] for r in batch])]).astype(np.int64)
    roff = np.concatenate([[0], np.cumsum([sizes[r] for r in batch])]).astype(np.int64)
    return boff, roff
