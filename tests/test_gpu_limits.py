"""GPU parity at the request limits the classifier's service page states
(prefill-only classification page, request limits: at most 32768 tokens in
one branch, at most 262144 tokens in one request, at most 64 labels).

Two workloads sit exactly on those limits, with the yes/no model's attention
shape (Hq 32, Hkv 4, d 128):

- one request of 8 branches of 32768 tokens each (262144 logical tokens): a
  30000-token shared state and 8 suffixes of 2768 tokens, 64 labels per
  branch;
- one request of a single 32768-token branch with nothing shared: plain
  causal attention at the longest allowed length.

Attention is compared on sampled rows (segment and tile boundaries, every
branch's last row, seeded random rows); the readout of every branch in
full.  A small hidden size and vocabulary keep the oracle's readout cheap;
the readout's own size limits are covered by the readout tests."""
import numpy as np
import pytest

from oracle import attention as OA
from oracle import staging as OS
from prefill_only_shared_gb300.workloads import small_case

from gpu_helpers import TOL_LSE, TOL_OUT, check_readout, run_gpu, sample_rows

pytestmark = pytest.mark.gpu

_ORACLE = {}

LIMIT_CASES = {
    "eight_full_branches": ((30000, [(2768, []) for _ in range(8)]), [[0], list(range(1, 8))]),
    "one_unshared_branch": ((32768, []), [[0]]),
}


@pytest.mark.parametrize("schedule", ["rounds", "tree"])
@pytest.mark.parametrize("name", list(LIMIT_CASES))
def test_request_at_the_token_limits(cuda_dev, lib, name, schedule):
    tree, rounds = LIMIT_CASES[name]
    wl = small_case(tree, seed=11, n_q_heads=32, n_kv_heads=4, head_dim=128, hidden=256,
                    vocab=4096, labels=("shared", 64))
    lens = wl.tok_offsets[1:] - wl.tok_offsets[:-1]
    assert (lens == 32768).all() and lens.sum() <= 262144
    g = run_gpu(wl, schedule=schedule)
    assert g["rounds"] == rounds
    st = g["plan"].stats()
    assert st["logical_tokens"] == int(lens.sum())
    if name not in _ORACLE:  # the oracle's rows, shared by both schedules
        plan = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
        rows = sample_rows(plan, 48, seed=3)
        _ORACLE[name] = (rows,) + OA.sampled_attention(plan, wl.q, wl.k, wl.v, rows)
    rows, so, sl = _ORACLE[name]
    assert np.abs(g["out"][rows] - so).max() <= TOL_OUT
    assert np.abs(g["lse"][rows] - sl).max() <= TOL_LSE
    check_readout(wl, g)
