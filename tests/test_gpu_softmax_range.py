"""Rows whose scores rise far above the running maximum of their first units.

The online softmax (FlashAttention's blockwise rescaling, which the sglang
article's prefill path runs per KV block) keeps a running maximum m and
weights every key by 2^(s - m); m cancels in O / l, so any reference keeps the
result exact in relative terms as long as 2^(s - m) stays finite.  The kernel
takes m on a row's first unit with a finite score and then again only when a
unit's sum shows a score far above it (or a value that is not finite), in which
case it redoes that unit with the new maximum.  Random N(0, 1) inputs never
reach that second pass, so these cases plant one prefix key whose score lies
far above every other key's:

- height 16: q . k* is about 100 in natural-log units (about 150 above the
  others in log2 units), so 2^(s - m) would overflow without the second pass;
- height 4: about 37 above them in log2 units, inside the range the kernel
  accepts without a second pass (P up to about 2^37 in bf16, sums in fp32).

Every row's output and lse are compared with the float64 oracle at the parity
tolerances, under the per-round and the single-call schedules, and with the
plan on one SM (no split parts, paired sibling tails)."""
import os
import sys

import numpy as np
import pytest

from oracle import staging as OS
from prefill_only_shared_gb300.workloads import small_case

sys.path.insert(0, os.path.dirname(__file__))
from gpu_helpers import check_attention_full, check_readout, run_gpu  # noqa: E402

PREFIX, KEY_AT = 600, 400


def planted(height):
    wl = small_case((PREFIX, [(50, []), (70, []), (3, [])]), seed=11, n_q_heads=8, n_kv_heads=2,
                    head_dim=64, hidden=128, vocab=1000)
    plan = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    root = plan.segments[plan.paths[0][0]]
    assert root.length == PREFIX
    # every query entry positive, one prefix key equal to `height` in every
    # entry of every KV head: q . k* is about height * 0.8 * 64 for every row
    wl.q = wl.q.abs()
    wl.k[root.node_start + KEY_AT] = height
    return wl


@pytest.mark.gpu
@pytest.mark.parametrize("n_sms", [None, 1])
@pytest.mark.parametrize("schedule", ["rounds", "tree"])
@pytest.mark.parametrize("height", [4.0, 16.0])
def test_a_key_far_above_the_rest(cuda_dev, lib, height, schedule, n_sms):
    wl = planted(height)
    g = run_gpu(wl, schedule=schedule, n_sms=n_sms)
    assert np.isfinite(g["out"]).all() and np.isfinite(g["lse"]).all()
    check_attention_full(wl, g)
    check_readout(wl, g)


def test_the_planted_key_dominates_in_the_oracle():
    """The case does what it is meant to: in the oracle the planted key takes
    almost all of the weight of every row that sees it (height 16)."""
    from oracle import attention as OA
    wl = planted(16.0)
    plan = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    out, lse, _ = OA.reference_attention(plan, wl.q, wl.k, wl.v)
    root = plan.segments[plan.paths[0][0]]
    j = root.node_start + KEY_AT
    v = wl.v.float().numpy()
    G = wl.shape.n_q_heads // wl.shape.n_kv_heads
    for row in (j, j + 1, root.node_start + PREFIX - 1, plan.branch_last_row(0)):
        for hq in range(wl.shape.n_q_heads):
            assert np.abs(out[row, hq] - v[j, hq // G]).max() < 1e-6
    # rows before the key do not see it
    assert np.abs(out[j - 1, 0] - v[j, 0]).max() > 1e-2
