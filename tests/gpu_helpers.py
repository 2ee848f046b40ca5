"""Shared helpers for the GPU parity tests: run a workload through libsp and
compare with the oracle at the tolerances of the parity bar.

Tolerances (bf16 inputs, fp32 accumulation in the kernels, float64 oracle):
attention outputs 2e-2 max abs; attention lse 1e-2; label logprobs and the
vocabulary lse 1e-2; normalised label probabilities 1e-3; argmax identical
wherever the oracle's top-2 probability margin exceeds 1e-2.
"""
import numpy as np
import torch

from oracle import attention as OA
from oracle import label_softmax as OL
from oracle import readout as OR
from oracle import staging as OS

TOL_OUT = 2e-2
TOL_LSE = 1e-2
TOL_LP = 1e-2
TOL_P = 1e-3
ARGMAX_MARGIN = 1e-2


def run_gpu(wl, stream=None, schedule="rounds", n_sms=None):
    """n_sms: plan for that many SMs (small values turn split parts off and
    the pairing of sibling leaf tails on)."""
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    dev = torch.device("cuda:0")
    sh = wl.shape
    clf = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=dev)
    if n_sms is not None:
        clf.plan_sms = n_sms
    q, k, v = wl.q.to(dev), wl.k.to(dev), wl.v.to(dev)
    h, W = wl.h.to(dev), wl.W.to(dev)
    off = torch.from_numpy(wl.label_off).to(dev)
    ids = torch.from_numpy(wl.label_ids).to(dev)
    res = clf.run(wl.req_of_branch, wl.tok_offsets, wl.tokens, q, k, v, h, W, off, ids, stream,
                  schedule)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    return {
        "out": res.out.float().cpu().numpy(),
        "lse": res.lse.cpu().numpy(),
        "logprobs": res.logprobs.cpu().numpy(),
        "lse_vocab": res.lse_vocab.cpu().numpy(),
        "probs": res.probs.cpu().numpy(),
        "argmax": res.argmax.cpu().numpy(),
        "rounds": res.plan.rounds(),
        "launches": clf.last_launches,
        "plan": res.plan,
    }


def label_slices(off, branches):
    return np.concatenate([np.arange(off[b], off[b + 1]) for b in branches])


def check_readout(wl, g, branches=None):
    N = wl.n_branches
    branches = list(range(N)) if branches is None else list(branches)
    lp, lse = OR.label_logprobs(wl.h, wl.W, wl.label_off, wl.label_ids, branches=branches)
    sel = label_slices(wl.label_off, branches)
    assert np.abs(g["logprobs"][sel] - lp).max() <= TOL_LP
    assert np.abs(g["lse_vocab"][branches] - lse).max() <= TOL_LP
    sub_off = np.concatenate([[0], np.cumsum([wl.label_off[b + 1] - wl.label_off[b] for b in branches])])
    probs, am = OL.label_softmax(lp, sub_off)
    assert np.abs(g["probs"][sel] - probs).max() <= TOL_P
    margin = OL.top2_margin(probs, sub_off)
    for i, b in enumerate(branches):
        if margin[i] > ARGMAX_MARGIN:
            assert g["argmax"][b] == am[i], (b, g["argmax"][b], am[i])
    # the GPU's own probabilities sum to one
    for b in branches:
        a, e = wl.label_off[b], wl.label_off[b + 1]
        assert abs(g["probs"][a:e].sum() - 1.0) < 1e-5


def check_attention_full(wl, g):
    plan = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    out, lse, worst = OA.reference_attention(plan, wl.q, wl.k, wl.v)
    assert worst < 1e-9
    assert np.abs(g["out"] - out).max() <= TOL_OUT
    assert np.abs(g["lse"] - lse).max() <= TOL_LSE
    return plan


def sample_rows(plan, n_random, seed=0):
    """Each branch's last row, the first and last row of every segment and of
    every 16-token tile boundary nearby, plus seeded random rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(len(plan.paths)):
        rows.add(plan.branch_last_row(b))
    for s in plan.segments:
        rows.update([s.node_start, s.node_start + s.length - 1])
        for t in (15, 16, 31, 32, 63, 64, 127, 128):
            if t < s.length:
                rows.add(s.node_start + t)
    rows.update(rng.integers(0, plan.node_tokens, n_random).tolist())
    return sorted(rows)


def check_attention_sampled(wl, g, n_random=64, seed=0):
    plan = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    rows = sample_rows(plan, n_random, seed)
    so, sl = OA.sampled_attention(plan, wl.q, wl.k, wl.v, rows)
    assert np.abs(g["out"][rows] - so).max() <= TOL_OUT
    assert np.abs(g["lse"][rows] - sl).max() <= TOL_LSE
    return plan, rows


def check_attention_suffix_rows(wl, g, branches=None):
    """Every row of each branch's own last segment (its suffix, the branch
    tokens the metric counts) against unshared float64 attention over the
    branch's whole sequence."""
    plan = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    worst_o = worst_l = 0.0
    for b in (range(len(plan.paths)) if branches is None else branches):
        rows, o, l = OA.branch_suffix_attention(plan, wl.q, wl.k, wl.v, b)
        worst_o = max(worst_o, float(np.abs(g["out"][rows] - o).max()))
        worst_l = max(worst_l, float(np.abs(g["lse"][rows] - l).max()))
    assert worst_o <= TOL_OUT, worst_o
    assert worst_l <= TOL_LSE, worst_l
    return worst_o, worst_l
