"""GPU parity of continuous batching across requests: a stream of independent
requests run through ContinuousBatcher (native sp_batcher_* admission, one
plan, attention call and readout per batch) must give every request the
results the oracle gives it alone: attention over its own token trie, the
readout and label softmax at its branches' last positions (openjev-
multimodal performance page, next steps: batching across requests).
Tolerances are the parity bar's (tests/gpu_helpers.py)."""
import numpy as np
import pytest
import torch

from oracle import batching as OB

from gpu_helpers import check_attention_full, check_readout

pytestmark = pytest.mark.gpu

TREES = [
    (40, [(9, []), (17, []), (3, [])]),
    (130, [(20, [(5, []), (33, [])]), (1, [])]),
    (7, [(64, []), (64, [])]),
    (300, [(16, []), (2, []), (40, []), (9, [])]),
    (1, [(1, []), (2, [])]),
    (90, [(31, []), (31, [])]),
    (260, [(48, []), (12, [])]),
    (16, [(16, []), (16, []), (16, [])]),
    (57, [(200, []), (3, [])]),
]


def _requests(G):
    from prefill_only_shared_gb300.workloads import small_case
    wls = [small_case(t, seed=10 + i, n_q_heads=2 * G, n_kv_heads=2, head_dim=64, hidden=96,
                      vocab=700, labels=("per_branch", 3)) for i, t in enumerate(TREES)]
    W = wls[0].W  # one model: every request reads out with the same LM head
    for wl in wls:
        wl.W = W
    return wls, W


@pytest.mark.parametrize("G,schedule", [(4, "tree"), (8, "all"), (1, "rounds")])
def test_batched_requests_match_the_oracle(cuda_dev, lib, G, schedule):
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import ContinuousBatcher, SharedPrefixClassifier
    wls, W = _requests(G)
    sh = wls[0].shape
    clf = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=cuda_dev)
    budget, cap = 700, 3
    cb = ContinuousBatcher(clf, W.to(cuda_dev), budget, cap, capacity_rows=8192,
                           capacity_branches=256, capacity_labels=1024, schedule=schedule)
    sizes = []
    for wl in wls:
        cb.submit(wl.tok_offsets, wl.tokens, wl.q, wl.k, wl.v, wl.h, wl.label_off, wl.label_ids)
        sizes.append(wl.node_tokens)
    n = cb.run()
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    want = OB.form_batches(sizes, budget, cap)
    assert cb.batch_sizes == [len(b) for b in want] and n == len(want)
    assert max(cb.batch_sizes) > 1
    for rid, wl in enumerate(wls):
        g = {k: v.float().cpu().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy()
             for k, v in cb.result(rid).items()}
        check_attention_full(wl, g)
        check_readout(wl, g)


def test_batched_equals_alone(cuda_dev, lib):
    """A request's label probabilities in a batch equal those of the same
    request run alone through the classifier (within the probability bar),
    and its argmax is the same wherever the margin exceeds 1e-2."""
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import ContinuousBatcher, SharedPrefixClassifier
    wls, W = _requests(4)
    sh = wls[0].shape
    Wd = W.to(cuda_dev)
    clf = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=cuda_dev)
    cb = ContinuousBatcher(clf, Wd, 10 ** 6, 64, capacity_rows=8192, capacity_branches=256,
                           capacity_labels=1024)
    for wl in wls:
        cb.submit(wl.tok_offsets, wl.tokens, wl.q, wl.k, wl.v, wl.h, wl.label_off, wl.label_ids)
    assert cb.run() == 1
    torch.cuda.synchronize()
    alone = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                   device=cuda_dev)
    for rid, wl in enumerate(wls):
        res = alone.run(wl.req_of_branch, wl.tok_offsets, wl.tokens, wl.q.to(cuda_dev),
                        wl.k.to(cuda_dev), wl.v.to(cuda_dev), wl.h.to(cuda_dev), Wd,
                        torch.from_numpy(wl.label_off).to(cuda_dev),
                        torch.from_numpy(wl.label_ids).to(cuda_dev), schedule="tree")
        torch.cuda.synchronize()
        got = cb.result(rid)
        assert (got["probs"] - res.probs).abs().max().item() <= 1e-3
        assert (got["out"].float() - res.out.float()).abs().max().item() <= 2e-2
    sp.sp_check_device_error()
