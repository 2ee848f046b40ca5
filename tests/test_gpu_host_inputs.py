"""run_from_host: a pass whose inputs are copied in from pinned host memory on
a side stream into one of two device input sets, overlapping the previous
pass's kernels (natively through sp_run_pass_host, or through torch
copies).  Consecutive calls with different inputs must each give the results
of `run` on device copies of their own inputs (the double buffering must
never let a copy overwrite inputs that a pass still reads), within 1e-6 on
the probabilities."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["tree", "rounds", "mixed"])
def test_host_input_passes_match_device_passes(cuda_dev, lib, mode):
    """tree: every call is one native sp_run_pass_host; rounds: copies through
    torch and the orchestrated calls; mixed: the two alternate on one
    classifier and share its input sets and their events.  A larger request in
    the sequence makes each input set grow while the other may still be in
    use."""
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    from prefill_only_shared_gb300.workloads import make_workload, small_case
    wls = [make_workload("tiny", seed=s) for s in (0, 1, 2)]
    sh = wls[0].shape
    wls.append(small_case((600, [(50, []) for _ in range(6)] + [(3, [])]), seed=7,
                          n_q_heads=sh.n_q_heads, n_kv_heads=sh.n_kv_heads,
                          head_dim=sh.head_dim, hidden=sh.hidden, vocab=sh.vocab))
    W = wls[0].W.to(cuda_dev)  # one model for every pass
    ref = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=cuda_dev)
    want = []
    for wl in wls:
        r = ref.run(wl.req_of_branch, wl.tok_offsets, wl.tokens, wl.q.to(cuda_dev),
                    wl.k.to(cuda_dev), wl.v.to(cuda_dev), wl.h.to(cuda_dev), W,
                    torch.from_numpy(wl.label_off).to(cuda_dev),
                    torch.from_numpy(wl.label_ids).to(cuda_dev), schedule="tree")
        torch.cuda.synchronize()
        want.append((r.probs.cpu().clone(), r.argmax.cpu().clone()))
    pinned = [tuple(t.pin_memory() for t in (wl.q, wl.k, wl.v, wl.h,
                                              torch.from_numpy(wl.label_off),
                                              torch.from_numpy(wl.label_ids))) for wl in wls]
    clf = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=cuda_dev)
    order = [0, 1, 3, 2, 0, 3, 1, 1, 0, 2]
    outs = []
    for j, i in enumerate(order):
        wl = wls[i]
        schedule = mode if mode != "mixed" else ("tree", "rounds")[j % 3 == 1]
        p = torch.empty(int(wl.label_off[-1]), dtype=torch.float32).pin_memory()
        a = torch.empty(wl.n_branches, dtype=torch.int32).pin_memory()
        clf.run_from_host(wl.req_of_branch, wl.tok_offsets, wl.tokens, *pinned[i][:4], W,
                          *pinned[i][4:], p, a, schedule=schedule)
        if schedule == "tree":
            assert clf.last_pass_launches >= 3
        outs.append((i, p, a))
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    # the readout hands its last vocab tiles to whichever CTA is free, so the
    # order of its per-CTA partial sums, hence the last bits, can change
    # from run to run
    for i, p, a in outs:
        assert (p - want[i][0]).abs().max().item() <= 1e-6, i
        wl = wls[i]
        for n in range(wl.n_branches):
            x = np.sort(want[i][0][wl.label_off[n]:wl.label_off[n + 1]].numpy())[::-1]
            if x[0] - x[1] > 1e-4:
                assert a[n] == want[i][1][n], (i, n)


def test_host_pass_checks_host_shapes(cuda_dev, lib):
    """Host inputs that do not match the model shape are refused before the
    native call reads them."""
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    from prefill_only_shared_gb300.workloads import make_workload
    wl = make_workload("tiny", seed=0)
    sh = wl.shape
    clf = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=cuda_dev)
    p = torch.empty(int(wl.label_off[-1]), dtype=torch.float32).pin_memory()
    a = torch.empty(wl.n_branches, dtype=torch.int32).pin_memory()
    with pytest.raises(ValueError):
        clf.run_from_host(wl.req_of_branch, wl.tok_offsets, wl.tokens, wl.q, wl.k[:-1], wl.v,
                          wl.h, wl.W.to(cuda_dev), torch.from_numpy(wl.label_off),
                          torch.from_numpy(wl.label_ids), p, a, schedule="tree")


@pytest.mark.parametrize("name", ["tiny", "yesno", "choice64"])
def test_native_pass_matches_the_orchestrated_pass(cuda_dev, lib, name):
    """sp_run_pass (plan, upload, tree attention, readout and softmax in one
    call) gives the results of the Python orchestration of the same calls;
    its first call grows the descriptor and workspace buffers from the sizes
    it reports."""
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    from prefill_only_shared_gb300.workloads import make_workload
    wl = make_workload(name, seed=0)
    sh = wl.shape
    dev = cuda_dev
    args = (wl.req_of_branch, wl.tok_offsets, wl.tokens, wl.q.to(dev), wl.k.to(dev),
            wl.v.to(dev), wl.h.to(dev), wl.W.to(dev), torch.from_numpy(wl.label_off).to(dev),
            torch.from_numpy(wl.label_ids).to(dev))
    ref = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=dev)
    r = ref.run(*args, schedule="tree")
    torch.cuda.synchronize()
    want = {k: getattr(r, k).float().cpu().clone() for k in ("out", "lse", "probs")}
    want_am = r.argmax.cpu().clone()
    nat = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=dev)
    for _ in range(2):  # the first call grows the buffers, the second reuses them
        g = nat.run_pass(*args)
        torch.cuda.synchronize()
        sp.sp_check_device_error()
        assert nat.last_pass_launches >= 3
        assert torch.equal(g.out.float().cpu(), want["out"])
        assert torch.equal(g.lse.cpu(), want["lse"])
        assert (g.probs.cpu() - want["probs"]).abs().max().item() <= 1e-6
        p = want["probs"].numpy()
        for n in range(wl.n_branches):
            x = np.sort(p[wl.label_off[n]:wl.label_off[n + 1]])[::-1]
            if x[0] - x[1] > 1e-4:
                assert g.argmax[n].item() == want_am[n].item()
