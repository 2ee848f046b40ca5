"""GPU parity of the question-type decision (sp_label_decide,
sp_candidate_decide) against oracle/postprocess.py on the same fp32 inputs,
plus its device-side error reporting and one end-to-end pass of the
two-level-tree workload.

Tolerances (fp32 kernel arithmetic with the fast exponential, float64 oracle,
identical fp32 inputs): probabilities and distributions 1e-5 abs, noul /
choice values 1e-5, score values 5e-4 (a sum of up to 64 terms i * p_i with
i <= 63), confidence 1e-4; argmax identical (both sides compare the same fp32
inputs).  The probabilities of sp_label_decide equal those of
sp_label_softmax bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import postprocess as PP

pytestmark = pytest.mark.gpu

TOL_P = 1e-5
TOL_V = 1e-5
TOL_SCORE = 5e-4
TOL_C = 1e-4


def _dev(a, dtype):
    return torch.as_tensor(np.ascontiguousarray(a)).to(dtype).cuda()


def _random_labels(rng, N, kmin=2, kmax=64):
    counts = rng.integers(kmin, kmax + 1, N)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    # logprobs of a softmax over a random vocabulary slice: negative, spread out
    lp = (-rng.gamma(2.0, 3.0, int(off[-1]))).astype(np.float32)
    return off, lp


def _check_values(val, ref_val, qtype, tol_score=TOL_SCORE):
    for n, qt in enumerate(qtype):
        tol = tol_score if qt == PP.SCORE else TOL_V
        assert abs(val[n] - ref_val[n]) <= tol, (n, qt, val[n], ref_val[n])


def test_label_decide_matches_oracle(cuda_dev, lib):
    from prefill_only_shared_gb300 import sp
    rng = np.random.default_rng(11)
    N = 1003
    off, lp = _random_labels(rng, N)
    lp[off[5]:off[5] + 2] = lp[off[5]:off[6]].max() + 1.0  # an exact tie: lowest index wins
    qtype = rng.integers(0, 3, N).astype(np.int32)
    d_lp, d_off, d_qt = _dev(lp, torch.float32), _dev(off, torch.int32), _dev(qtype, torch.int32)
    probs = torch.empty(int(off[-1]), device=cuda_dev)
    am = torch.empty(N, dtype=torch.int32, device=cuda_dev)
    val = torch.empty(N, device=cuda_dev)
    conf = torch.empty(N, device=cuda_dev)
    sp.sp_label_decide(d_lp, d_off, d_qt, probs, am, val, conf)
    probs2 = torch.empty_like(probs)
    am2 = torch.empty_like(am)
    sp.sp_label_softmax(d_lp, d_off, probs2, am2)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    assert torch.equal(probs, probs2) and torch.equal(am, am2)
    r_p, r_am, r_v, r_c = PP.label_decide(lp.astype(np.float64), off, qtype)
    assert np.abs(probs.cpu().numpy() - r_p).max() <= TOL_P
    assert (am.cpu().numpy() == r_am).all()
    assert am[5].item() == 0
    _check_values(val.cpu().numpy(), r_v, qtype)
    assert np.abs(conf.cpu().numpy() - r_c).max() <= TOL_C


def test_label_decide_printed_examples(cuda_dev, lib):
    """The refund example (P(yes) 0.77), the confidence example (0.641) and
    the score example (1.0), through the kernel."""
    from prefill_only_shared_gb300 import sp
    groups = [[-0.3, -1.5], list(np.log([0.9, 0.05, 0.05])), list(np.log([0.2, 0.6, 0.2]))]
    off = np.concatenate([[0], np.cumsum([len(g) for g in groups])]).astype(np.int32)
    lp = np.concatenate(groups).astype(np.float32)
    qtype = np.array([PP.NOUL, PP.CHOICE, PP.SCORE], np.int32)
    probs = torch.empty(len(lp), device=cuda_dev)
    am = torch.empty(3, dtype=torch.int32, device=cuda_dev)
    val = torch.empty(3, device=cuda_dev)
    conf = torch.empty(3, device=cuda_dev)
    sp.sp_label_decide(_dev(lp, torch.float32), _dev(off, torch.int32), _dev(qtype, torch.int32),
                       probs, am, val, conf)
    sp.sp_check_device_error()
    v, c = val.cpu().numpy(), conf.cpu().numpy()
    assert round(float(v[0]), 2) == 0.77
    assert round(float(c[1]), 3) == 0.641 and abs(v[1] - 0.9) < 1e-5
    assert abs(v[2] - 1.0) < 1e-5 and am.cpu().tolist() == [0, 0, 1]


def test_label_decide_device_errors(cuda_dev, lib):
    from prefill_only_shared_gb300 import sp
    off = np.array([0, 1, 3, 68, 70], np.int32)  # counts 1, 2, 65, 2
    lp = np.linspace(-3, -0.1, 70).astype(np.float32)
    qtype = np.array([0, 1, 2, 9], np.int32)  # the last type is not a question type
    probs = torch.zeros(70, device=cuda_dev)
    am = torch.empty(4, dtype=torch.int32, device=cuda_dev)
    val = torch.empty(4, device=cuda_dev)
    conf = torch.empty(4, device=cuda_dev)
    sp.sp_label_decide(_dev(lp, torch.float32), _dev(off, torch.int32), _dev(qtype, torch.int32),
                       probs, am, val, conf)
    with pytest.raises(sp.SpError) as e:
        sp.sp_check_device_error()
    assert e.value.status == 6
    a, v, c = am.cpu().tolist(), val.cpu().numpy(), conf.cpu().numpy()
    assert a[0] == -1 and a[2] == -1 and np.isnan(v[[0, 2]]).all() and np.isnan(c[[0, 2]]).all()
    assert np.isnan(probs[0].item()) and torch.isnan(probs[3:68]).all()
    assert a[1] == 1 and not np.isnan(v[1])
    assert np.isnan(v[3]) and not np.isnan(c[3]) and a[3] == 1  # probabilities still written
    sp.sp_check_device_error()  # cleared


def test_candidate_decide_matches_oracle(cuda_dev, lib):
    from prefill_only_shared_gb300 import sp
    rng = np.random.default_rng(12)
    sizes, qtype = [], []
    for q in range(300):
        t = int(rng.integers(0, 3))
        sizes.append(1 if t == PP.NOUL else int(rng.integers(2, 65)))
        qtype.append(t)
    sizes[3], qtype[3] = 64, PP.SCORE
    cand_off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    n_branches = int(cand_off[-1]) + 5  # trailing branches outside every question
    off, lp = _random_labels(rng, n_branches, 2, 8)
    # branch probabilities from a float64 softmax, stored as fp32
    probs = np.empty(len(lp), np.float32)
    for b in range(n_branches):
        x = lp[off[b]:off[b + 1]].astype(np.float64)
        e = np.exp(x - x.max())
        probs[off[b]:off[b + 1]] = e / e.sum()
    Q = len(sizes)
    qtype = np.asarray(qtype, np.int32)
    dist = torch.full((n_branches,), -7.0, device=cuda_dev)
    am = torch.empty(Q, dtype=torch.int32, device=cuda_dev)
    val = torch.empty(Q, device=cuda_dev)
    conf = torch.empty(Q, device=cuda_dev)
    sp.sp_candidate_decide(_dev(probs, torch.float32), _dev(off, torch.int32),
                           _dev(cand_off, torch.int32), _dev(qtype, torch.int32), dist, am, val, conf)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    r_d, r_am, r_v, r_c = PP.candidate_decide(probs.astype(np.float64), off, cand_off, qtype)
    g_d = dist.cpu().numpy()
    assert np.abs(g_d[:cand_off[-1]] - r_d).max() <= TOL_P
    assert (g_d[cand_off[-1]:] == -7.0).all()  # nothing written past the last question
    assert (am.cpu().numpy() == r_am).all()
    _check_values(val.cpu().numpy(), r_v, qtype)
    assert np.abs(conf.cpu().numpy() - r_c).max() <= TOL_C


def test_candidate_decide_device_errors(cuda_dev, lib):
    from prefill_only_shared_gb300 import sp
    n_branches = 6
    off = np.arange(0, 13, 2).astype(np.int32)
    probs = np.full(12, 0.5, np.float32)
    cases = [
        (np.array([0, 2], np.int32), [PP.NOUL]),     # noul with two candidates
        (np.array([0, 1], np.int32), [PP.CHOICE]),   # choice with one candidate
        (np.array([0, 3], np.int32), [7]),           # not a question type
        (np.array([0, 3, 9], np.int32), [PP.CHOICE, PP.SCORE]),  # past n_branches
    ]
    for cand_off, qtype in cases:
        Q = len(qtype)
        dist = torch.zeros(n_branches, device=cuda_dev)
        am = torch.empty(Q, dtype=torch.int32, device=cuda_dev)
        val = torch.empty(Q, device=cuda_dev)
        conf = torch.empty(Q, device=cuda_dev)
        sp.sp_candidate_decide(_dev(probs, torch.float32), _dev(off, torch.int32),
                               _dev(cand_off, torch.int32), _dev(np.asarray(qtype, np.int32), torch.int32),
                               dist, am, val, conf)
        with pytest.raises(sp.SpError) as e:
            sp.sp_check_device_error()
        assert e.value.status == 6
        assert am[-1].item() == -1 and torch.isnan(val[-1]) and torch.isnan(conf[-1])
    sp.sp_check_device_error()


def test_two_level_tree_end_to_end(cuda_dev, lib):
    """The two-level-tree workload as the LLM2Jev page's request: question 0
    (department, a choice) over branches 0..2 and question 1 (severity, a
    score) over branches 3..5, every branch a yes/no readout.  Branch
    probabilities are checked against the oracle's from its own logprobs; the
    assembly against the oracle applied to the GPU's probabilities."""
    from oracle import label_softmax as OL
    from oracle import readout as OR
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.workloads import make_workload
    wl = make_workload("tree2")
    sh = wl.shape
    clf = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=cuda_dev)
    N = wl.n_branches
    qt_branch = torch.full((N,), PP.NOUL, dtype=torch.int32, device=cuda_dev)
    res = clf.run(wl.req_of_branch, wl.tok_offsets, wl.tokens, wl.q.cuda(), wl.k.cuda(),
                  wl.v.cuda(), wl.h.cuda(), wl.W.cuda(), _dev(wl.label_off, torch.int32),
                  _dev(wl.label_ids, torch.int32), qtype=qt_branch)
    cand_off = _dev(np.array([0, 3, 6], np.int32), torch.int32)
    qtype = _dev(np.array([PP.CHOICE, PP.SCORE], np.int32), torch.int32)
    dist, am, val, conf = clf.candidates(res.probs, _dev(wl.label_off, torch.int32), cand_off, qtype)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    lp, _ = OR.label_logprobs(wl.h, wl.W, wl.label_off, wl.label_ids)
    r_probs, _ = OL.label_softmax(lp, wl.label_off)
    g_probs = res.probs.cpu().numpy()
    assert np.abs(g_probs - r_probs).max() <= 1e-3
    assert np.abs(res.value.cpu().numpy() - r_probs[wl.label_off[:-1]]).max() <= 1e-3
    r_d, r_am, r_v, r_c = PP.candidate_decide(g_probs.astype(np.float64), wl.label_off,
                                              np.array([0, 3, 6]), [PP.CHOICE, PP.SCORE])
    assert np.abs(dist.cpu().numpy()[:6] - r_d).max() <= TOL_P
    assert (am.cpu().numpy() == r_am).all()
    v = val.cpu().numpy()
    assert abs(v[0] - r_v[0]) <= TOL_V and abs(v[1] - r_v[1]) <= TOL_SCORE
    assert np.abs(conf.cpu().numpy() - r_c).max() <= TOL_C
