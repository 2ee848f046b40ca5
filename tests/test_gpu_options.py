"""GPU parity of multi-token option scoring and label-prior calibration
(sp_label_logprobs with one label per row, then sp_option_softmax) against
oracle/options.py on the same seeded bf16 inputs, through the C-ABI.

Tolerances: row log-probabilities 1e-2 (the readout's bar); an option score
sums m row terms, so m * 1e-2; the option softmax against the oracle taken
from the kernel's own fp32 row log-probabilities 1e-5 (fp32 sums and the
fast exponential over float64); the argmax identical wherever the oracle's
top-2 probability margin exceeds 1e-2, and equal to the argmax of the float64
softmax of the kernel's own row log-probabilities wherever that has no
near-tie.
"""
import numpy as np
import pytest
import torch

from oracle import options as OP
from oracle import label_softmax as LS

pytestmark = pytest.mark.gpu

TOL_LP = 1e-2
TOL_P_SELF = 1e-5
MARGIN = 1e-2


def _dev(a, dtype):
    return torch.as_tensor(np.ascontiguousarray(a)).to(dtype).cuda()


def _run(wl, prior):
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    dev = torch.device("cuda:0")
    clf = SharedPrefixClassifier(8, 2, 64, wl.hidden, wl.vocab, device=dev)
    sp.sp_check_options(wl.opt_off, wl.n_rows, wl.q_off)
    pr = _dev(wl.prior, torch.float32) if prior else None
    lp, sc, pb, am = clf.options(wl.h_rows.to(dev), wl.W.to(dev), _dev(wl.opt_off, torch.int32),
                                 _dev(wl.tokens, torch.int32), _dev(wl.q_off, torch.int32), pr)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    return (lp.cpu().numpy().astype(np.float64), sc.cpu().numpy(), pb.cpu().numpy(),
            am.cpu().numpy(), clf.last_option_launches)


def _check(wl, prior):
    lp, sc, pb, am, launches = _run(wl, prior)
    assert launches == 2  # the readout and the option softmax
    pri = wl.prior.astype(np.float64) if prior else None
    ref_lp, ref_sc, ref_p, ref_am = OP.option_readout(wl.h_rows, wl.W, wl.opt_off, wl.tokens,
                                                      wl.q_off, pri)
    assert np.abs(lp - ref_lp).max() <= TOL_LP
    m = np.diff(wl.opt_off)
    assert np.all(np.abs(sc - ref_sc) <= m * TOL_LP)
    # the kernel's own arithmetic, from its fp32 row log-probabilities
    self_sc, self_p, self_am = OP.option_softmax(lp, wl.opt_off, wl.q_off, pri)
    assert np.abs(sc - self_sc).max() <= 1e-4 * np.abs(self_sc).max()
    assert np.abs(pb - self_p).max() <= TOL_P_SELF
    clear = LS.top2_margin(self_p, wl.q_off) > 1e-6  # no near-tie within fp32 rounding
    assert np.array_equal(am[clear], self_am[clear])
    margin = LS.top2_margin(ref_p, wl.q_off)
    sel = margin > MARGIN
    assert np.array_equal(am[sel], ref_am[sel])
    return sel.sum()


@pytest.mark.parametrize("prior", [False, True])
def test_options_small_vocab(cuda_dev, lib, prior):
    from prefill_only_shared_gb300.workloads import make_options
    wl = make_options(seed=5, n_questions=23, opts=(2, 64), tokens=(1, 5), hidden=200,
                      vocab=1000, w_std=0.3)
    assert _check(wl, prior) > 0


@pytest.mark.parametrize("prior", [False, True])
def test_options_full_vocab(cuda_dev, lib, prior):
    """The yes/no configuration's LM head (H 2048, V 151936): 16 questions of
    2..8 options of 1..4 tokens."""
    from prefill_only_shared_gb300.workloads import make_options
    wl = make_options(seed=0, w_std=0.05)
    _check(wl, prior)


def test_one_token_options_equal_the_label_softmax(cuda_dev, lib):
    """One-token options without a prior give the label softmax bit for bit."""
    from prefill_only_shared_gb300 import sp
    rng = np.random.default_rng(2)
    q_off = np.concatenate([[0], np.cumsum(rng.integers(2, 65, 40))]).astype(np.int32)
    n = int(q_off[-1])
    lp = (-rng.gamma(2.0, 3.0, n)).astype(np.float32)
    d_lp = _dev(lp, torch.float32)
    opt_off = _dev(np.arange(n + 1), torch.int32)
    d_q = _dev(q_off, torch.int32)
    sc = torch.empty(n, device=cuda_dev)
    pb = torch.empty(n, device=cuda_dev)
    am = torch.empty(len(q_off) - 1, dtype=torch.int32, device=cuda_dev)
    sp.sp_option_softmax(d_lp, opt_off, d_q, sc, pb, am)
    p2 = torch.empty(n, device=cuda_dev)
    a2 = torch.empty_like(am)
    sp.sp_label_softmax(d_lp, d_q, p2, a2)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    assert torch.equal(sc.cpu(), d_lp.cpu())
    assert torch.equal(pb.cpu(), p2.cpu()) and torch.equal(am.cpu(), a2.cpu())


def test_option_bounds_reported(cuda_dev, lib):
    """A question with one option, and an option without rows: NaN / -1 for
    that question, SP_ERR_DEVICE_BOUNDS from the error word; the other
    question is computed."""
    from prefill_only_shared_gb300 import sp
    lp = _dev(np.array([-1.0, -2.0, -3.0, -0.5, -0.7], np.float32), torch.float32)
    for opt_off, q_off in (([0, 1, 2, 3, 5], [0, 1, 4]),      # 1 option, then 3
                           ([0, 1, 1, 3, 5], [0, 2, 4])):     # option 1 has no rows
        d_oo, d_q = _dev(opt_off, torch.int32), _dev(q_off, torch.int32)
        n_opts, Q = len(opt_off) - 1, len(q_off) - 1
        sc = torch.zeros(n_opts, device=cuda_dev)
        pb = torch.zeros(n_opts, device=cuda_dev)
        am = torch.zeros(Q, dtype=torch.int32, device=cuda_dev)
        sp.sp_option_softmax(lp, d_oo, d_q, sc, pb, am)
        with pytest.raises(sp.SpError) as e:
            sp.sp_check_device_error()
        assert e.value.status == 6  # SP_ERR_DEVICE_BOUNDS
        a = am.cpu().numpy()
        assert a[0] == -1 and np.isnan(pb.cpu().numpy()[q_off[0]:q_off[1]]).all()
        assert a[1] >= 0 and np.isfinite(pb.cpu().numpy()[q_off[1]:q_off[2]]).all()
