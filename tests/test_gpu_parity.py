"""GPU parity: libsp (through the C-ABI) against the CPU oracle on the same
seeded inputs.  Small cases are compared element by element; the full-size
workloads on sampled rows / branches."""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import staging as OS
from prefill_only_shared_gb300.workloads import make_workload, small_case

from gpu_helpers import (TOL_LSE, TOL_OUT, check_attention_full, check_attention_sampled,
                         check_attention_suffix_rows, check_readout, run_gpu)

pytestmark = pytest.mark.gpu

_CACHE = {}


def workload(name):
    if name not in _CACHE:
        _CACHE[name] = make_workload(name)
    return _CACHE[name]


def test_tiny_full(cuda_dev, lib):
    wl = workload("tiny")
    g = run_gpu(wl)
    assert g["rounds"] == [[0], [1, 2, 3]]
    check_attention_full(wl, g)
    check_readout(wl, g)


SMALL = [
    # (trees, Hq, Hkv, d, hidden, vocab, labels)
    ([(130, [(70, [(3, []), (65, []), (1, [])]), (17, [])]), (40, []), (5, [(1, []), (200, [])])],
     8, 2, 64, 128, 1000, ("per_branch", 2)),
    ([(33, [(1, []), (2, []), (150, [])])], 32, 4, 128, 200, 129, ("per_branch_range", (2, 64))),
    ([(300, [(45, []) for _ in range(7)])], 16, 1, 128, 64, 4096, ("shared", 64)),
    ([(1, [(1, []), (1, [])]), (257, [])], 2, 2, 64, 256, 5000, ("per_branch", 3)),
    ([(77, [(20, [(9, []), (10, [])]), (21, [(11, []), (12, [])])])], 4, 4, 128, 512, 777,
     ("per_branch", 5)),
]


@pytest.mark.parametrize("schedule", ["rounds", "all", "tree"])
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_ragged_cases(cuda_dev, lib, case, schedule):
    trees, Hq, Hkv, d, H, V, labels = SMALL[case]
    wl = small_case(trees, seed=case, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, hidden=H,
                    vocab=V, labels=labels)
    g = run_gpu(wl, schedule=schedule)
    check_attention_full(wl, g)
    check_readout(wl, g)


@pytest.mark.parametrize("schedule", ["rounds", "tree"])
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_cases_with_paired_tails(cuda_dev, lib, case, schedule):
    """Planned for one SM: no split parts, and sibling leaf tails that fit a
    half share a CTA (half A one leaf's tail, half B the other's)."""
    import sys
    sys.path.insert(0, __import__("os").path.dirname(__file__))
    from test_plan_descriptor import decode
    trees, Hq, Hkv, d, H, V, labels = SMALL[case]
    wl = small_case(trees, seed=case, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, hidden=H,
                    vocab=V, labels=labels)
    g = run_gpu(wl, schedule=schedule, n_sms=1)
    check_attention_full(wl, g)
    check_readout(wl, g)
    tiles = decode(g["plan"].descriptor())[4]
    if case in (0, 1, 3, 4):  # cases with sibling leaf tails short enough to pair
        assert (tiles["seg2"] >= 0).any()


def test_recomputed_final_rows(cuda_dev, lib):
    """Branches equal to, or prefixes of, other branches: their last row is
    cached before their round and is recomputed (same value)."""
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    rng = np.random.default_rng(5)
    base = list(rng.integers(0, 50, 90))
    seqs = [base, base + [7, 8, 9], base, base[:40], base[:40] + [3] * 20]
    off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
    toks = np.concatenate(seqs).astype(np.int32)
    req = np.zeros(len(seqs), np.int32)
    ref = OS.build_plan(req, off, toks)
    assert any(ref.recompute)
    T = ref.node_tokens
    gen = torch.Generator().manual_seed(0)
    q = torch.randn(T, 8, 64, generator=gen).bfloat16()
    k = torch.randn(T, 2, 64, generator=gen).bfloat16()
    v = torch.randn(T, 2, 64, generator=gen).bfloat16()
    clf = SharedPrefixClassifier(8, 2, 64, 64, 100, device=cuda_dev)
    plan = clf.plan(req, off, toks)
    ro, rl, _ = OA.reference_attention(ref, q, k, v)
    for schedule in ("rounds", "all", "tree"):
        out, lse = clf.attention(plan, q.cuda(), k.cuda(), v.cuda(), schedule=schedule)
        torch.cuda.synchronize()
        sp.sp_check_device_error()
        assert np.abs(out.float().cpu().numpy() - ro).max() <= TOL_OUT
        assert np.abs(lse.cpu().numpy() - rl).max() <= TOL_LSE


@pytest.mark.parametrize("schedule", ["rounds", "all", "tree"])
@pytest.mark.parametrize("name", ["yesno", "tree2", "choice64"])
def test_full_size_configs(cuda_dev, lib, name, schedule):
    wl = workload(name)
    g = run_gpu(wl, schedule=schedule)
    expected = {"yesno": [[0], [1, 2, 3, 4]], "tree2": [[0], [1, 2, 3], [4, 5]],
                "choice64": [[0], list(range(1, 64))]}[name]
    assert g["rounds"] == expected
    check_attention_sampled(wl, g, n_random=96)
    # every branch: all of its suffix rows, its readout, softmax and argmax
    check_attention_suffix_rows(wl, g)
    check_readout(wl, g)


@pytest.mark.parametrize("schedule", ["rounds", "tree"])
def test_full_size_batch64(cuda_dev, lib, schedule):
    wl = workload("batch64")
    g = run_gpu(wl, schedule=schedule)
    assert len(g["rounds"]) == 2 and len(g["rounds"][0]) == 64
    check_attention_sampled(wl, g, n_random=128)
    if schedule == "tree":
        # the bench's schedule: every one of the 768 branches, all 49152 suffix
        # rows and every readout, softmax and argmax
        check_attention_suffix_rows(wl, g)
        check_readout(wl, g)
    else:
        check_readout(wl, g, [0, 1, 11, 12, 100, 383, 500, 767])
    if schedule == "tree":
        _CACHE.pop("batch64", None)


@pytest.mark.parametrize("N,V,H", [(1, 1000, 64), (17, 129, 128), (300, 3000, 136), (1100, 700, 64)])
def test_readout_shapes(cuda_dev, lib, N, V, H):
    """Branch counts across the 16-column granularity and two column chunks,
    vocab sizes with a partial last tile, hidden sizes that end mid-stage."""
    from prefill_only_shared_gb300 import sp
    gen = torch.Generator().manual_seed(N + V)
    h = torch.randn(N, H, generator=gen).bfloat16()
    W = (torch.randn(V, H, generator=gen) * 0.5).bfloat16()
    counts = torch.randint(2, 9, (N,), generator=gen).numpy()
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ids = torch.randint(0, V, (int(off[-1]),), generator=gen).numpy().astype(np.int32)
    ids[0], ids[-1] = 0, V - 1
    from types import SimpleNamespace
    wl = SimpleNamespace(h=h, W=W, label_off=off, label_ids=ids, n_branches=N)
    dev = cuda_dev
    ws = torch.empty(sp.sp_label_workspace_bytes(N, V), dtype=torch.uint8, device=dev)
    lp = torch.full((int(off[-1]),), float("nan"), device=dev)
    lse = torch.empty(N, device=dev)
    probs = torch.empty_like(lp)
    am = torch.empty(N, dtype=torch.int32, device=dev)
    offd, idsd = torch.from_numpy(off).to(dev), torch.from_numpy(ids).to(dev)
    sp.sp_label_logprobs(h.to(dev), W.to(dev), offd, idsd, int(off[-1]), lp, lse, ws)
    sp.sp_label_softmax(lp, offd, probs, am)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    g = {"logprobs": lp.cpu().numpy(), "lse_vocab": lse.cpu().numpy(), "probs": probs.cpu().numpy(),
         "argmax": am.cpu().numpy()}
    check_readout(wl, g, list(range(N)) if N <= 64 else list(range(0, N, 7)) + [N - 1])


def test_device_bounds_errors(cuda_dev, lib):
    """An id outside [0, V) and a label count of 1 are reported through the
    device error word, with NaN / -1 outputs, and the context stays usable."""
    from prefill_only_shared_gb300 import sp
    dev = cuda_dev
    N, V, H = 3, 500, 64
    h = torch.randn(N, H, device=dev).bfloat16()
    W = torch.randn(V, H, device=dev).bfloat16()
    off = torch.tensor([0, 2, 4, 6], dtype=torch.int32, device=dev)
    ids = torch.tensor([1, 2, 3, V + 5, 7, 8], dtype=torch.int32, device=dev)
    ws = torch.empty(sp.sp_label_workspace_bytes(N, V), dtype=torch.uint8, device=dev)
    lp = torch.empty(6, device=dev)
    lse = torch.empty(N, device=dev)
    sp.sp_label_logprobs(h, W, off, ids, 6, lp, lse, ws)
    with pytest.raises(sp.SpError) as e:
        sp.sp_check_device_error()
    assert e.value.status == 6
    assert torch.isnan(lp[3]) and not torch.isnan(lp[[0, 1, 2, 4, 5]]).any()
    sp.sp_check_device_error()  # cleared
    off1 = torch.tensor([0, 1, 3], dtype=torch.int32, device=dev)
    probs = torch.empty(3, device=dev)
    am = torch.empty(2, dtype=torch.int32, device=dev)
    sp.sp_label_softmax(lp[:3].contiguous(), off1, probs, am)
    with pytest.raises(sp.SpError) as e:
        sp.sp_check_device_error()
    assert e.value.status == 6
    assert am[0].item() == -1 and am[1].item() in (0, 1)


def test_host_argument_errors(cuda_dev, lib):
    from prefill_only_shared_gb300 import sp
    dev = cuda_dev
    h = torch.randn(2, 60, device=dev).bfloat16()  # hidden not a multiple of 8
    W = torch.randn(10, 60, device=dev).bfloat16()
    off = torch.tensor([0, 2, 4], dtype=torch.int32, device=dev)
    ids = torch.tensor([1, 2, 3, 4], dtype=torch.int32, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    lp = torch.empty(4, device=dev)
    lse = torch.empty(2, device=dev)
    with pytest.raises(sp.SpError) as e:
        sp.sp_label_logprobs(h, W, off, ids, 4, lp, lse, ws)
    assert e.value.status == 1
    h = torch.randn(2, 64, device=dev).bfloat16()
    W = torch.randn(10, 64, device=dev).bfloat16()
    with pytest.raises(sp.SpError) as e:
        sp.sp_label_logprobs(h, W, off, ids, 4, lp, lse, ws[:8])
    assert e.value.status == 7
