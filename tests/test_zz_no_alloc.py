"""The no-allocation readout entry point (sp_label_logprobs_noalloc).

It exists for callers that cannot allocate device memory, such as a serving
loop that hands out every device buffer from an arena sized at start-up and
allows no allocation afterwards, or a plain C host program that links only
libsp and has no device allocator of its own.  Its scratch is a static device
array inside the library, shared by every call.

Checked here through the C-ABI, on calls in a row (each with a different
branch count, so stale scratch contents from the call before would show):
against the float64 oracle (oracle/readout.py) at the readout's parity
tolerance (1e-2 on log-probabilities and lse), and against the
workspace-taking entry point at the same tolerance.  The largest accepted
branch count (1024: four column chunks, the largest partials footprint in the
array) is one of the cases.  Every successful call is one launch, and the
size limit is rejected before anything is launched.  This file is collected
last on purpose.
"""
import numpy as np
import pytest
import torch

from oracle import readout as OR

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _inputs(N, V, H, seed, dev):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(N, H, generator=g).bfloat16()
    W = (torch.randn(V, H, generator=g) * 0.05).bfloat16()
    counts = torch.randint(2, 9, (N,), generator=g)
    off = torch.cat([torch.zeros(1, dtype=torch.int64), counts.cumsum(0)]).to(torch.int32)
    ids = torch.randint(0, V, (int(off[-1]),), generator=g, dtype=torch.int32)
    return h, W, off, ids, int(off[-1])


def _with_workspace(sp, h, W, off, ids, n_labels, dev):
    N, V = h.shape[0], W.shape[0]
    ws = torch.empty(sp.sp_label_workspace_bytes(N, V), dtype=torch.uint8, device=dev)
    lp = torch.empty(n_labels, device=dev)
    lse = torch.empty(N, device=dev)
    sp.sp_label_logprobs(h, W, off, ids, n_labels, lp, lse, ws)
    return lp, lse


def test_noalloc_matches_oracle_and_workspace_entry_point(cuda_dev, lib):
    sp = lib
    dev = cuda_dev
    # (N, V, H, seed): two column chunks; the yes/no LM head; the largest N
    cases = [(300, 20000, 256, 1), (7, 151936, 2048, 2), (1024, 3000, 128, 3)]
    for N, V, H, seed in cases:
        h, W, off, ids, n_labels = _inputs(N, V, H, seed, dev)
        ref_lp, ref_lse = OR.label_logprobs(h, W, off.numpy(), ids.numpy())
        hd, Wd, offd, idsd = h.to(dev), W.to(dev), off.to(dev), ids.to(dev)
        ws_lp, ws_lse = _with_workspace(sp, hd, Wd, offd, idsd, n_labels, dev)
        lp = torch.full((n_labels,), float("nan"), device=dev)
        lse = torch.full((N,), float("nan"), device=dev)
        sp.sp_label_logprobs_noalloc(hd, Wd, offd, idsd, n_labels, lp, lse)
        assert sp.sp_last_launch_count() == 1
        torch.cuda.synchronize()
        sp.sp_check_device_error()
        assert not torch.isnan(lp).any() and not torch.isnan(lse).any()
        lp_np, lse_np = lp.cpu().numpy(), lse.cpu().numpy()
        assert np.abs(lp_np - ref_lp).max() <= TOL, f"N={N}: logprobs vs oracle"
        assert np.abs(lse_np - ref_lse).max() <= TOL, f"N={N}: lse vs oracle"
        assert (lp - ws_lp).abs().max().item() <= TOL
        assert (lse - ws_lse).abs().max().item() <= TOL


def test_noalloc_rejects_too_many_branches(cuda_dev, lib):
    sp = lib
    dev = cuda_dev
    N = 1025
    h = torch.zeros(N, 64, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(100, 64, dtype=torch.bfloat16, device=dev)
    off = torch.arange(0, 2 * N + 1, 2, dtype=torch.int32, device=dev)
    ids = torch.zeros(2 * N, dtype=torch.int32, device=dev)
    lp = torch.empty(2 * N, device=dev)
    lse = torch.empty(N, device=dev)
    with pytest.raises(sp.SpError) as e:
        sp.sp_label_logprobs_noalloc(h, W, off, ids, 2 * N, lp, lse)
    assert e.value.status == 7
    assert sp.sp_last_launch_count() == 0
