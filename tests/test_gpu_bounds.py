"""Device-side bounds checks of the attention path.

The openjev-sglang article's limits section rejects bad input before
inference; the kernels add the device form of that rule for what the host
cannot see, a stale or mismatched launch descriptor.  A page id outside the
pages the plan may name, or a row outside the q / k / v / out inputs, sets the
bounds bit of the device error word (SP_ERR_DEVICE_BOUNDS) and the access is
skipped: a pool store is not made, a pool fetch reads the pool maps'
out-of-range fill (NaN), so the rows that use it come out NaN.

No out-of-bounds access happens here: the pool is allocated with more pages
than the plan declares, and the corrupted page id points inside that
allocation, past the plan's pages.  The extra pages hold a sentinel that must
survive.
"""
import math
import os
import sys

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import staging as OS
from prefill_only_shared_gb300.workloads import small_case

sys.path.insert(0, os.path.dirname(__file__))
from gpu_helpers import TOL_OUT  # noqa: E402
from test_plan_descriptor import decode  # noqa: E402

pytestmark = pytest.mark.gpu

EXTRA_PAGES = 8
SENTINEL = 7.0


def _setup(dev):
    from prefill_only_shared_gb300 import sp
    wl = small_case((200, [(20, []), (20, []), (20, [])]), seed=3, n_q_heads=8, n_kv_heads=2,
                    head_dim=64)
    sh = wl.shape
    shape = sp.make_shape(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, 16, sh.hidden, sh.vocab)
    plan = sp.sp_plan_build(shape, wl.req_of_branch, wl.tok_offsets, wl.tokens, 1 << 20, 152)
    st = plan.stats()
    pool = torch.full((st["pages_used"] + EXTRA_PAGES, 2, sh.n_kv_heads, 16, sh.head_dim),
                      SENTINEL, dtype=torch.bfloat16, device=dev)
    T = st["node_tokens"]
    io = dict(q=wl.q.to(dev), k=wl.k.to(dev), v=wl.v.to(dev),
              out=torch.full((T, sh.n_q_heads, sh.head_dim), float("nan"), dtype=torch.bfloat16,
                             device=dev),
              lse=torch.full((T, sh.n_q_heads), float("nan"), device=dev),
              ws=torch.empty(max(st["attn_workspace_bytes"], 16), dtype=torch.uint8, device=dev))
    return sp, wl, plan, pool, io


def _upload(blob, dev):
    raw = torch.empty(len(blob) + 256, dtype=torch.uint8, device=dev)
    off = (-raw.data_ptr()) % 256
    d = raw[off:off + len(blob)]
    d.copy_(torch.frombuffer(bytearray(blob), dtype=torch.uint8))
    return d, raw


def _corrupt(blob, page_index, value):
    """The descriptor with page-table entry `page_index` set to `value`."""
    h = np.frombuffer(blob, dtype="<i8", count=12)
    b = bytearray(blob)
    pos = int(h[1]) + 4 * page_index
    b[pos:pos + 4] = np.int32(value).tobytes()
    return bytes(b)


def _prefix_seg(blob):
    segs = decode(blob)[0]
    idx = [i for i, s in enumerate(segs) if s["shared"] == 1]
    assert len(idx) == 1
    return segs[idx[0]]


def _call(sp, fn, plan, desc, rnd, pool, io):
    fn(plan, desc, rnd, io["q"], io["k"], io["v"], pool, io["out"], io["lse"], io["ws"])


def test_pool_fetch_with_bad_page_id(cuda_dev, lib):
    """Round 0's branch call reads the prefix from the pool; one of its page
    ids points past the plan's pages.  The bounds bit is set, the rows of the
    branch that read it are NaN, the prefix rows (the good call) match the
    oracle, and the pages past the plan keep their sentinel."""
    sp, wl, plan, pool, io = _setup(cuda_dev)
    n_pages = plan.stats()["pages_used"]
    blob = plan.descriptor()
    good, _g = _upload(blob, cuda_dev)
    pre = _prefix_seg(blob)
    bad, _b = _upload(_corrupt(blob, int(pre["page_off"]), n_pages + 2), cuda_dev)
    assert plan.rounds()[0] == [0]
    _call(sp, sp.sp_prefix_attn, plan, good, 0, pool, io)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    _call(sp, sp.sp_branch_attn, plan, bad, 0, pool, io)
    torch.cuda.synchronize()
    with pytest.raises(sp.SpError) as e:
        sp.sp_check_device_error()
    assert e.value.status == 6
    sp.sp_check_device_error()  # the word was cleared
    ref = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    leaf0 = ref.segments[ref.paths[0][-1]]
    rows = slice(leaf0.node_start, leaf0.node_start + leaf0.length)
    out = io["out"].float().cpu().numpy()
    lse = io["lse"].cpu().numpy()
    assert np.isnan(out[rows]).all() and np.isnan(lse[rows]).all()
    ro, _, _ = OA.reference_attention(ref, wl.q, wl.k, wl.v)
    prows = slice(int(pre["node_start"]), int(pre["node_start"]) + int(pre["len"]))
    assert np.abs(out[prows] - ro[prows]).max() <= TOL_OUT
    assert (pool[n_pages:].float() == SENTINEL).all()


def test_pool_store_with_bad_page_id(cuda_dev, lib):
    """The prefix call's second page id points past the plan's pages: its 16
    tokens are not stored (the bounds bit is set), the other pages of the
    prefix are, every page past the plan keeps its sentinel, and the prefix
    rows themselves (computed from the inputs) still match the oracle."""
    sp, wl, plan, pool, io = _setup(cuda_dev)
    n_pages = plan.stats()["pages_used"]
    blob = plan.descriptor()
    pre = _prefix_seg(blob)
    p0 = int(decode(blob)[1][int(pre["page_off"])])
    bad, _b = _upload(_corrupt(blob, int(pre["page_off"]) + 1, n_pages + 3), cuda_dev)
    _call(sp, sp.sp_prefix_attn, plan, bad, 0, pool, io)
    torch.cuda.synchronize()
    with pytest.raises(sp.SpError) as e:
        sp.sp_check_device_error()
    assert e.value.status == 6
    assert (pool[n_pages:].float() == SENTINEL).all()
    # the first page of the prefix holds its first 16 tokens' K (head 0)
    k0 = wl.k[int(pre["node_start"]):int(pre["node_start"]) + 16, 0].float()
    assert torch.equal(pool[p0, 0, 0].float().cpu(), k0)
    ref = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    ro, _, _ = OA.reference_attention(ref, wl.q, wl.k, wl.v)
    out = io["out"].float().cpu().numpy()
    prows = slice(int(pre["node_start"]), int(pre["node_start"]) + int(pre["len"]))
    assert np.abs(out[prows] - ro[prows]).max() <= TOL_OUT
    assert math.isfinite(float(io["lse"][prows].abs().max()))


def test_valid_descriptor_sets_no_bounds_bit(cuda_dev, lib):
    """The same calls with the plan's own descriptor: no error, every row of
    every branch matches the oracle."""
    sp, wl, plan, pool, io = _setup(cuda_dev)
    good, _g = _upload(plan.descriptor(), cuda_dev)
    for r in range(plan.stats()["n_rounds"]):
        _call(sp, sp.sp_prefix_attn, plan, good, r, pool, io)
        _call(sp, sp.sp_branch_attn, plan, good, r, pool, io)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    ref = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    ro, rl, _ = OA.reference_attention(ref, wl.q, wl.k, wl.v)
    assert np.abs(io["out"].float().cpu().numpy() - ro).max() <= TOL_OUT
    assert (pool[plan.stats()["pages_used"]:].float() == SENTINEL).all()
