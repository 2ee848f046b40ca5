"""Pins for the attention oracle (independent of its own formula code)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle import staging as S


def brute_force(q, k, v):
    """Scalar loops, Python floats: the definition written a second way."""
    L, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros((L, Hq, d))
    lse = np.zeros((L, Hq))
    for h in range(Hq):
        g = h // G
        for i in range(L):
            scores = []
            for j in range(i + 1):
                scores.append(sum(q[i, h, c] * k[j, g, c] for c in range(d)) / math.sqrt(d))
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            z = sum(w)
            for c in range(d):
                out[i, h, c] = sum(w[j] * v[j, g, c] for j in range(i + 1)) / z
            lse[i, h] = m + math.log(z)
    return out, lse


@pytest.mark.parametrize("L,Hq,Hkv,d", [(5, 4, 2, 8), (8, 2, 1, 4), (3, 6, 3, 5), (1, 2, 2, 3)])
def test_matches_brute_force(L, Hq, Hkv, d):
    rng = np.random.default_rng(L * 100 + d)
    q = rng.standard_normal((L, Hq, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, d))
    o, l = A.causal_attention(q, k, v)
    ob, lb = brute_force(q, k, v)
    assert np.abs(o - ob).max() < 1e-12
    assert np.abs(l - lb).max() < 1e-12


@pytest.mark.parametrize("L,Hq,Hkv,d", [(37, 8, 2, 64), (64, 32, 4, 128), (17, 4, 4, 16)])
def test_matches_library_sdpa(L, Hq, Hkv, d):
    """torch's scaled_dot_product_attention (float64, causal, GQA by
    repeat-interleave) is an independent library routine."""
    g = torch.Generator().manual_seed(L)
    q = torch.randn(L, Hq, d, generator=g, dtype=torch.float64)
    k = torch.randn(L, Hkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(L, Hkv, d, generator=g, dtype=torch.float64)
    ref = F.scaled_dot_product_attention(
        q.transpose(0, 1)[None], k.transpose(0, 1)[None], v.transpose(0, 1)[None],
        is_causal=True, enable_gqa=True)[0].transpose(0, 1).numpy()
    o, _ = A.causal_attention(q.numpy(), k.numpy(), v.numpy())
    assert np.abs(o - ref).max() < 1e-12


def test_single_key_returns_value():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 4, 8))
    k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 8))
    o, l = A.causal_attention(q, k, v)
    for h in range(4):
        assert np.allclose(o[0, h], v[0, h // 2], atol=0, rtol=1e-15)
        # lse of a single score is the score itself
        assert abs(l[0, h] - q[0, h] @ k[0, h // 2] / math.sqrt(8)) < 1e-14


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    L = 6
    q = rng.standard_normal((L, 2, 4))
    k = np.repeat(rng.standard_normal((1, 1, 4)), L, axis=0)
    v = rng.standard_normal((L, 1, 4))
    o, l = A.causal_attention(q, k, v)
    for i in range(L):
        assert np.allclose(o[i, 0], v[:i + 1, 0].mean(axis=0), atol=1e-14)
        s = q[i, 0] @ k[0, 0] / 2.0
        assert abs(l[i, 0] - (s + math.log(i + 1))) < 1e-13


def test_cascade_merge_equals_unshared():
    """Attention over [prefix | suffix] == LSE-weighted merge of the prefix
    part (all keys visible) and the causal suffix part."""
    rng = np.random.default_rng(3)
    P, Sfx, Hq, Hkv, d = 11, 7, 4, 2, 16
    q = rng.standard_normal((P + Sfx, Hq, d))
    k = rng.standard_normal((P + Sfx, Hkv, d))
    v = rng.standard_normal((P + Sfx, Hkv, d))
    full, full_l = A.causal_attention(q, k, v)
    for i in range(P, P + Sfx):
        o_pre, l_pre = A.attention_at(q[i], k[:P], v[:P])
        o_suf, l_suf = A.attention_at(q[i], k[P:i + 1], v[P:i + 1])
        lt = np.logaddexp(l_pre, l_suf)
        merged = np.exp(l_pre - lt)[:, None] * o_pre + np.exp(l_suf - lt)[:, None] * o_suf
        assert np.abs(merged - full[i]).max() < 1e-12
        assert np.abs(lt - full_l[i]).max() < 1e-12


def test_shared_rows_agree_and_sampling():
    from prefill_only_shared_gb300.workloads import small_case
    wl = small_case((9, [(5, [(3, []), (2, [])]), (4, [])]), n_q_heads=4, n_kv_heads=2, head_dim=8)
    plan = S.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    out, lse, worst = A.reference_attention(plan, wl.q, wl.k, wl.v)
    assert worst < 1e-12
    assert not np.isnan(out).any()
    rows = [0, 8, 9, 13, 15, 17]
    so, sl = A.sampled_attention(plan, wl.q, wl.k, wl.v, rows)
    assert np.abs(so - out[rows]).max() < 1e-12
    assert np.abs(sl - lse[rows]).max() < 1e-12


def test_prefix_free_sequence_is_plain_causal():
    """A request with one branch and no shared prefix is ordinary causal
    attention over that branch."""
    from prefill_only_shared_gb300.workloads import small_case
    wl = small_case((13, []), n_q_heads=4, n_kv_heads=1, head_dim=8)
    plan = S.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    out, _, _ = A.reference_attention(plan, wl.q, wl.k, wl.v)
    ob, _ = brute_force(A.to64(wl.q), A.to64(wl.k), A.to64(wl.v))
    assert np.abs(out - ob).max() < 1e-12


def test_branch_suffix_rows_match_brute_force_and_sdpa():
    """Every branch's suffix rows, computed for those rows alone, equal the
    scalar brute force over the branch's whole sequence (small tree) and
    torch's float64 SDPA over it (a larger GQA tree)."""
    from prefill_only_shared_gb300.workloads import small_case
    wl = small_case((6, [(4, [(3, []), (2, [])]), (5, [])]), n_q_heads=4, n_kv_heads=2, head_dim=8)
    plan = S.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    for b in range(len(plan.paths)):
        rows = A.branch_rows(plan, b)
        ob, lb = brute_force(A.to64(wl.q[rows]), A.to64(wl.k[rows]), A.to64(wl.v[rows]))
        srows, o, l = A.branch_suffix_attention(plan, wl.q, wl.k, wl.v, b)
        n = len(srows)
        assert (srows == rows[-n:]).all()
        assert np.abs(o - ob[-n:]).max() < 1e-12
        assert np.abs(l - lb[-n:]).max() < 1e-12
    wl = small_case((70, [(33, []), (9, [(20, []), (1, [])])]), n_q_heads=16, n_kv_heads=2,
                    head_dim=32)
    plan = S.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    for b in range(len(plan.paths)):
        rows = A.branch_rows(plan, b)
        qb, kb, vb = (torch.from_numpy(A.to64(t[rows])) for t in (wl.q, wl.k, wl.v))
        ref = F.scaled_dot_product_attention(
            qb.transpose(0, 1)[None], kb.transpose(0, 1)[None], vb.transpose(0, 1)[None],
            is_causal=True, enable_gqa=True)[0].transpose(0, 1).numpy()
        srows, o, _ = A.branch_suffix_attention(plan, wl.q, wl.k, wl.v, b)
        assert np.abs(o - ref[-len(srows):]).max() < 1e-12
