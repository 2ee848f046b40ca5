"""GPU parity of the prefix cache across calls: a sequence of calls through
one classifier whose shared segments persist in the KV pool.  Every row a warm
plan computes must match float64 attention over its branch's whole sequence,
with the K/V of cached positions read from pool pages that earlier calls
wrote (LLM2Jev page, section on reusing the radix cache; openjev-sglang
article, section on the repeated state)."""
import math

import numpy as np
import pytest
import torch

from oracle import cache as C

from gpu_helpers import TOL_LSE, TOL_OUT

pytestmark = pytest.mark.gpu


def csr(seqs):
    off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
    toks = np.concatenate([np.asarray(s, np.int32) for s in seqs])
    return off, toks


class PrefixVectors:
    """q / k / v of a position as a fixed function of its token prefix (bf16
    values, as a model's K/V depend only on the tokens up to the position)."""

    def __init__(self, Hq, Hkv, d):
        self.shapes = ((Hq, d), (Hkv, d), (Hkv, d))
        self.memo = {}

    def __call__(self, seq):
        out, h = [], 0
        for t in seq:
            h = (h * 1000003 + int(t) + 1) % (1 << 61)
            if h not in self.memo:
                r = np.random.default_rng(h)
                self.memo[h] = tuple(
                    torch.from_numpy(r.standard_normal(s)).bfloat16() for s in self.shapes)
            out.append(self.memo[h])
        return out


def causal_attention(vecs, G):
    """float64 attention of every position of one branch over its prefix."""
    Q = torch.stack([x[0] for x in vecs]).double()
    K = torch.stack([x[1] for x in vecs]).double().repeat_interleave(G, dim=1)
    V = torch.stack([x[2] for x in vecs]).double().repeat_interleave(G, dim=1)
    L, _, d = Q.shape
    sc = torch.einsum("qhd,khd->hqk", Q, K) / math.sqrt(d)
    sc = sc.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), -math.inf)
    lse = torch.logsumexp(sc, dim=-1)
    out = torch.einsum("hqk,khd->qhd", torch.exp(sc - lse[..., None]), V)
    return out.numpy(), lse.T.numpy()


def request_sequence(rng):
    """(seqs, req) per call: cold state, repeated state with new questions
    (two of them share an instruction), a match ending inside the cached
    state, a call mixing a cold and a warm request, a hot re-run, and a new
    state that needs an eviction."""
    A = list(rng.integers(0, 1000, 300))
    B = list(rng.integers(0, 1000, 200))
    Cst = list(rng.integers(0, 1000, 230))

    def qs(n, lo=12, hi=40):
        return [list(rng.integers(1000, 2000, int(rng.integers(lo, hi)))) for _ in range(n)]

    instr = list(rng.integers(2000, 3000, 37))
    warm_qs = [instr + x for x in qs(2)] + qs(2)
    calls = [
        ([A + x for x in qs(4)], [0] * 4),
        ([A + x for x in warm_qs], [0] * 4),
        ([A[:150] + x for x in qs(3)], [0] * 3),
        ([B + x for x in qs(3)] + [A + x for x in qs(2)], [0] * 3 + [1] * 2),
        ([A + x for x in warm_qs], [0] * 4),
        ([A + instr], [0]),  # ends inside a cached segment's remainder
        ([Cst + x for x in qs(2)], [0] * 2),
    ]
    return [(s, np.asarray(r, np.int32)) for s, r in calls]


@pytest.mark.parametrize("schedule", ["rounds", "all", "tree"])
@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 64), (32, 4, 128)])
def test_warm_calls_through_the_cache(cuda_dev, lib, schedule, Hq, Hkv, d):
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    rng = np.random.default_rng(Hq + d)
    n_pages = 48  # A, B and the instruction fit; the last state evicts
    clf = SharedPrefixClassifier(Hq, Hkv, d, 64, 100, device=cuda_dev, prefix_cache_pages=n_pages)
    ocache = C.RadixCache(n_pages)
    vec = PrefixVectors(Hq, Hkv, d)
    G = Hq // Hkv
    hits = []
    for seqs, req in request_sequence(rng):
        off, toks = csr(seqs)
        ocp = C.plan_with_cache(ocache, req, off, toks)
        plan = clf.plan(req, off, toks)
        st = plan.stats()
        assert st["cache_hit_tokens"] == sum(ocp.reused)
        assert plan.rounds() == ocp.plan.rounds
        hits.append(st["cache_hit_tokens"])
        T = st["node_tokens"]
        full = [vec(s) for s in seqs]
        ref = [causal_attention(f, G) for f in full]
        q = torch.empty(T, Hq, d, dtype=torch.bfloat16)
        k = torch.empty(T, Hkv, d, dtype=torch.bfloat16)
        v = torch.empty(T, Hkv, d, dtype=torch.bfloat16)
        want_o = np.zeros((T, Hq, d))
        want_l = np.zeros((T, Hq))
        for s in ocp.plan.segments:
            b = s.members[0]
            for t in range(s.length):
                row, pos = s.node_start + t, ocp.reused[b] + s.start + t
                q[row], k[row], v[row] = full[b][pos]
                want_o[row], want_l[row] = ref[b][0][pos], ref[b][1][pos]
        out, lse = clf.attention(plan, q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev),
                                 schedule=schedule)
        torch.cuda.synchronize()
        sp.sp_check_device_error()
        assert np.abs(out.float().cpu().numpy() - want_o).max() <= TOL_OUT
        assert np.abs(lse.cpu().numpy() - want_l).max() <= TOL_LSE
        C.commit(ocache, ocp)
        C.release(ocache, ocp)
        assert clf.cache.stats()["evictions"] == ocache.evictions
        del plan
    # cold, full state, part of it, the warm request of the mixed call, hot
    assert hits[0] == 0 and hits[1] == 4 * 300 and hits[2] == 3 * 150
    assert hits[3] == 2 * 300 and hits[4] > hits[1] and ocache.evictions > 0
