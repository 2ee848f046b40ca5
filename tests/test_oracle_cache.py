"""Pins of the prefix cache model (oracle/cache.py): the cold case reduces to
the cold staging, closed-form accounting for a repeated state and for a hot
re-run of the LLM2Jev page's printed example, LRU eviction order, and
brute-force invariants over random request sequences."""
import json
import os

import numpy as np
import pytest

from oracle import cache as C
from oracle import staging as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def csr(seqs):
    off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
    toks = np.concatenate([np.asarray(s, np.int64) for s in seqs])
    return off, toks


def run(cache, seqs, req=None, commit=True):
    req = np.zeros(len(seqs), np.int32) if req is None else np.asarray(req, np.int32)
    off, toks = csr(seqs)
    cp = C.plan_with_cache(cache, req, off, toks)
    if commit:
        C.commit(cache, cp)
    C.release(cache, cp)
    return cp, off


def path_tokens(cache, n):
    out = []
    while n > 0:
        out = list(cache.nodes[n].tokens) + out
        n = cache.nodes[n].parent
    return out


def test_cold_cache_is_the_cold_plan():
    rng = np.random.default_rng(0)
    seqs = [list(rng.integers(0, 9, 40)) for _ in range(3)]
    seqs += [seqs[0][:25] + [7, 7, 7], seqs[1] + [1, 2]]
    cache = C.RadixCache(1000)
    off, toks = csr(seqs)
    cold = S.build_plan(np.zeros(len(seqs), np.int32), off, toks)
    cp, _ = run(cache, seqs, commit=False)
    assert cp.reused == [0] * len(seqs)
    assert cp.plan.rounds == cold.rounds
    assert [(s.start, s.end, s.members) for s in cp.plan.segments] == \
        [(s.start, s.end, s.members) for s in cold.segments]


def test_repeated_state_reads_only_the_questions():
    """openjev article, repeated state: the second request with the same state
    and new questions computes only its questions."""
    rng = np.random.default_rng(1)
    state = list(rng.integers(100, 200, 300))
    q1 = [[i] + list(rng.integers(0, 50, 20 + i)) for i in range(4)]
    q2 = [[10 + i] + list(rng.integers(0, 50, 15 + 2 * i)) for i in range(4)]
    cache = C.RadixCache(1000)
    run(cache, [state + q for q in q1])
    assert [path_tokens(cache, n) for n in range(1, len(cache.nodes))] == [state]
    cp, off = run(cache, [state + q for q in q2])
    assert cp.reused == [len(state)] * 4
    st = C.warm_stats(cp, off)
    assert st["computed_tokens"] == sum(len(q) for q in q2)
    assert st["cache_hit_tokens"] == 4 * len(state)
    assert cp.plan.rounds == [[0, 1, 2, 3]]


def test_hot_rerun_of_the_printed_example():
    """LLM2Jev page: the cold request takes the three printed rounds; the same
    request again is hot -- every candidate reuses the state and its
    question's instructions (the shared segments the cold run cached), only
    its own criteria are computed, and all candidates go in one round."""
    g = json.load(open(os.path.join(GOLDEN, "staging_example.json")))
    seqs = [sum((g["segments"][name] for name in path), []) for path in g["branch_paths"]]
    names = g["branch_names"]
    printed = [[names.index(x) for x in rnd] for rnd in g["printed_rounds"]]
    cache = C.RadixCache(4000)
    cold, _ = run(cache, seqs)
    assert cold.plan.rounds == printed
    hot, off = run(cache, seqs)
    shared = [len(g["segments"][p[0]]) + len(g["segments"][p[1]]) for p in g["branch_paths"]]
    assert hot.reused == shared
    assert hot.plan.rounds == [list(range(len(seqs)))]
    own = sum(len(g["segments"][p[2]]) for p in g["branch_paths"])
    assert C.warm_stats(hot, off)["computed_tokens"] == own


def test_lru_eviction_order():
    cache = C.RadixCache(8)  # 8 pages of 16 tokens
    a = list(range(1000, 1032))     # 32 tokens -> 2 pages
    b = list(range(2000, 2048))     # 48 tokens -> 3 pages
    c = list(range(3000, 3032))
    for st in (a, b):
        run(cache, [st + [1], st + [2]])
    assert cache.free_count() == 3
    run(cache, [a + [5], a + [6]])  # a used again: b is now the least recent
    run(cache, [c + [1], c + [2]])  # needs 2 pages, 3 free: no eviction
    assert cache.evictions == 0
    d = list(range(4000, 4048))     # 3 pages, 1 free: evict b (oldest), 3 free
    run(cache, [d + [1], d + [2]])
    assert cache.evictions == 1
    alive = [path_tokens(cache, n) for n in range(1, len(cache.nodes)) if cache.nodes[n].alive]
    assert b not in alive and a in alive and c in alive and d in alive


def test_pool_full_when_nothing_can_be_evicted():
    cache = C.RadixCache(2)
    st = list(range(500, 560))  # 60 tokens -> 4 pages
    with pytest.raises(MemoryError):
        run(cache, [st + [1], st + [2]])
    assert cache.free_count() == 2


@pytest.mark.parametrize("seed", range(12))
def test_random_request_sequences(seed):
    rng = np.random.default_rng(seed)
    cache = C.RadixCache(int(rng.integers(20, 60)))
    bases = [list(rng.integers(0, 5, int(rng.integers(20, 90)))) for _ in range(3)]
    for step in range(8):
        seqs, req = [], []
        for r in range(int(rng.integers(1, 3))):
            base = bases[int(rng.integers(0, 3))][: int(rng.integers(10, 90))]
            for _ in range(int(rng.integers(1, 5))):
                tail = list(rng.integers(0, 5, int(rng.integers(0, 12))))
                s = base + tail
                if not s:
                    s = [1]
                seqs.append(s)
                req.append(r)
        alive_paths = [path_tokens(cache, n) for n in range(1, len(cache.nodes))
                       if cache.nodes[n].alive]
        try:
            cp, off = run(cache, seqs, req)
        except MemoryError:
            continue
        for b, s in enumerate(seqs):
            # reused = longest common prefix with any cached path, capped
            best = max([0] + [S._lcp(np.asarray(s), np.asarray(p)) for p in alive_paths])
            assert cp.reused[b] == min(best, len(s) - 1)
            # the chain's visible tokens are the branch's first tokens
            got = []
            for node, vis in cp.chains[b]:
                got += list(cache.nodes[node].tokens[:vis])
            assert got == s[:cp.reused[b]]
        # pages: alive nodes own disjoint, allocated pages
        owned = [p for n in cache.nodes[1:] if n.alive for p in n.pages]
        assert len(owned) == len(set(owned))
        assert all(not cache.free[p] for p in owned)
        assert cache.free_count() == len(cache.free) - len(owned)
        assert all(n.pins == 0 for n in cache.nodes)
        # an alive node's children start with distinct tokens
        for n in cache.nodes:
            if n.alive:
                firsts = [cache.nodes[c].tokens[0] for c in n.children]
                assert len(firsts) == len(set(firsts))
