"""The library's prefix cache (sp_cache_*, sp_plan_build_cached) against the
oracle's radix cache model, on the host: over sequences of requests the two
must agree bit for bit on what every branch reuses, the remainders' segments
and rounds, the pool pages given to new shared segments, the cached levels
each segment reads, evictions and the cache's contents.  Then a float64
emulation of the descriptor over a persistent pool must reproduce, for every
row a warm plan computes, brute-force attention over the branch's whole
sequence (K/V of cached positions come from the pool that earlier plans
wrote)."""
import math

import numpy as np
import pytest

from oracle import cache as C

from test_plan_descriptor import PAGE, decode, emulate

SHAPE_ARGS = (4, 2, 64, 16, 64, 1000)  # Hq, Hkv, head_dim, page, hidden, vocab


def csr(seqs):
    off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
    toks = np.concatenate([np.asarray(s, np.int32) for s in seqs])
    return off, toks


def random_requests(rng, bases, n_steps):
    """Requests that reuse a few long states with varying question tails."""
    out = []
    for _ in range(n_steps):
        seqs, req = [], []
        for r in range(int(rng.integers(1, 3))):
            base = bases[int(rng.integers(0, len(bases)))][: int(rng.integers(10, 90))]
            for _ in range(int(rng.integers(1, 5))):
                tail = list(rng.integers(0, 5, int(rng.integers(0, 12))))
                s = base + tail
                seqs.append(s if s else [1])
                req.append(r)
        out.append((seqs, np.asarray(req, np.int32)))
    return out


def build_both(lib, shape, lcache, ocache, seqs, req):
    """(lib plan, oracle cached plan), or (None, None) when both find the pool
    full."""
    off, toks = csr(seqs)
    try:
        cp = C.plan_with_cache(ocache, req, off, toks)
    except MemoryError:
        cp = None
    try:
        plan = lib.sp_plan_build_cached(shape, lcache, req, off, toks, n_sms=16)
    except lib.SpError as e:
        assert e.status == 3 and cp is None  # SP_ERR_POOL_FULL on both sides
        return None, None
    assert cp is not None, "the library planned a request the oracle finds too large"
    return plan, cp


def compare_plan(plan, cp, ocache, seqs):
    st = plan.stats()
    ws = C.warm_stats(cp, csr(seqs)[0])
    for key in ("cache_hit_tokens", "computed_tokens", "reused_tokens", "node_tokens",
                "n_rounds", "logical_tokens"):
        assert st[key] == ws[key], key
    assert plan.rounds() == cp.plan.rounds
    seg = plan.segments()
    ref = cp.plan.segments
    assert len(seg["len"]) == len(ref)
    segs, pages, chain, _, _, _ = decode(plan.descriptor())
    for i, s in enumerate(ref):
        assert seg["len"][i] == s.length
        assert seg["parent"][i] == s.parent
        assert seg["node_start"][i] == s.node_start
        assert seg["shared"][i] == int(s.shared)
        assert seg["req"][i] == cp.groups[cp.seg_group[i]][0]
        want_round = cp.plan.claimed_round[i] if s.shared else cp.plan.branch_round[s.members[0]]
        assert seg["round"][i] == want_round
        if s.shared:  # the cache's pages, in the oracle's allocation order
            n = -(-s.length // PAGE)
            f = int(seg["first_page"][i])
            assert pages[f:f + n].tolist() == cp.seg_pages[i]
        # cached levels first (the group's match chain), then the new ancestors
        x = segs[i]
        levels = chain[x["chain_off"]:x["chain_off"] + x["chain_len"]]
        cached = [segs[c] for c in levels if segs[c]["shared"] == 2]
        mchain = cp.groups[cp.seg_group[i]][2]
        assert len(cached) == len(mchain)
        assert all(levels[j] >= len(ref) for j in range(len(mchain)))
        for lv, (node, vis) in zip(cached, mchain):
            assert lv["len"] == vis
            npg = -(-vis // PAGE)
            got = pages[lv["page_off"]:lv["page_off"] + npg].tolist()
            assert got == ocache.nodes[node].pages[:npg]
        anc = []
        p = s.parent
        while p >= 0:
            anc.append(p)
            p = ref[p].parent
        assert levels[len(mchain):].tolist() == anc[::-1]


def compare_cache(lcache, ocache):
    alive = [n for n in ocache.nodes[1:] if n.alive]
    assert lcache.stats() == {
        "segments": len(alive),
        "tokens": sum(len(n.tokens) for n in alive),
        "pages_used": len(ocache.free) - ocache.free_count(),
        "pages_free": ocache.free_count(),
        "evictions": ocache.evictions,
    }


@pytest.mark.parametrize("seed", range(16))
def test_cached_planner_matches_the_oracle(lib, seed):
    rng = np.random.default_rng(seed)
    n_pages = int(rng.integers(3, 16))  # small: evictions and full pools occur
    ocache = C.RadixCache(n_pages)
    lcache = lib.Cache(n_pages)
    shape = lib.make_shape(*SHAPE_ARGS)
    bases = [list(rng.integers(0, 5, int(rng.integers(20, 90)))) for _ in range(3)]
    for seqs, req in random_requests(rng, bases, 10):
        plan, cp = build_both(lib, shape, lcache, ocache, seqs, req)
        if plan is None:
            compare_cache(lcache, ocache)
            continue
        compare_plan(plan, cp, ocache, seqs)
        lib.sp_cache_commit(lcache, plan)
        C.commit(ocache, cp)
        lib.sp_cache_commit(lcache, plan)  # a second commit changes nothing
        plan.free()
        C.release(ocache, cp)
        compare_cache(lcache, ocache)


def test_pinned_nodes_survive_eviction(lib):
    """A plan that is not freed keeps the nodes it reads: a later plan that
    needs their pages finds the pool full instead of evicting them."""
    shape = lib.make_shape(*SHAPE_ARGS)
    lcache = lib.Cache(4)
    state = list(range(100, 148))  # 3 pages
    off, toks = csr([state + [1], state + [2]])
    p1 = lib.sp_plan_build_cached(shape, lcache, [0, 0], off, toks)
    lib.sp_cache_commit(lcache, p1)
    p1.free()
    assert lcache.stats()["pages_used"] == 3
    p2 = lib.sp_plan_build_cached(shape, lcache, [0, 0], *csr([state + [3], state + [4]]))
    assert p2.stats()["cache_hit_tokens"] == 2 * len(state)
    other = list(range(500, 532))  # 2 pages, 1 free, the cached state pinned by p2
    with pytest.raises(lib.SpError) as e:
        lib.sp_plan_build_cached(shape, lcache, [0, 0], *csr([other + [1], other + [2]]))
    assert e.value.status == 3
    assert lcache.stats()["evictions"] == 0
    p2.free()
    p3 = lib.sp_plan_build_cached(shape, lcache, [0, 0], *csr([other + [1], other + [2]]))
    assert lcache.stats()["evictions"] == 1
    p3.free()  # never committed: its pages go back to the pool
    assert lcache.stats() == {"segments": 0, "tokens": 0, "pages_used": 0, "pages_free": 4,
                              "evictions": 1}


def test_cache_argument_errors(lib):
    shape = lib.make_shape(*SHAPE_ARGS)
    with pytest.raises(lib.SpError):
        lib.Cache(0)
    a, b = lib.Cache(8), lib.Cache(8)
    plan = lib.sp_plan_build_cached(shape, a, [0], *csr([[1, 2, 3]]))
    with pytest.raises(lib.SpError):
        lib.sp_cache_commit(b, plan)  # a plan commits only to its own cache
    lib.sp_cache_commit(a, plan)
    assert a.stats()["segments"] == 0  # a single branch has no shared segment


# ---- descriptor emulation over a persistent pool ---------------------------

Hq, Hkv, D = 4, 2, 8


def row_vectors(seq, memo):
    """Per position: (q, k, v), a fixed function of the token prefix (as in a
    model, where a position's K/V depend only on the tokens up to it)."""
    out, h = [], 0
    for t in seq:
        h = (h * 1000003 + int(t) + 1) % (1 << 61)
        if h not in memo:
            r = np.random.default_rng(h)
            memo[h] = (r.standard_normal((Hq, D)), r.standard_normal((Hkv, D)),
                       r.standard_normal((Hkv, D)))
        out.append(memo[h])
    return out


def brute_row(vecs, pos):
    """Unshared causal attention of position pos over positions 0..pos."""
    G = Hq // Hkv
    q = vecs[pos][0]
    K = np.stack([vecs[j][1] for j in range(pos + 1)])
    V = np.stack([vecs[j][2] for j in range(pos + 1)])
    o, l = np.zeros((Hq, D)), np.zeros(Hq)
    for h in range(Hq):
        sc = K[:, h // G] @ q[h] / math.sqrt(D)
        m = sc.max()
        p = np.exp(sc - m)
        o[h] = p @ V[:, h // G] / p.sum()
        l[h] = m + math.log(p.sum())
    return o, l


@pytest.mark.parametrize("seed", range(6))
def test_warm_plans_over_a_persistent_pool(lib, seed):
    """Each plan of a request sequence, emulated over the pool that earlier
    plans filled, gives every computed row exactly the attention over its
    branch's full sequence; the pool starts as NaN, so a cached level whose
    pages were not written (or were reused after an eviction) shows up."""
    rng = np.random.default_rng(100 + seed)
    n_pages = int(rng.integers(8, 24))
    lcache = lib.Cache(n_pages)
    ocache = C.RadixCache(n_pages)
    shape = lib.make_shape(Hq, Hkv, 64, 16, 64, 1000)
    pool = np.full((n_pages, 2, Hkv, PAGE, D), np.nan)
    memo = {}
    bases = [list(rng.integers(0, 4, int(rng.integers(30, 140)))) for _ in range(2)]
    schedules = ("rounds", "all", "tree", "tree_rounds")
    n_warm = 0
    for step, (seqs, req) in enumerate(random_requests(rng, bases, 6)):
        plan, cp = build_both(lib, shape, lcache, ocache, seqs, req)
        if plan is None:
            continue
        n_warm += any(cp.reused)
        vecs = [row_vectors(s, memo) for s in seqs]
        T = plan.stats()["node_tokens"]
        q, k, v = np.zeros((T, Hq, D)), np.zeros((T, Hkv, D)), np.zeros((T, Hkv, D))
        want_o, want_l = np.zeros((T, Hq, D)), np.zeros((T, Hq))
        for s in cp.plan.segments:
            b = s.members[0]
            for t in range(s.length):
                pos = cp.reused[b] + s.start + t
                q[s.node_start + t], k[s.node_start + t], v[s.node_start + t] = vecs[b][pos]
                want_o[s.node_start + t], want_l[s.node_start + t] = brute_row(vecs[b], pos)
        after = None
        for schedule in schedules[step % 2::2]:
            trial = pool.copy()
            out, lse, _ = emulate(plan, q, k, v, Hq, Hkv, D, schedule, pool=trial)
            assert np.abs(out - want_o).max() < 1e-10
            assert np.abs(lse - want_l).max() < 1e-10
            after = trial
        pool = after
        lib.sp_cache_commit(lcache, plan)
        C.commit(ocache, cp)
        plan.free()
        C.release(ocache, cp)
    assert n_warm > 0


@pytest.mark.parametrize("seed", range(4))
def test_row_sources(lib, seed):
    """Every node-token row names a (branch, position) holding the row's token;
    with a cache the positions skip exactly the reused tokens."""
    rng = np.random.default_rng(200 + seed)
    n_pages = 64
    lcache = lib.Cache(n_pages)
    ocache = C.RadixCache(n_pages)
    shape = lib.make_shape(*SHAPE_ARGS)
    bases = [list(rng.integers(0, 5, int(rng.integers(20, 90)))) for _ in range(3)]
    for seqs, req in random_requests(rng, bases, 6):
        plan, cp = build_both(lib, shape, lcache, ocache, seqs, req)
        b, pos = plan.row_sources()
        T = plan.stats()["node_tokens"]
        assert len(b) == T
        want = np.zeros(T, np.int64)
        for s in cp.plan.segments:
            m = s.members[0]
            want[s.node_start:s.node_start + s.length] = \
                seqs[m][cp.reused[m] + s.start:cp.reused[m] + s.end]
        assert [seqs[x][p] for x, p in zip(b, pos)] == want.tolist()
        for x, p in zip(b, pos):
            assert p >= cp.reused[x]
        lib.sp_cache_commit(lcache, plan)
        C.commit(ocache, cp)
        plan.free()
        C.release(ocache, cp)
    # without a cache: positions of the full sequences
    seqs = [[1, 2, 3, 4], [1, 2, 9], [5]]
    plan = lib.sp_plan_build(shape, [0, 0, 1], *csr(seqs), 100)
    b, pos = plan.row_sources()
    assert [seqs[x][p] for x, p in zip(b, pos)] == [1, 2, 3, 4, 9, 5]
