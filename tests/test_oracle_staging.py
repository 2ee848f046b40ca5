"""Pins for the staging / trie oracle: the page's printed example and
brute-force invariants on random tries."""
import json
import os

import numpy as np
import pytest

from oracle import staging as S
from prefill_only_shared_gb300.workloads import make_workload, small_case

from conftest import GOLDEN


def csr(seqs):
    off = np.zeros(len(seqs) + 1, dtype=np.int64)
    off[1:] = np.cumsum([len(s) for s in seqs])
    toks = np.concatenate([np.asarray(s, dtype=np.int32) for s in seqs]) if seqs else np.zeros(0, np.int32)
    return off, toks


def golden_staging():
    g = json.load(open(os.path.join(GOLDEN, "staging_example.json")))
    seqs = [sum((g["segments"][s] for s in path), []) for path in g["branch_paths"]]
    return g, seqs


def test_printed_example_rounds():
    g, seqs = golden_staging()
    off, toks = csr(seqs)
    plan = S.build_plan(np.zeros(len(seqs), np.int32), off, toks)
    names = g["branch_names"]
    got = [[names[b] for b in r] for r in plan.rounds]
    assert got == g["printed_rounds"]
    # the shared segments first computed in each round
    seg_name = {}
    for name, toks_ in g["segments"].items():
        for sid, s in enumerate(plan.segments):
            b = s.members[0]
            if list(seqs[b][s.start:s.end]) == toks_ and s.shared:
                seg_name[sid] = name
    new = [[] for _ in plan.rounds]
    for sid, r in sorted(plan.claimed_round.items()):
        new[r].append(seg_name[sid])
    assert new == g["printed_new_shared_per_round"]
    # no extra warm-up: every branch scored exactly once, no recomputation
    assert sorted(sum(plan.rounds, [])) == list(range(6))
    assert not any(plan.recompute)


def random_request(rng, n, alphabet=3, max_len=7):
    seqs = []
    for i in range(n):
        r = rng.random()
        if seqs and r < 0.5:
            base = seqs[rng.integers(len(seqs))]
            cut = int(rng.integers(0, len(base) + 1))
            tail = list(rng.integers(0, alphabet, int(rng.integers(0, 4))))
            s = list(base[:cut]) + tail
        elif seqs and r < 0.6:
            s = list(seqs[rng.integers(len(seqs))])  # duplicate branch
        else:
            s = list(rng.integers(0, alphabet, int(rng.integers(1, max_len))))
        if not s:
            s = [int(rng.integers(alphabet))]
        seqs.append(s)
    return seqs


def random_case(seed):
    rng = np.random.default_rng(seed)
    n_req = int(rng.integers(1, 4))
    seqs, req = [], []
    for r in range(n_req):
        ss = random_request(rng, int(rng.integers(1, 8)))
        seqs += ss
        req += [r] * len(ss)
    # interleave requests to test grouping by request id
    perm = rng.permutation(len(seqs)) if rng.random() < 0.5 else np.arange(len(seqs))
    seqs = [seqs[i] for i in perm]
    req = np.array([req[i] for i in perm], dtype=np.int32)
    return req, seqs


@pytest.mark.parametrize("seed", range(60))
def test_random_tries_brute_force(seed):
    req, seqs = random_case(seed)
    off, toks = csr(seqs)
    plan = S.build_plan(req, off, toks)
    N = len(seqs)
    segs = plan.segments
    pos_seg = []
    for b in range(N):
        # a path covers exactly the branch's tokens, in order
        p = plan.paths[b]
        assert segs[p[0]].start == 0 and segs[p[-1]].end == len(seqs[b])
        for a, c in zip(p[:-1], p[1:]):
            assert segs[a].end == segs[c].start
            assert segs[c].parent == a
            assert set(segs[c].members) < set(segs[a].members)  # strictly shrinks
        m = {}
        for sid in p:
            for i in range(segs[sid].start, segs[sid].end):
                m[i] = sid
        pos_seg.append(m)
        for sid in p:
            assert b in segs[sid].members
    # two branches share the segment at position i iff same request and equal (i+1)-prefix
    for b in range(N):
        for b2 in range(N):
            for i in range(min(len(seqs[b]), len(seqs[b2]))):
                same = req[b] == req[b2] and seqs[b][:i + 1] == seqs[b2][:i + 1]
                assert (pos_seg[b][i] == pos_seg[b2][i]) == same
    # node-token layout: contiguous rows, depth-first pre-order
    row = 0
    for s in segs:
        assert s.node_start == row
        row += s.length
    subtree_end = {}
    for i in reversed(range(len(segs))):
        e = segs[i].node_start + segs[i].length
        for j in range(len(segs)):
            if segs[j].parent == i:
                e = max(e, subtree_end[j])
        subtree_end[i] = e
    for i, s in enumerate(segs):
        kids = [j for j in range(len(segs)) if segs[j].parent == i]
        nxt = s.node_start + s.length
        for j in sorted(kids, key=lambda j: segs[j].members[0]):
            assert segs[j].node_start == nxt
            nxt = subtree_end[j]
    # staging invariants
    flat = sum(plan.rounds, [])
    assert sorted(flat) == list(range(N))
    for r in plan.rounds:
        assert r == sorted(r)
    by_req = {}
    for b in range(N):
        by_req.setdefault(int(req[b]), []).append(b)
    for members in by_req.values():
        assert max(plan.branch_round[b] for b in members) < len(members)
        # the first unscored branch always joins: round 0 holds the request's first branch
        assert plan.branch_round[members[0]] == 0
    for sid, s in enumerate(segs):
        if s.shared:
            # built exactly once, in the round of a member, no later than any member
            r = plan.claimed_round[sid]
            assert r == min(plan.branch_round[b] for b in s.members)
    for b in range(N):
        for sid in plan.paths[b]:
            if segs[sid].shared:
                assert plan.claimed_round[sid] <= plan.branch_round[b]
    # no two branches of one round build the same shared segment
    for rnd in range(len(plan.rounds)):
        builders = {}
        for b in plan.rounds[rnd]:
            for sid in plan.paths[b]:
                if segs[sid].shared and plan.claimed_round[sid] == rnd:
                    builders.setdefault(sid, set()).add(b)
        # greedy rule: exactly one claimer; others in the round never need it uncached
        for sid, bs in builders.items():
            assert len(bs) >= 1
    # a branch recomputes its last row only when its end segment was cached earlier
    for b in range(N):
        last = plan.paths[b][-1]
        expect = segs[last].shared and plan.claimed_round[last] < plan.branch_round[b]
        assert plan.recompute[b] == expect


def test_prefix_and_duplicate_branches():
    seqs = [[1, 2, 3], [1, 2, 3, 4, 5], [1, 2, 3], [1, 2, 6]]
    off, toks = csr(seqs)
    plan = S.build_plan(np.zeros(4, np.int32), off, toks)
    assert plan.rounds == [[0], [1, 2, 3]]
    assert plan.recompute == [False, False, True, False]
    st = S.plan_stats(plan)
    assert st["logical_tokens"] == 3 + 5 + 3 + 3
    assert st["node_tokens"] == 3 + 2 + 1
    assert st["computed_tokens"] == 7


def expected_config_rounds(wl):
    N = wl.n_branches
    if wl.name == "tree2":
        return [[0], [1, 2, 3], [4, 5]]
    if wl.name == "batch64":
        firsts = [b for b in range(N) if b % 12 == 0]
        return [firsts, [b for b in range(N) if b % 12 != 0]]
    return [[0], list(range(1, N))]


@pytest.mark.parametrize("name", ["tiny", "yesno", "choice64", "tree2", "batch64"])
def test_config_layout_and_rounds(name):
    wl = make_workload(name, tokens_only=True)
    plan = S.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    assert plan.rounds == expected_config_rounds(wl)
    # the generator's segment tree is the trie's node-token layout
    assert len(plan.segments) == len(wl.seg_len)
    for i, s in enumerate(plan.segments):
        assert s.node_start == wl.seg_start[i] and s.length == wl.seg_len[i]
        assert s.parent == wl.seg_parent[i]
    assert [p[-1] for p in plan.paths] == list(wl.branch_leaf)


def test_small_case_layout_matches_generator():
    wl = small_case((9, [(5, [(3, []), (2, [])]), (4, [])]))
    plan = S.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    for i, s in enumerate(plan.segments):
        assert s.node_start == wl.seg_start[i] and s.length == wl.seg_len[i]
