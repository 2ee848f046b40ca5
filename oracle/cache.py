"""Prefix persistence across calls: a radix cache of computed shared segments.

Test infrastructure: only tests, the smoke check and the benchmark's CPU legs
use this module.

Source: LLM2Jev "shared prefix" page, sections on reusing SGLang's radix cache
(the cache keeps token prefixes whose KV has been computed; a later candidate
continues from the first uncached position; the engine may keep prefixes
across requests and evicts them when memory is short; a hot request finds its
prefix already cached) and on outputs (the final scoring position of every
candidate is always computed); openjev-sglang article, section on the repeated
state (consecutive requests that repeat a state and change only the questions
read only their own questions; several states can be kept and used in turn).

Readings taken where the pages are silent (each listed in the design notes):

* What is cached: the shared segments (inner trie nodes) that a plan computed,
  inserted after the plan ran, with the pool pages holding their K/V.  Leaves
  (a branch's own suffix) are not cached: nothing later reads them.
* Match: a branch walks the cache from the root, following the child whose
  first token is its next token; whole nodes are reused, and the walk may end
  inside a node (its first k tokens are reused).  The reused length is capped
  at the branch length minus one, so the last position is always computed.
* The uncached remainders are planned and staged exactly like a cold request,
  in groups of the branches of one request that end their match at the same
  place (group order: request id, then smallest branch index).
* Insertion: a new shared segment goes under the node where its group's match
  ended (or under its new parent segment), only when that match ended on a node
  boundary and no child of that node starts with the same token.
* Pages: a new shared segment takes ceil(len / 16) pages, the lowest run of
  free consecutive pages, else the lowest free pages.  When the free pages do
  not cover the plan, cache leaves that the plan does not use are evicted,
  least recently used first (ties: older node first).  Every node a plan uses
  is marked used at build time; inserted nodes at commit time.

Parity: pinned by the page's printed cold-request rounds (a warm request whose
state is cached re-stages only the remainders), closed-form token accounting,
and brute-force invariants on random request sequences (tests).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from oracle import staging as S

PAGE = 16


@dataclass
class Node:
    tokens: tuple
    pages: list
    parent: int
    children: list = field(default_factory=list)
    last_used: int = 0
    pins: int = 0
    alive: bool = True


class RadixCache:
    def __init__(self, n_pages: int):
        self.nodes = [Node(tokens=(), pages=[], parent=-1)]
        self.free = [True] * n_pages
        self.clock = 0
        self.evictions = 0

    # -- lookup ---------------------------------------------------------------
    def match(self, seq):
        """[(node, visible length)] from the root and the matched length."""
        cur, pos, chain = 0, 0, []
        while pos < len(seq):
            nxt = None
            for c in self.nodes[cur].children:
                if self.nodes[c].tokens[0] == seq[pos]:
                    nxt = c
                    break
            if nxt is None:
                break
            toks = self.nodes[nxt].tokens
            m = 0
            while m < len(toks) and pos + m < len(seq) and toks[m] == seq[pos + m]:
                m += 1
            chain.append((nxt, m))
            pos += m
            if m < len(toks):
                break
            cur = nxt
        return chain, pos

    # -- pages ----------------------------------------------------------------
    def free_count(self):
        return sum(self.free)

    def evict_one(self):
        cand = [i for i, n in enumerate(self.nodes)
                if i > 0 and n.alive and n.pins == 0
                and not any(self.nodes[c].alive for c in n.children)]
        if not cand:
            return False
        i = min(cand, key=lambda j: (self.nodes[j].last_used, j))
        n = self.nodes[i]
        n.alive = False
        for p in n.pages:
            self.free[p] = True
        self.nodes[n.parent].children.remove(i)
        self.evictions += 1
        return True

    def alloc(self, n):
        run = 0
        for p in range(len(self.free)):
            run = run + 1 if self.free[p] else 0
            if run == n:
                pages = list(range(p - n + 1, p + 1))
                break
        else:
            pages = [p for p in range(len(self.free)) if self.free[p]][:n]
        for p in pages:
            self.free[p] = False
        return pages


@dataclass
class CachedPlan:
    plan: S.Plan          # the remainders' plan (segments, rounds, layout)
    groups: list          # per group: (request, [branches], chain)
    group_of_branch: list
    reused: list          # per branch: tokens taken from the cache
    chains: list          # per branch: [(node, visible length)]
    seg_group: list       # per segment of the plan: its group
    seg_tokens: list      # per segment: its token tuple
    seg_pages: dict       # shared segment -> its pages
    pinned: list
    inserted: dict = field(default_factory=dict)  # shared segment -> cache node


def plan_with_cache(cache: RadixCache, req_of_branch, tok_offsets, tokens) -> CachedPlan:
    N = len(req_of_branch)
    seqs = [tuple(int(t) for t in tokens[tok_offsets[b]:tok_offsets[b + 1]]) for b in range(N)]
    chains, reused = [], []
    for b in range(N):
        chain, m = cache.match(seqs[b])
        if m > len(seqs[b]) - 1:  # the last position is always computed
            node, vis = chain[-1]
            chain = chain[:-1] + ([(node, vis - 1)] if vis > 1 else [])
            m -= 1
        chains.append(chain)
        reused.append(m)
    # groups: branches of one request whose match ends at the same place
    keys = {}
    for b in range(N):
        end = chains[b][-1] if chains[b] else (0, 0)
        keys.setdefault((int(req_of_branch[b]), end), []).append(b)
    ordered = sorted(keys.items(), key=lambda kv: (kv[0][0], kv[1][0]))
    group_of_branch = [0] * N
    groups = []
    for g, ((r, _end), members) in enumerate(ordered):
        groups.append((r, members, chains[members[0]]))
        for b in members:
            group_of_branch[b] = g
    rem = [seqs[b][reused[b]:] for b in range(N)]
    off = np.concatenate([[0], np.cumsum([len(x) for x in rem])]).astype(np.int64)
    toks = np.concatenate([np.asarray(x, np.int64) for x in rem])
    plan = S.build_plan(group_of_branch, off, toks)
    seg_group, seg_tokens = [], []
    for s in plan.segments:
        g = s.req
        b = s.members[0]
        seg_group.append(g)
        seg_tokens.append(rem[b][s.start:s.end])
    # pin the nodes this plan reads, mark them used
    pinned = sorted({node for ch in chains for node, _ in ch})
    for node in pinned:
        cache.nodes[node].pins += 1
        cache.nodes[node].last_used = cache.clock
    cache.clock += 1
    # pages for the new shared segments, in node-token order
    need = sum(-(-s.length // PAGE) for s in plan.segments if s.shared)
    while cache.free_count() < need:
        if not cache.evict_one():
            for node in pinned:
                cache.nodes[node].pins -= 1
            raise MemoryError("pool full")
    seg_pages = {}
    for i, s in enumerate(plan.segments):
        if s.shared:
            seg_pages[i] = cache.alloc(-(-s.length // PAGE))
    return CachedPlan(plan=plan, groups=groups, group_of_branch=group_of_branch, reused=reused,
                      chains=chains, seg_group=seg_group, seg_tokens=seg_tokens,
                      seg_pages=seg_pages, pinned=pinned)


def commit(cache: RadixCache, cp: CachedPlan):
    """Insert the plan's eligible shared segments (after its calls ran)."""
    stamp = cache.clock
    cache.clock += 1
    for i, s in enumerate(cp.plan.segments):
        if not s.shared:
            continue
        if s.parent >= 0:
            parent = cp.inserted.get(s.parent)
            if parent is None:
                continue
        else:
            chain = cp.groups[cp.seg_group[i]][2]
            if chain and chain[-1][1] < len(cache.nodes[chain[-1][0]].tokens):
                continue  # the match ended inside a node
            parent = chain[-1][0] if chain else 0
        toks = cp.seg_tokens[i]
        if any(cache.nodes[c].tokens[0] == toks[0] for c in cache.nodes[parent].children):
            continue
        cache.nodes.append(Node(tokens=tuple(toks), pages=cp.seg_pages[i], parent=parent,
                                last_used=stamp))
        nid = len(cache.nodes) - 1
        cache.nodes[parent].children.append(nid)
        cp.inserted[i] = nid


def release(cache: RadixCache, cp: CachedPlan):
    """Unpin the plan's nodes and free the pages of segments not inserted."""
    for node in cp.pinned:
        cache.nodes[node].pins -= 1
    for i, pages in cp.seg_pages.items():
        if i not in cp.inserted:
            for p in pages:
                cache.free[p] = True


def warm_stats(cp: CachedPlan, tok_offsets) -> dict:
    st = S.plan_stats(cp.plan)
    logical = int(tok_offsets[-1])
    return {
        "logical_tokens": logical,
        "computed_tokens": st["computed_tokens"],
        "reused_tokens": logical - st["computed_tokens"],
        "cache_hit_tokens": int(sum(cp.reused)),
        "node_tokens": st["node_tokens"],
        "n_rounds": st["n_rounds"],
    }
