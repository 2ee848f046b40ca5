"""Seeded synthetic inputs for the shared-prefix classifier path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (through the binding) and the CPU
oracle consume the tensors it returns, so the two sides always see the same
bf16 values.

Workload shapes follow the five synthetic configurations that stand in for the
pages' request mixes (a customer ticket with a few questions, a long
conversation with yes/no questions, a 64-way choice, a state -> instructions ->
criteria tree, and a batch of independent requests):

========  ===================================================================
tiny      Hq 8, Hkv 2, d 64; prefix 256 + 4 branches x 32; h [4x512]; W [4096x512]
yesno     Hq 32, Hkv 4, d 128; prefix 2000 + 5 x 48; H 2048; V 151936; 2 labels
choice64  prefix 1200 + 64 x 40; one shared set of 64 label ids
tree2     state 2000 -> 2 instructions x 200 -> 3 criteria x 30 each (6 branches)
batch64   64 requests, prefix U[3072, 5120], 12 branches x 64; 2..8 labels
========  ===================================================================

Recipe (fixed draw order, one ``torch.Generator`` seeded with ``seed``):

1. per-request prefix lengths (``batch64`` only), integer-uniform;
2. token ids, request by request, segment by segment in depth-first order:
   uniform over the vocabulary; the first token of every child segment is
   redrawn until it differs from the first tokens of its earlier siblings, so
   the token trie forks exactly at the segment boundaries;
3. q, k, v per segment in the same order, ``randn`` in fp32 rounded to bf16
   (round-to-nearest-even), ~N(0, 1);
4. final hidden states h [N, H] ~ N(0, 1) in bf16;
5. LM head W [V, H] ~ N(0, 0.02) in bf16;
6. label ids per branch: distinct ids drawn uniformly (duplicates redrawn);
   ``choice64`` draws one set of 64 ids shared by every branch; ``batch64``
   first draws the label count per branch from U{2..8}.

Token rows of q/k/v are stored in "node-token" order: requests in order, and
within a request the segments of its token trie in depth-first pre-order with
children ordered by the smallest branch index that passes through them.  For
the trees built here that is exactly the order in which the generator visits
the segments.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

CONFIG_NAMES = ("tiny", "yesno", "choice64", "tree2", "batch64")


@dataclass
class Shape:
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    hidden: int
    vocab: int


@dataclass
class Workload:
    name: str
    shape: Shape
    seed: int
    # branch token sequences (CSR)
    req_of_branch: np.ndarray  # int32 [N]
    tok_offsets: np.ndarray  # int64 [N+1]
    tokens: np.ndarray  # int32 [sum L]
    # the generator's own segment tree, in node-token order
    seg_req: np.ndarray  # int32 [n_seg]
    seg_parent: np.ndarray  # int32 [n_seg], -1 for a request root
    seg_start: np.ndarray  # int64 [n_seg], first node-token row
    seg_len: np.ndarray  # int32 [n_seg]
    branch_leaf: np.ndarray  # int32 [N], the segment holding the branch's last token
    # activations and weights (CPU, bf16)
    q: torch.Tensor  # [T, Hq, d]
    k: torch.Tensor  # [T, Hkv, d]
    v: torch.Tensor  # [T, Hkv, d]
    h: torch.Tensor  # [N, H]
    W: torch.Tensor  # [V, H]
    label_off: np.ndarray  # int32 [N+1]
    label_ids: np.ndarray  # int32 [sum k]
    meta: dict = field(default_factory=dict)

    @property
    def n_branches(self) -> int:
        return int(self.req_of_branch.shape[0])

    @property
    def node_tokens(self) -> int:
        return int(self.q.shape[0])

    def branch_tokens(self, b: int) -> np.ndarray:
        return self.tokens[self.tok_offsets[b]:self.tok_offsets[b + 1]]


# A request tree is (length, [children]); leaves are branches.
def _tree_yesno(prefix, n_branches, suffix):
    return (prefix, [(suffix, []) for _ in range(n_branches)])


def _config_trees(name, g):
    """Returns (shape, list of request trees, label spec)."""
    big = dict(n_q_heads=32, n_kv_heads=4, head_dim=128, page_size=16, hidden=2048, vocab=151936)
    if name == "tiny":
        shape = Shape(8, 2, 64, 16, 512, 4096)
        return shape, [_tree_yesno(256, 4, 32)], ("per_branch", 2)
    if name == "yesno":
        return Shape(**big), [_tree_yesno(2000, 5, 48)], ("per_branch", 2)
    if name == "choice64":
        return Shape(**big), [_tree_yesno(1200, 64, 40)], ("shared", 64)
    if name == "tree2":
        crit = [(30, []) for _ in range(3)]
        tree = (2000, [(200, list(crit)), (200, list(crit))])
        return Shape(**big), [tree], ("per_branch", 2)
    if name == "batch64":
        lens = torch.randint(3072, 5121, (64,), generator=g, dtype=torch.int64).tolist()
        return Shape(**big), [_tree_yesno(p, 12, 64) for p in lens], ("per_branch_range", (2, 8))
    raise ValueError(f"unknown workload {name!r}")


def _flatten(trees):
    """Depth-first segments: (req, parent, length, is_leaf) in node-token order."""
    segs = []

    def walk(req, node, parent):
        length, children = node
        idx = len(segs)
        segs.append([req, parent, length, len(children) == 0])
        for ch in children:
            walk(req, ch, idx)

    for r, t in enumerate(trees):
        walk(r, t, -1)
    return segs


def _draw_distinct(g, vocab, count):
    ids = []
    while len(ids) < count:
        x = int(torch.randint(vocab, (1,), generator=g).item())
        if x not in ids:
            ids.append(x)
    return ids


def make_workload(name: str, seed: int = 0, trees=None, shape: Shape | None = None,
                  label_spec=None, tokens_only: bool = False) -> Workload:
    """Builds one seeded workload.

    ``trees``/``shape``/``label_spec`` override the named configuration, which
    the tests use for small ragged cases (any tree of (length, children)).
    ``tokens_only`` stops after the token draws (same tokens, no tensors).
    """
    g = torch.Generator().manual_seed(seed)
    if trees is None:
        shape, trees, label_spec = _config_trees(name, g)
    assert shape is not None and label_spec is not None
    segs = _flatten(trees)
    n_seg = len(segs)
    V = shape.vocab

    # 2. tokens per segment, depth-first, sibling first tokens distinct
    seg_tokens = [None] * n_seg
    first_of_children = {}
    for i, (req, parent, length, _leaf) in enumerate(segs):
        if length <= 0:
            raise ValueError("segments must be non-empty")
        t = torch.randint(V, (length,), generator=g, dtype=torch.int64)
        key = (req, parent)
        used = first_of_children.setdefault(key, set())
        while int(t[0]) in used:
            t[0] = torch.randint(V, (1,), generator=g, dtype=torch.int64)[0]
        used.add(int(t[0]))
        seg_tokens[i] = t.to(torch.int32).numpy()

    seg_len = np.array([s[2] for s in segs], dtype=np.int32)
    seg_start = np.zeros(n_seg, dtype=np.int64)
    seg_start[1:] = np.cumsum(seg_len.astype(np.int64))[:-1]
    T = int(seg_len.astype(np.int64).sum())

    # branches = leaves in depth-first order; path = ancestors + leaf
    leaves = [i for i, s in enumerate(segs) if s[3]]
    paths = []
    for lf in leaves:
        p = []
        x = lf
        while x >= 0:
            p.append(x)
            x = segs[x][1]
        paths.append(p[::-1])
    N = len(leaves)
    req_of_branch = np.array([segs[lf][0] for lf in leaves], dtype=np.int32)
    blens = [int(sum(seg_len[s] for s in p)) for p in paths]
    tok_offsets = np.zeros(N + 1, dtype=np.int64)
    tok_offsets[1:] = np.cumsum(blens)
    tokens = np.concatenate([np.concatenate([seg_tokens[s] for s in p]) for p in paths]).astype(np.int32)

    if tokens_only:
        empty = torch.zeros(0)
        return Workload(
            name=name, shape=shape, seed=seed,
            req_of_branch=req_of_branch, tok_offsets=tok_offsets, tokens=tokens,
            seg_req=np.array([s[0] for s in segs], dtype=np.int32),
            seg_parent=np.array([s[1] for s in segs], dtype=np.int32),
            seg_start=seg_start, seg_len=seg_len,
            branch_leaf=np.array(leaves, dtype=np.int32),
            q=empty, k=empty, v=empty, h=empty, W=empty,
            label_off=np.zeros(N + 1, dtype=np.int32), label_ids=np.zeros(0, dtype=np.int32),
            meta={"trees": trees, "label_spec": label_spec, "tokens_only": True},
        )

    # 3. q, k, v per segment
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    q = torch.empty((T, Hq, d), dtype=torch.bfloat16)
    k = torch.empty((T, Hkv, d), dtype=torch.bfloat16)
    v = torch.empty((T, Hkv, d), dtype=torch.bfloat16)
    for i in range(n_seg):
        a, L = int(seg_start[i]), int(seg_len[i])
        q[a:a + L] = torch.randn((L, Hq, d), generator=g).to(torch.bfloat16)
        k[a:a + L] = torch.randn((L, Hkv, d), generator=g).to(torch.bfloat16)
        v[a:a + L] = torch.randn((L, Hkv, d), generator=g).to(torch.bfloat16)

    # 4./5. hidden states and LM head
    h = torch.randn((N, shape.hidden), generator=g).to(torch.bfloat16)
    W = (torch.randn((V, shape.hidden), generator=g) * 0.02).to(torch.bfloat16)

    # 6. labels
    kind, arg = label_spec
    label_lists = []
    if kind == "per_branch":
        for _ in range(N):
            label_lists.append(_draw_distinct(g, V, arg))
    elif kind == "shared":
        shared = _draw_distinct(g, V, arg)
        label_lists = [list(shared) for _ in range(N)]
    elif kind == "per_branch_range":
        lo, hi = arg
        for _ in range(N):
            cnt = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
            label_lists.append(_draw_distinct(g, V, cnt))
    elif kind == "explicit":
        label_lists = [list(x) for x in arg]
    else:
        raise ValueError(kind)
    label_off = np.zeros(N + 1, dtype=np.int32)
    label_off[1:] = np.cumsum([len(x) for x in label_lists])
    label_ids = np.array([i for x in label_lists for i in x], dtype=np.int32)

    return Workload(
        name=name, shape=shape, seed=seed,
        req_of_branch=req_of_branch, tok_offsets=tok_offsets, tokens=tokens,
        seg_req=np.array([s[0] for s in segs], dtype=np.int32),
        seg_parent=np.array([s[1] for s in segs], dtype=np.int32),
        seg_start=seg_start, seg_len=seg_len,
        branch_leaf=np.array(leaves, dtype=np.int32),
        q=q, k=k, v=v, h=h, W=W, label_off=label_off, label_ids=label_ids,
        meta={"trees": trees, "label_spec": label_spec},
    )


def small_case(trees, seed=0, n_q_heads=4, n_kv_heads=2, head_dim=64, hidden=128, vocab=512,
               labels=("per_branch", 2), page_size=16) -> Workload:
    """A small custom workload for ragged / edge-case tests.

    ``trees`` is one request tree ``(length, [children])`` or a list of them."""
    if isinstance(trees, tuple):
        trees = [trees]
    shape = Shape(n_q_heads, n_kv_heads, head_dim, page_size, hidden, vocab)
    return make_workload("custom", seed=seed, trees=trees, shape=shape, label_spec=labels)


@dataclass
class OptionWorkload:
    """Multi-token options: question q owns options q_off[q] .. q_off[q+1]-1,
    option o owns rows opt_off[o] .. opt_off[o+1]-1, one row per option token:
    the hidden state at the position before that token (h_rows, bf16) and the
    token itself (tokens).  prior: a per-option log-probability for
    calibration (fp32), drawn here as a stand-in for the readout of a
    content-free input."""
    hidden: int
    vocab: int
    h_rows: torch.Tensor
    W: torch.Tensor | None
    tokens: np.ndarray
    opt_off: np.ndarray
    q_off: np.ndarray
    prior: np.ndarray

    @property
    def n_rows(self):
        return int(self.opt_off[-1])

    @property
    def n_opts(self):
        return len(self.opt_off) - 1

    @property
    def n_questions(self):
        return len(self.q_off) - 1


def make_options(seed: int = 0, n_questions: int = 16, opts=(2, 8), tokens=(1, 4),
                 hidden: int = 2048, vocab: int = 151936, w_std: float = 0.02,
                 with_W: bool = True) -> OptionWorkload:
    """Seeded option workload.  Draw order (one torch.Generator): options per
    question U{opts}, tokens per option U{tokens}, token ids uniform over the
    vocabulary, h_rows ~ N(0, 1) bf16 [rows, hidden], prior ~ N(-ln vocab, 1)
    fp32 per option, W ~ N(0, w_std) bf16 [vocab, hidden] (last, so
    with_W=False, for a caller that has its LM head already, leaves every
    other value unchanged)."""
    g = torch.Generator().manual_seed(seed)
    k = torch.randint(opts[0], opts[1] + 1, (n_questions,), generator=g)
    q_off = np.concatenate([[0], np.cumsum(k.numpy())]).astype(np.int32)
    n_opts = int(q_off[-1])
    m = torch.randint(tokens[0], tokens[1] + 1, (n_opts,), generator=g)
    opt_off = np.concatenate([[0], np.cumsum(m.numpy())]).astype(np.int32)
    n_rows = int(opt_off[-1])
    toks = torch.randint(0, vocab, (n_rows,), generator=g).numpy().astype(np.int32)
    h_rows = torch.randn(n_rows, hidden, generator=g).bfloat16()
    prior = (torch.randn(n_opts, generator=g) - float(np.log(vocab))).numpy().astype(np.float32)
    W = (torch.randn(vocab, hidden, generator=g) * w_std).bfloat16() if with_W else None
    return OptionWorkload(hidden, vocab, h_rows, W, toks, opt_off, q_off, prior)


@dataclass
class Request:
    """One request of a stream: branch token CSR, q / k / v in the node-token
    order of its own plan, final hidden states and label CSR (CPU)."""
    tok_offsets: np.ndarray
    tokens: np.ndarray
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    h: torch.Tensor
    label_off: np.ndarray
    label_ids: np.ndarray


def make_request_stream(n_requests: int, seed: int = 0, prefix: int = 2000, n_branches: int = 5,
                        suffix: int = 48, shape: Shape | None = None,
                        n_labels: int = 2) -> list:
    """Independent requests shaped like the yes/no configuration (a shared
    prefix and n_branches suffixes), for continuous batching; the LM head is
    the caller's.  Draw order per request (one torch.Generator): prefix
    tokens, each suffix's tokens (its first token redrawn until distinct from
    the earlier suffixes' first tokens), q, k, v ~ N(0, 1) bf16 in node-token
    order (prefix rows, then each suffix's rows), h ~ N(0, 1) bf16, label ids
    (distinct per branch)."""
    sh = shape or Shape(32, 4, 128, 16, 2048, 151936)
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(n_requests):
        pre = torch.randint(0, sh.vocab, (prefix,), generator=g)
        sufs, firsts = [], set()
        for _ in range(n_branches):
            s = torch.randint(0, sh.vocab, (suffix,), generator=g)
            while int(s[0]) in firsts:
                s[0] = torch.randint(0, sh.vocab, (1,), generator=g)
            firsts.add(int(s[0]))
            sufs.append(s)
        seqs = [torch.cat([pre, s]).numpy().astype(np.int32) for s in sufs]
        off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
        T = prefix + n_branches * suffix
        q = torch.randn(T, sh.n_q_heads, sh.head_dim, generator=g).bfloat16()
        k = torch.randn(T, sh.n_kv_heads, sh.head_dim, generator=g).bfloat16()
        v = torch.randn(T, sh.n_kv_heads, sh.head_dim, generator=g).bfloat16()
        h = torch.randn(n_branches, sh.hidden, generator=g).bfloat16()
        ids = np.concatenate([_draw_distinct(g, sh.vocab, n_labels) for _ in range(n_branches)])
        loff = np.arange(0, n_labels * (n_branches + 1), n_labels, dtype=np.int32)
        out.append(Request(off, np.concatenate(seqs), q, k, v, h, loff, ids.astype(np.int32)))
    return out
