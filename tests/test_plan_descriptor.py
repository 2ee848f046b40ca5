"""The planner's device descriptor, checked on the host: a float64 emulation
of what the attention kernels do with it (walk each tile's KV units over
ancestor and own levels with the causal bound, reading a level from the k / v
inputs when the call computes it and from the pool otherwise; write the
call's shared segments into the pool after its tiles; merge split partials)
must reproduce the oracle's unshared attention exactly.  The pool starts as
NaN, so a level read from the pool before a call has written it shows up.

This pins the work decomposition (pages, chains, units, splits, merges,
recomputed rows) independently of any GPU arithmetic."""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import staging as S
from prefill_only_shared_gb300.workloads import make_workload, small_case

from test_oracle_staging import csr, random_case

SEG = np.dtype([("node_start", "<i8"), ("len", "<i4"), ("page_off", "<i4"), ("chain_off", "<i4"),
                ("chain_len", "<i4"), ("round", "<i4"), ("shared", "<i4")])
TILE = np.dtype([("seg", "<i4"), ("t0", "<i4"), ("nt", "<i4"), ("u_lo", "<i4"), ("u_hi", "<i4"),
                 ("part", "<i4"), ("merge", "<i4"), ("seg2", "<i4"), ("t0b", "<i4"), ("ntb", "<i4"),
                 ("p0", "<i4"), ("p1", "<i4")])
MERGE = np.dtype([("seg", "<i4"), ("t0", "<i4"), ("nt", "<i4"), ("part0", "<i4"), ("nparts", "<i4"),
                  ("p0", "<i4"), ("p1", "<i4"), ("p2", "<i4")])
APP = np.dtype([("seg", "<i4"), ("page", "<i4")])
ROWS, UNIT, PAGE = 256, 128, 16


def decode(blob):
    h = np.frombuffer(blob, dtype="<i8", count=12)
    off = dict(zip(["segs", "pages", "chain", "append", "tiles", "merges"], h[:6]))
    n = dict(zip(["segs", "pages", "chain", "append", "tiles", "merges"], h[6:]))

    def arr(name, dt):
        return np.frombuffer(blob, dtype=dt, count=int(n[name]), offset=int(off[name]))

    return (arr("segs", SEG), arr("pages", "<i4"), arr("chain", "<i4"), arr("append", APP),
            arr("tiles", TILE), arr("merges", MERGE))


def emulate(plan, q, k, v, Hq, Hkv, d, schedule="rounds", pool=None):
    """pool: a persistent (pages, 2, Hkv, PAGE, d) array for plans built with a
    prefix cache (cached levels are read from it, new shared segments written
    to it); None = a fresh NaN pool."""
    segs, pages, chain, app, tiles, merges = decode(plan.descriptor())
    st = plan.stats()
    G = Hq // Hkv
    if pool is None:
        pool = np.full((max(st["pages_used"], 1), 2, Hkv, PAGE, d), np.nan)
    T = st["node_tokens"]
    out = np.full((T, Hq, d), np.nan)
    lse = np.full((T, Hq), np.nan)
    scale = 1.0 / math.sqrt(d)
    seen = np.zeros(T, dtype=np.int64)
    per_round = schedule in ("rounds", "tree_rounds")
    kinds = (2,) if schedule.startswith("tree") else (0, 1)
    for r in (range(st["n_rounds"]) if per_round else [-1]):
        for kind in kinds:
            ci = plan.call_info(r, kind)

            def in_call(x):
                if x["shared"] == 2:  # a cached level: K/V only in the pool
                    return False
                kind_ok = kind == 2 or (x["shared"] == 1) == (kind == 0)
                return kind_ok and (r < 0 or x["round"] == r)

            # the call writes exactly its shared segments' pages into the pool
            apps = app[ci["append_off"]:ci["append_off"] + ci["n_append"]]
            want = sorted((i, p) for i, x in enumerate(segs) if in_call(x) and x["shared"] == 1
                          for p in range((x["len"] + PAGE - 1) // PAGE))
            assert sorted((int(a["seg"]), int(a["page"])) for a in apps) == want
            parts = {}

            def attend_rows(seg, t0, nt, keys):
                for tok in range(nt):
                    row = seg["node_start"] + t0 + tok
                    seen[row] += 1
                    vis = [kv for kv in keys if kv[2] <= t0 + tok]
                    for hq in range(Hq):
                        g = hq // G
                        sc = np.array([kk[0][g] @ q[row, hq] for kk in vis]) * scale
                        m = sc.max()
                        pr = np.exp(sc - m)
                        out[row, hq] = (pr @ np.array([kk[1][g] for kk in vis])) / pr.sum()
                        lse[row, hq] = m + math.log(pr.sum())

            def level_keys(x, ln, own):
                ks = []
                for pos in range(ln):
                    if in_call(x):
                        kk, vv = k[x["node_start"] + pos], v[x["node_start"] + pos]
                    else:
                        pg = pages[x["page_off"] + pos // PAGE]
                        kk, vv = pool[pg, 0, :, pos % PAGE], pool[pg, 1, :, pos % PAGE]
                    ks.append((kk, vv, pos if own else -1))
                return ks

            def paired_tile(td, in_call):
                # two sibling leaves' last tokens, each in one half: common
                # ancestors, then each half's own segment (never split)
                sa, sb = segs[td["seg"]], segs[td["seg2"]]
                assert td["part"] < 0 and td["merge"] == -1 and td["u_lo"] == 0
                assert sa["shared"] == 0 and sb["shared"] == 0 and td["nt"] <= ROWS // 2 // G
                assert td["ntb"] <= ROWS // 2 // G
                assert td["t0"] + td["nt"] == sa["len"] and td["t0b"] + td["ntb"] == sb["len"]
                ca = chain[sa["chain_off"]:sa["chain_off"] + sa["chain_len"]]
                cb = chain[sb["chain_off"]:sb["chain_off"] + sb["chain_len"]]
                assert list(ca) == list(cb) and len(ca) > 0
                anc = []
                n_units = 0
                for c in ca:
                    x = segs[c]
                    anc += level_keys(x, x["len"], False)
                    n_units += (x["len"] + UNIT - 1) // UNIT
                n_units += (sa["len"] + UNIT - 1) // UNIT + (sb["len"] + UNIT - 1) // UNIT
                assert td["u_hi"] == n_units
                attend_rows(sa, td["t0"], td["nt"], anc + level_keys(sa, sa["len"], True))
                attend_rows(sb, td["t0b"], td["ntb"], anc + level_keys(sb, sb["len"], True))

            call_merges = merges[ci["merge_off"]:ci["merge_off"] + ci["n_merges"]]
            for td in tiles[ci["tile_off"]:ci["tile_off"] + ci["n_tiles"]]:
                if td["seg2"] >= 0:
                    paired_tile(td, in_call)
                    continue
                s = segs[td["seg"]]
                if td["part"] >= 0:  # a split part names its merge entry
                    md = call_merges[td["merge"]]
                    assert md["part0"] <= td["part"] < md["part0"] + md["nparts"]
                    assert (md["seg"], md["t0"], md["nt"]) == (td["seg"], td["t0"], td["nt"])
                else:
                    assert td["merge"] == -1
                levels = [segs[c] for c in chain[s["chain_off"]:s["chain_off"] + s["chain_len"]]]
                lv = [(x, x["len"], False) for x in levels]
                lv.append((s, td["t0"] + td["nt"], True))
                keys = []  # (K, V, position within own level or -1)
                u = 0
                for x, ln, own in lv:
                    for j in range((ln + UNIT - 1) // UNIT):
                        if td["u_lo"] <= u < td["u_hi"]:
                            for pos in range(j * UNIT, min(ln, (j + 1) * UNIT)):
                                if in_call(x):
                                    kk, vv = k[x["node_start"] + pos], v[x["node_start"] + pos]
                                else:
                                    pg = pages[x["page_off"] + pos // PAGE]
                                    kk, vv = pool[pg, 0, :, pos % PAGE], pool[pg, 1, :, pos % PAGE]
                                keys.append((kk, vv, pos if own else -1))
                        u += 1
                assert td["u_hi"] <= u
                for tok in range(td["nt"]):
                    row = s["node_start"] + td["t0"] + tok
                    if td["part"] < 0:
                        seen[row] += 1
                    vis = [kv for kv in keys if kv[2] <= td["t0"] + tok]
                    for hq in range(Hq):
                        g = hq // G
                        if vis:
                            sc = np.array([kk[0][g] @ q[row, hq] for kk in vis]) * scale
                            m = sc.max()
                            p = np.exp(sc - m)
                            o = (p @ np.array([kk[1][g] for kk in vis])) / p.sum()
                            l = m + math.log(p.sum())
                        else:
                            o, l = np.zeros(d), -np.inf
                        if td["part"] < 0:
                            out[row, hq], lse[row, hq] = o, l
                        else:
                            parts[(td["part"], row, hq)] = (o, l)
            for a in apps:  # after the tiles: no tile of the call reads them
                x = segs[a["seg"]]
                pg = pages[x["page_off"] + a["page"]]
                for slot in range(PAGE):
                    t = a["page"] * PAGE + slot
                    if t < x["len"]:
                        pool[pg, 0, :, slot] = k[x["node_start"] + t]
                        pool[pg, 1, :, slot] = v[x["node_start"] + t]
                    else:
                        pool[pg, :, :, slot] = 0.0
            for md in merges[ci["merge_off"]:ci["merge_off"] + ci["n_merges"]]:
                s = segs[md["seg"]]
                for tok in range(md["nt"]):
                    row = s["node_start"] + md["t0"] + tok
                    seen[row] += 1
                    for hq in range(Hq):
                        ps = [parts[(md["part0"] + i, row, hq)] for i in range(md["nparts"])]
                        L = np.logaddexp.reduce([p[1] for p in ps])
                        out[row, hq] = sum(np.exp(p[1] - L) * p[0] for p in ps if p[1] > -np.inf)
                        lse[row, hq] = L
    return out, lse, seen


def check(req, offs, toks, q, k, v, Hq, Hkv, d, lib, n_sms):
    plan = lib.sp_plan_build(lib.make_shape(Hq, Hkv, d, 16, 64, 1000), req, offs, toks, 1 << 20,
                             n_sms=n_sms)
    ref = S.build_plan(req, offs, toks)
    ro, rl, _ = A.reference_attention(ref, q, k, v)
    for schedule in ("rounds", "all", "tree", "tree_rounds"):
        out, lse, seen = emulate(plan, q, k, v, Hq, Hkv, d, schedule)
        assert np.abs(out - ro).max() < 1e-10
        assert np.abs(lse - rl).max() < 1e-10
        # every row written once, plus one more for each recomputed final row
        extra = np.zeros_like(seen)
        for b in range(len(ref.paths)):
            if ref.recompute[b]:
                extra[ref.branch_last_row(b)] += 1
        assert (seen == 1 + extra).all()
    return plan


@pytest.mark.parametrize("n_sms", [1, 8, 152])
@pytest.mark.parametrize("G,Hkv", [(4, 2), (8, 1), (1, 2)])
def test_descriptor_tree_cases(lib, n_sms, G, Hkv):
    trees = [(130, [(70, [(3, []), (65, []), (1, [])]), (17, [])]), (40, []),
             (5, [(1, []), (200, [])])]
    wl = small_case(trees, n_q_heads=G * Hkv, n_kv_heads=Hkv, head_dim=64)
    plan = check(wl.req_of_branch, wl.tok_offsets, wl.tokens, A.to64(wl.q), A.to64(wl.k),
                 A.to64(wl.v), G * Hkv, Hkv, 64, lib, n_sms)
    if n_sms == 1:  # calls of a wave or more: sibling leaf tails share CTAs
        tiles = decode(plan.descriptor())[4]
        ci = plan.call_info(-1, 2)
        tree_tiles = tiles[ci["tile_off"]:ci["tile_off"] + ci["n_tiles"]]
        assert (tree_tiles["seg2"] >= 0).sum() >= 1


@pytest.mark.parametrize("seed", range(12))
def test_descriptor_random_tries(lib, seed):
    req, seqs = random_case(seed)
    # longer sequences so several units, pages and splits appear
    rng = np.random.default_rng(seed)
    seqs = [list(s) + list(rng.integers(0, 2, int(rng.integers(0, 90)))) if rng.random() < 0.3 else s
            for s in seqs]
    offs, toks = csr(seqs)
    ref = S.build_plan(req, offs, toks)
    T = ref.node_tokens
    Hq, Hkv, d = 4, 2, 8
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    # head_dim 8 is not a kernel shape; the descriptor does not depend on it
    plan = lib.sp_plan_build(lib.make_shape(Hq, Hkv, 64, 16, 64, 1000), req, offs, toks, 1 << 20,
                             n_sms=int(rng.integers(1, 40)))
    out, lse, seen = emulate(plan, q, k, v, Hq, Hkv, d)
    ro, rl, _ = A.reference_attention(ref, q, k, v)
    assert np.abs(out - ro).max() < 1e-10
    assert np.abs(lse - rl).max() < 1e-10


def test_descriptor_tiny_config(lib):
    wl = make_workload("tiny")
    sh = wl.shape
    plan = check(wl.req_of_branch, wl.tok_offsets, wl.tokens, A.to64(wl.q), A.to64(wl.k),
                 A.to64(wl.v), sh.n_q_heads, sh.n_kv_heads, sh.head_dim, lib, 152)
    assert plan.rounds() == [[0], [1, 2, 3]]


@pytest.mark.parametrize("n_sms", [1, 8, 152])
@pytest.mark.parametrize("name", ["tiny", "yesno", "choice64", "tree2", "batch64"])
def test_tiles_are_listed_longest_first(lib, name, n_sms):
    """Blocks start in list order, so every call lists its tiles (and split
    parts) request by request, in increasing request id (the KV a moment's
    CTAs read stays in L2), and within a request by non-increasing KV units;
    paired tiles appear only in calls that are not split."""
    wl = make_workload(name, tokens_only=True)
    sh = wl.shape
    plan = lib.sp_plan_build(lib.make_shape(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, 16,
                                            sh.hidden, sh.vocab), wl.req_of_branch,
                             wl.tok_offsets, wl.tokens, 1 << 20, n_sms=n_sms)
    tiles = decode(plan.descriptor())[4]
    n_rounds = plan.stats()["n_rounds"]
    for rnd in list(range(n_rounds)) + [-1]:
        for kind in (0, 1, 2):
            ci = plan.call_info(rnd, kind)
            t = tiles[ci["tile_off"]:ci["tile_off"] + ci["n_tiles"]]
            units = (t["u_hi"] - t["u_lo"]).astype(np.int64)
            req = plan.segments()["req"][t["seg"]]
            assert (np.diff(req) >= 0).all(), (rnd, kind)
            for r in np.unique(req):
                assert (np.diff(units[req == r]) <= 0).all(), (rnd, kind, r)
            if ci["n_parts"] > 0:
                assert (t["seg2"] < 0).all(), (rnd, kind)
