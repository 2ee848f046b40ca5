"""The C++ continuous batcher against the oracle's admission rule, and each
request's part of a batch plan against the request's own plan.  Host only:
no GPU needed."""
import numpy as np
import pytest

from oracle import batching as OB


def _stream(rng, n_req, vocab=7):
    reqs = []
    for _ in range(n_req):
        base = list(rng.integers(0, vocab, int(rng.integers(1, 120))))
        seqs = []
        for _ in range(int(rng.integers(1, 7))):
            cut = int(rng.integers(0, len(base) + 1))
            s = base[:cut] + list(rng.integers(0, vocab, int(rng.integers(0, 30))))
            seqs.append(s if s else [1])
        off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
        reqs.append((off, np.concatenate([np.asarray(s, np.int32) for s in seqs])))
    return reqs


def _shape(lib):
    return lib.make_shape(8, 2, 64, 16, 64, 100)


@pytest.mark.parametrize("seed", range(12))
def test_batches_match_the_oracle(lib, seed):
    rng = np.random.default_rng(seed)
    reqs = _stream(rng, int(rng.integers(1, 25)))
    max_tokens = int(rng.integers(30, 600))
    max_requests = int(rng.integers(1, 7))
    b = lib.Batcher(_shape(lib), max_tokens, max_requests)
    sizes, nbr = [], []
    for i, (off, tok) in enumerate(reqs):
        rid, nt = b.submit(off, tok)
        assert rid == i
        assert nt == OB.node_tokens(off, tok)
        sizes.append(nt)
        nbr.append(len(off) - 1)
    assert b.pending() == (len(reqs), sum(sizes))
    want = OB.form_batches(sizes, max_tokens, max_requests)
    for batch in want:
        plan, ids, boff, roff = b.next()
        assert ids.tolist() == batch
        wb, wr = OB.batch_offsets(batch, sizes, nbr)
        assert boff.tolist() == wb.tolist() and roff.tolist() == wr.tolist()
        st = plan.stats()
        assert st["node_tokens"] == roff[-1] and st["n_requests"] == len(batch)
        # each request's segments are its own plan's, shifted by its row offset
        segs = plan.segments()
        rounds = plan.branches()["round"]
        for i, r in enumerate(batch):
            off, tok = reqs[r]
            alone = lib.sp_plan_build(_shape(lib), np.zeros(len(off) - 1, np.int32), off, tok,
                                      (1 << 31) - 1)
            sa = alone.segments()
            mine = segs["req"] == i
            assert np.array_equal(segs["len"][mine], sa["len"])
            assert np.array_equal(segs["shared"][mine], sa["shared"])
            assert np.array_equal(segs["round"][mine], sa["round"])
            assert np.array_equal(segs["node_start"][mine] - roff[i], sa["node_start"])
            assert np.array_equal(rounds[boff[i]:boff[i + 1]], alone.branches()["round"])
    assert b.next() is None and b.pending() == (0, 0)


def test_batcher_arguments_and_limits(lib):
    b = lib.Batcher(_shape(lib), 100, 4)
    with pytest.raises(lib.SpError) as e:
        b.submit([0, 0], [])  # an empty branch
    assert e.value.status == 1
    with pytest.raises(lib.SpError) as e:
        b.submit([0, 32769], np.zeros(32769, np.int32))  # a branch over 32768 tokens
    assert e.value.status == 2
    with pytest.raises(lib.SpError) as e:
        lib.Batcher(_shape(lib), 0, 4)
    assert e.value.status == 1
    assert b.pending() == (0, 0) and b.next() is None


def test_pool_full_leaves_the_queue(lib):
    """A batch whose plan needs more pages than the pool has returns
    SP_ERR_POOL_FULL and leaves every request queued."""
    b = lib.Batcher(_shape(lib), 10 ** 6, 8)
    for r in range(3):
        b.submit([0, 40, 80], np.concatenate([np.arange(40), np.arange(40) + 1000 * (r + 1)]))
    with pytest.raises(lib.SpError) as e:
        b.next(max_pages=2)
    assert e.value.status == 3
    assert b.pending()[0] == 3
    plan, ids, _, _ = b.next()
    assert ids.tolist() == [0, 1, 2]
