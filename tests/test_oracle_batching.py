"""Pins of the continuous-batching rule (oracle/batching.py): brute-force
prefix counting, closed forms and invariants.  CPU only."""
import numpy as np
import pytest

from oracle import batching as OB


def _csr(seqs):
    off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
    return off, np.concatenate([np.asarray(s, np.int32) for s in seqs])


@pytest.mark.parametrize("seed", range(20))
def test_node_tokens_count_distinct_prefixes(seed):
    """A request's node tokens are the distinct non-empty prefixes of its
    branches, counted by brute force over tuples."""
    rng = np.random.default_rng(seed)
    base = list(rng.integers(0, 4, int(rng.integers(1, 30))))
    seqs = []
    for _ in range(int(rng.integers(1, 7))):
        cut = int(rng.integers(0, len(base) + 1))
        s = base[:cut] + list(rng.integers(0, 4, int(rng.integers(0, 10))))
        seqs.append(s if s else [7])
    want = len({tuple(s[:i]) for s in seqs for i in range(1, len(s) + 1)})
    assert OB.node_tokens(*_csr(seqs)) == want


def test_closed_forms():
    # equal requests of t tokens, budget B: batches of floor(B / t) requests
    assert [len(b) for b in OB.form_batches([100] * 10, 350, 64)] == [3, 3, 3, 1]
    # a batch may fill its budget exactly
    assert OB.form_batches([100] * 4, 300, 64) == [[0, 1, 2], [3]]
    # the request cap binds before the budget
    assert [len(b) for b in OB.form_batches([10] * 10, 10 ** 6, 4)] == [4, 4, 2]
    # a request larger than the budget runs alone, and so does everything
    # when the budget is below every request
    assert OB.form_batches([500, 10, 10], 100, 8) == [[0], [1, 2]]
    assert OB.form_batches([50, 60, 70], 10, 8) == [[0], [1], [2]]
    # the rule is first-in first-out: it does not skip a big request to take
    # a smaller later one
    assert OB.form_batches([60, 50, 10], 100, 8) == [[0], [1, 2]]


@pytest.mark.parametrize("seed", range(30))
def test_rule_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    sizes = list(rng.integers(1, 400, int(rng.integers(1, 40))))
    max_tokens = int(rng.integers(50, 1500))
    max_requests = int(rng.integers(1, 9))
    batches = OB.form_batches(sizes, max_tokens, max_requests)
    # every request exactly once, in submission order
    assert [r for b in batches for r in b] == list(range(len(sizes)))
    for i, b in enumerate(batches):
        total = sum(sizes[r] for r in b)
        assert len(b) <= max_requests
        assert total <= max_tokens or len(b) == 1
        # maximal: the next request would break a limit
        if i + 1 < len(batches):
            nxt = batches[i + 1][0]
            assert len(b) == max_requests or total + sizes[nxt] > max_tokens
    boff, roff = OB.batch_offsets(batches[0], sizes, [2] * len(sizes))
    assert boff[-1] == 2 * len(batches[0]) and roff[-1] == sum(sizes[r] for r in batches[0])
