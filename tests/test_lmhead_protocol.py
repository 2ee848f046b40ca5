"""A host model of the readout kernel's barrier protocol (lmhead.cu, one CTA
up to the grid barrier): the TMA producer, which publishes each work unit's
index in a four-slot ring (a fixed run, then units taken from the shared
tail, then -1) and streams the unit's W / h stages; the MMA issuer, which
accumulates a unit into one of two TMEM buffers; the four epilogue warps,
which read a buffer and free it; and the tensor pipe, which completes in
issue order.  Random interleavings, stage counts and unit lists must

- always finish, every role leaving on the -1 sentinel;
- never let a barrier complete twice past a phase some role still waits for
  (the hardware waits on the phase's parity);
- keep every ring slot until the issuer and all four epilogue warps have
  read it, feed each product the stage of its own unit and k-step, and hand
  the epilogue a buffer that holds exactly its unit's products, which the
  issuer overwrites only after the four warps are done with it."""
import random

import pytest

RING = 4


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, self.name
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


class Model:
    def __init__(self, units, stages, nk, seed, slip=None):
        self.units, self.stages, self.nk = units, stages, nk
        self.rng, self.slip = random.Random(seed), slip
        B = Barrier
        self.full = [B(f"full{s}", 1) for s in range(stages)]
        self.empty = [B(f"empty{s}", 1) for s in range(stages)]
        self.acc_full = [B(f"acc_full{b}", 1) for b in range(2)]
        # the kernel counts 128 threads; one arrival per warp here
        self.acc_empty = [B(f"acc_empty{b}", 3 if slip == "acc_empty_3" else 4) for b in range(2)]
        self.unit_full = [B(f"unit_full{r}", 1) for r in range(RING)]
        self.unit_empty = [B(f"unit_empty{r}", 5) for r in range(RING)]
        self.ring = [None] * RING
        self.ring_readers = [set() for _ in range(RING)]
        self.stage = [None] * stages   # (unit position, k) loaded
        self.acc = [None, None]        # (unit position, k-steps accumulated)
        self.acc_readers = [set(), set()]
        self.pipe, self.tma = [], []

    def ready(self, b, k):
        assert b.done <= k + 1, f"{b.name}: completion {b.done} past awaited {k}"
        return b.done > k

    def producer(self):
        s = 0
        n_loads = 0
        seq = list(self.units) + [-1]
        for i, u in enumerate(seq):
            r = i % RING
            if i >= RING and self.slip != "no_unit_empty_wait":
                yield self.unit_empty[r], i // RING - 1
            assert self.ring[r] is None or self.ring_readers[r] == {"issuer", 0, 1, 2, 3}, (
                "ring slot overwritten before every reader", r, self.ring_readers[r])
            self.ring[r] = (i, u)
            self.ring_readers[r] = set()
            self.unit_full[r].arrive()
            if u < 0:
                return
            for k in range(self.nk):
                yield self.empty[s], n_loads // self.stages - 1
                self.stage[s] = None
                self.tma.append((s, (i, k)))
                n_loads += 1
                s = (s + 1) % self.stages

    def issuer(self):
        n_reads = 0
        for i in range(len(self.units) + 1):
            r = i % RING
            yield self.unit_full[r], i // RING
            assert self.ring[r][0] == i
            u = self.ring[r][1]
            self.ring_readers[r].add("issuer")
            self.unit_empty[r].arrive()
            if u < 0:
                break
            b = i & 1
            yield self.acc_empty[b], (i >> 1) - 1
            for k in range(self.nk):
                s = n_reads % self.stages
                yield self.full[s], n_reads // self.stages
                self.pipe.append(("mma", b, i, k, s))
                self.pipe.append(("commit", self.empty[s]))
                n_reads += 1
            self.pipe.append(("commit", self.acc_full[b]))

    def epilogue_warp(self, q):
        for i in range(len(self.units) + 1):
            r = i % RING
            yield self.unit_full[r], i // RING
            assert self.ring[r][0] == i
            u = self.ring[r][1]
            self.ring_readers[r].add(q)
            self.unit_empty[r].arrive()
            if u < 0:
                break
            b = i & 1
            yield self.acc_full[b], i >> 1
            assert self.acc[b] == (i, self.nk), ("epilogue reads an incomplete buffer", b, i,
                                                 self.acc[b])
            self.acc_readers[b].add(q)
            self.acc_empty[b].arrive()

    def step_pipe(self):
        op = self.pipe.pop(0)
        if op[0] == "mma":
            _, b, i, k, s = op
            assert self.stage[s] == (i, k), ("MMA reads the wrong stage", i, k, self.stage[s])
            if k == 0:
                assert self.acc[b] is None or self.acc_readers[b] == {0, 1, 2, 3}, (
                    "buffer overwritten before the epilogue read it", b, i)
                self.acc[b] = (i, 0)
                self.acc_readers[b] = set()
            assert self.acc[b] == (i, k)
            self.acc[b] = (i, k + 1)
        else:
            op[1].arrive()

    def step_tma(self):
        j = self.rng.randrange(len(self.tma)) if self.rng.random() < 0.3 else 0
        s, what = self.tma.pop(j)
        self.stage[s] = what
        self.full[s].arrive()

    def run(self):
        roles = [self.producer(), self.issuer()] + [self.epilogue_warp(q) for q in range(4)]
        waiting = [None] * len(roles)
        live = set(range(len(roles)))

        def advance(i):
            try:
                waiting[i] = next(roles[i])
            except StopIteration:
                live.discard(i)
                waiting[i] = None

        for i in range(len(roles)):
            advance(i)
        while True:
            runnable = [i for i in live if waiting[i] is None or self.ready(*waiting[i])]
            choices = [("role", i) for i in runnable]
            if self.pipe:
                choices.append(("pipe", None))
            if self.tma:
                choices.append(("tma", None))
            if not choices:
                break
            kind, i = self.rng.choice(choices)
            if kind == "role":
                advance(i)
            elif kind == "pipe":
                self.step_pipe()
            else:
                self.step_tma()
        assert not live, "deadlock: " + str(
            [(waiting[i][0].name, waiting[i][1]) for i in sorted(live)])
        assert not self.pipe and not self.tma


@pytest.mark.parametrize("stages", [2, 3, 4, 6, 9, 16])
@pytest.mark.parametrize("nk", [1, 2, 5])
def test_protocol_random_interleavings(stages, nk):
    rng = random.Random(stages * 10 + nk)
    for seed in range(120):
        units = list(range(rng.randrange(0, 11)))  # fixed run and tail: the order is what matters
        Model(units, stages, nk, seed).run()


@pytest.mark.parametrize("slip", ["no_unit_empty_wait", "acc_empty_3"])
def test_planted_slips_are_caught(slip):
    """The ring wait only matters when the stages let the producer run more
    than four units ahead of the slowest reader: six stages of one k-step."""
    caught = 0
    for seed in range(150):
        try:
            Model(list(range(12)), 6, 1, seed, slip).run()
        except AssertionError:
            caught += 1
    assert caught > 0
