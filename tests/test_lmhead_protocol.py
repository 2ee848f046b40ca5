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
  issuer overwrites only after the four warps are done with it.

The abort paths are modelled too: any wait may give up (its time limit ran
out), which raises the CTA's abort flag; every other role's wait then returns
false unless its phase is already complete, and each role follows the
kernel's abort sequence (the producer waits for the loads it issued, the
issuer commits and waits for its products on the drain barrier, the epilogue
warps leave their loop).  Every role must still end, with no product or load
in flight when the CTA releases TMEM."""
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
    def __init__(self, units, stages, nk, seed, slip=None, timeout_p=0.0):
        self.units, self.stages, self.nk = units, stages, nk
        self.rng, self.slip = random.Random(seed), slip
        self.timeout_p, self.timed_out, self.abort = timeout_p, False, False
        B = Barrier
        self.full = [B(f"full{s}", 1) for s in range(stages)]
        self.empty = [B(f"empty{s}", 1) for s in range(stages)]
        self.acc_full = [B(f"acc_full{b}", 1) for b in range(2)]
        # the kernel counts 128 threads; one arrival per warp here
        self.acc_empty = [B(f"acc_empty{b}", 3 if slip == "acc_empty_3" else 4) for b in range(2)]
        self.unit_full = [B(f"unit_full{r}", 1) for r in range(RING)]
        self.unit_empty = [B(f"unit_empty{r}", 5) for r in range(RING)]
        self.drain = B("drain", 1)
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
        issued = [None] * self.stages
        ok = True
        seq = list(self.units) + [-1]
        for i, u in enumerate(seq):
            r = i % RING
            if i >= RING and self.slip != "no_unit_empty_wait":
                ok = yield ("wait", self.unit_empty[r], i // RING - 1, True)
                if not ok:
                    break
            assert self.ring[r] is None or self.ring_readers[r] == {"issuer", 0, 1, 2, 3}, (
                "ring slot overwritten before every reader", r, self.ring_readers[r])
            self.ring[r] = (i, u)
            self.ring_readers[r] = set()
            self.unit_full[r].arrive()
            if u < 0:
                break
            for k in range(self.nk):
                ok = yield ("wait", self.empty[s], n_loads // self.stages - 1, True)
                if not ok:
                    break
                self.stage[s] = None
                self.tma.append((s, (i, k)))
                issued[s] = n_loads // self.stages
                n_loads += 1
                s = (s + 1) % self.stages
            if not ok:
                break
        if not ok:
            self.abort = True
        # the loads issued have landed before the CTA exits
        if self.slip != "producer_leaves_loads":
            for st in range(self.stages):
                if issued[st] is not None:
                    yield ("wait", self.full[st], issued[st], False)

    def issuer(self):
        n_reads = 0
        ok = True
        for i in range(len(self.units) + 1):
            r = i % RING
            ok = yield ("wait", self.unit_full[r], i // RING, True)
            if not ok:
                break
            assert self.ring[r][0] == i
            u = self.ring[r][1]
            self.ring_readers[r].add("issuer")
            self.unit_empty[r].arrive()
            if u < 0:
                break
            b = i & 1
            ok = yield ("wait", self.acc_empty[b], (i >> 1) - 1, True)
            if not ok:
                break
            for k in range(self.nk):
                s = n_reads % self.stages
                ok = yield ("wait", self.full[s], n_reads // self.stages, True)
                if not ok:
                    break
                self.pipe.append(("mma", b, i, k, s))
                self.pipe.append(("commit", self.empty[s]))
                n_reads += 1
            if not ok:
                break
            self.pipe.append(("commit", self.acc_full[b]))
        if not ok:
            self.abort = True
        # every product issued finishes before TMEM is released
        if self.slip != "issuer_leaves_products":
            self.pipe.append(("commit", self.drain))
            yield ("wait", self.drain, 0, False)

    def epilogue_warp(self, q):
        for i in range(len(self.units) + 1):
            r = i % RING
            ok = yield ("wait", self.unit_full[r], i // RING, True)
            if not ok:
                self.abort = True
                return
            assert self.ring[r][0] == i
            u = self.ring[r][1]
            self.ring_readers[r].add(q)
            self.unit_empty[r].arrive()
            if u < 0:
                break
            b = i & 1
            ok = yield ("wait", self.acc_full[b], i >> 1, True)
            if not ok:
                self.abort = True
                return
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

        def advance(i, value=None):
            try:
                waiting[i] = roles[i].send(value) if value is not None else next(roles[i])
            except StopIteration:
                live.discard(i)
                waiting[i] = None

        for i in range(len(roles)):
            advance(i)
        while live:
            choices = []
            for i in live:
                _, bar, k, abortable = waiting[i]
                if self.ready(bar, k):
                    choices.append(("go", i))
                elif abortable and self.abort:
                    choices.append(("stop", i))
                elif (abortable and self.timeout_p and not self.timed_out
                      and self.rng.random() < self.timeout_p):
                    # (the abort sequences' own waits are bounded too, but
                    # their engines always finish, so they are not modelled
                    # as giving up)
                    choices.append(("timeout", i))
            if self.pipe:
                choices.append(("pipe", None))
            if self.tma:
                choices.append(("tma", None))
            if not choices:
                break
            kind, i = self.rng.choice(choices)
            if kind == "go":
                advance(i, True)
            elif kind == "stop":
                advance(i, False)
            elif kind == "timeout":
                self.timed_out = True
                advance(i, False)
            elif kind == "pipe":
                self.step_pipe()
            else:
                self.step_tma()
        assert not live, "deadlock: " + str(
            [(waiting[i][1].name, waiting[i][2]) for i in sorted(live)])
        # every role reached the block barrier before TMEM is released
        assert not self.pipe, "products or commits in flight at exit"
        assert not self.tma, "loads in flight at exit"
        return self


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


@pytest.mark.parametrize("stages", [2, 3, 6])
@pytest.mark.parametrize("nk", [1, 3])
def test_any_wait_may_give_up(stages, nk):
    """One wait, anywhere, runs out of time: the abort flag stops the others,
    every role ends and nothing is left in flight."""
    aborted = 0
    for seed in range(300):
        m = Model(list(range(7)), stages, nk, seed, timeout_p=0.02).run()
        aborted += m.abort
    assert aborted > 50


@pytest.mark.parametrize("slip", ["producer_leaves_loads", "issuer_leaves_products"])
def test_abort_slips_are_caught(slip):
    caught = 0
    for seed in range(300):
        try:
            Model(list(range(7)), 4, 2, seed, slip, timeout_p=0.05).run()
        except AssertionError:
            caught += 1
    assert caught > 0
