"""A host model of the attention kernel's barrier protocol (attn.cu, one
CTA): the K and V producers, the two halves' MMA issuers, the eight softmax
warps and the tensor pipe, which completes products in issue order.  Random
interleavings of those roles must

- always finish (no role waits forever);
- never let a barrier complete twice past a phase some role still waits for
  (the hardware waits on the phase's parity, so that wait would never end);
- give every product and every softmax the data of the right unit: S_h(j)
  read by the softmax of unit j, P_h(j) (written over S_h in TMEM) read by
  P.V of unit j before QK of unit j+1 overwrites it, K(j) and V(j) in their
  stage when read, O_h rescaled only between P.V of units j-1 and j.

The model follows the kernel's order of waits, arrivals and commits,
including the halves' turns on the tensor pipe (A0 B0 A1 B1 ...: p_full of
one half also counts the other half's issue); each barrier counts its
completions, and a wait names the completion it needs (the parity the kernel
passes is that index's low bit).

The abort paths are modelled too: any wait may give up (its time limit ran
out), which raises the CTA's abort flag; every other role's wait then returns
false unless its phase is already complete.  Each role then follows the
kernel's abort sequence: a producer waits for the loads it issued (it always
does, before the exit), an issuer commits and waits for all of its products
on a drain barrier of its own (o_full completes only when all of a half's
products ran, so the softmax never reads a partial O), the softmax stops.
Every role must still end, with no product or load in flight when the CTA
releases TMEM and exits, and TMEM released once.

Planted slips (a missing wait, a wrong arrival count, an abort path that
leaves work in flight) are caught; see the last tests."""
import random

import pytest

K_STAGES, V_STAGES = 3, 2


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
    def __init__(self, n_units, n_halves, seed, slip=None, timeout_p=0.0):
        self.n, self.H, self.rng, self.slip = n_units, n_halves, random.Random(seed), slip
        self.timeout_p, self.timed_out, self.abort = timeout_p, False, False
        self.tmem_frees = 0
        B = Barrier
        paired = n_halves == 2
        self.q_full = B("q_full", 1)
        self.k_full = [B(f"k_full{s}", 1) for s in range(K_STAGES)]
        self.k_empty = [B(f"k_empty{s}", n_halves) for s in range(K_STAGES)]
        self.v_full = [B(f"v_full{s}", 1) for s in range(V_STAGES)]
        v_count = 1 if slip == "v_empty_one_half" else n_halves
        self.v_empty = [B(f"v_empty{s}", v_count) for s in range(V_STAGES)]
        self.s_full = [B(f"s_full{h}", 1) for h in range(2)]
        self.p_full = [B(f"p_full{h}", 4 + (1 if paired else 0)) for h in range(2)]
        self.o_full = [B(f"o_full{h}", 1) for h in range(2)]
        self.drain = [B(f"drain{h}", 1) for h in range(2)]
        self.first_turn = B("first_turn", 1)
        # data: what each buffer holds (None: being loaded)
        self.k_stage = [None] * K_STAGES
        self.v_stage = [None] * V_STAGES
        # per half and softmax warp (its 32 TMEM lanes): ("S", j) after QK(j),
        # ("P", j) once that warp has written P over S
        self.S = [[None] * 4 for _ in range(2)]
        self.o_units = [0, 0]       # P.V products accumulated into O_h
        self.pv_in_flight = [0, 0]  # issued, not completed
        self.pipe = []              # issued products / commits, completed in order
        self.tma = []               # loads in flight

    def ready(self, b, k):
        """A wait for completion k of b: done when b.done > k; the kernel's
        parity wait is only sound while b.done <= k + 1."""
        assert b.done <= k + 1, f"{b.name}: completion {b.done} past awaited {k}"
        return b.done > k

    def producer(self, is_k):
        n_st = K_STAGES if is_k else V_STAGES
        full = self.k_full if is_k else self.v_full
        empty = self.k_empty if is_k else self.v_empty
        stage = self.k_stage if is_k else self.v_stage
        if is_k:
            self.tma.append((None, None, None, self.q_full))
        issued = [None] * n_st
        ok = True
        for it in range(self.n):
            s = it % n_st
            if it >= n_st:  # the stage's previous use is done
                ok = yield ("wait", empty[s], it // n_st - 1, True)
                if not ok:
                    break
            stage[s] = None
            self.tma.append((stage, s, it, full[s]))
            issued[s] = it // n_st
        if not ok:
            self.abort = True
        # every load issued has landed before the CTA exits
        if self.slip != "producer_leaves_loads":
            if is_k:
                yield ("wait", self.q_full, 0, False)
            for s in range(n_st):
                if issued[s] is not None:
                    yield ("wait", full[s], issued[s], False)

    def issuer(self, h):
        """Group g = PV_h(g-1) (g > 0) then QK_h(g) (g < n); the data waits,
        then the turn, then the issues; with two halves an arrival hands the
        turn to the other half."""
        paired = self.H == 2
        ok = yield ("wait", self.q_full, 0, True)
        g = 0
        while ok and g <= self.n:
            do_pv, do_qk = g > 0, g < self.n
            if do_qk:
                ok = yield ("wait", self.k_full[g % K_STAGES], g // K_STAGES, True)
            if ok and do_pv:
                ok = yield ("wait", self.v_full[(g - 1) % V_STAGES], (g - 1) // V_STAGES, True)
                if ok and self.slip != "no_p_full_wait":
                    ok = yield ("wait", self.p_full[h], g - 1, True)
            if ok and paired and h == 1 and g == 0:
                ok = yield ("wait", self.first_turn, 0, True)
            if not ok:
                break
            if do_pv:
                self.pv_in_flight[h] += 1
                self.pipe.append(("pv", h, g - 1, (g - 1) % V_STAGES))
            if do_qk:
                self.pipe.append(("qk", h, g, g % K_STAGES))
            if paired:
                (self.p_full[0] if h == 1 else self.first_turn if g == 0 else self.p_full[1]).arrive()
            if do_pv:
                self.pipe.append(("commit", self.v_empty[(g - 1) % V_STAGES]))
            if do_qk:
                self.pipe.append(("commit", self.s_full[h]))
                self.pipe.append(("commit", self.k_empty[g % K_STAGES]))
            g += 1
        if ok:
            self.pipe.append(("commit", self.o_full[h]))
            yield ("wait", self.o_full[h], 0, False)
        else:
            # gave up: o_full stays incomplete; the products issued so far
            # drain before the exit
            self.abort = True
            if self.slip == "o_full_on_abort":  # the softmax could read a partial O
                self.pipe.append(("commit", self.o_full[h]))
                yield ("wait", self.o_full[h], 0, False)
            elif self.slip != "issuer_leaves_products":
                self.pipe.append(("commit", self.drain[h]))
                yield ("wait", self.drain[h], 0, False)

    def softmax_warp(self, h, w):
        for it in range(self.n):
            ok = yield ("wait", self.s_full[h], it, True)
            if not ok:
                self.abort = True
                return
            assert self.S[h][w] == ("S", it), ("softmax reads S", h, w, it, self.S[h][w])
            if it > 0:
                # the commit after QK_h(it) covers P.V of unit it-1: O_h is stable
                assert self.pv_in_flight[h] == 0 and self.o_units[h] == it
            self.S[h][w] = ("P", it)  # this warp's rows of P_h, over S_h
            self.p_full[h].arrive()
        ok = yield ("wait", self.o_full[h], 0, True)
        if not ok:
            self.abort = True
            return
        assert self.o_units[h] == self.n, ("epilogue reads a partial O", h)

    def step_pipe(self):
        op = self.pipe.pop(0)
        if op[0] == "qk":
            _, h, g, s = op
            assert self.k_stage[s] == g, ("QK reads K", h, g, self.k_stage[s])
            assert g == 0 or self.S[h] == [("P", g - 1)] * 4, ("QK overwrites live P", h, g)
            self.S[h] = [("S", g)] * 4
        elif op[0] == "pv":
            _, h, g, s = op
            assert self.v_stage[s] == g, ("PV reads V", h, g, self.v_stage[s])
            assert self.S[h] == [("P", g)] * 4, ("PV reads P", h, g, self.S[h])
            assert self.o_units[h] == g
            self.o_units[h] += 1
            self.pv_in_flight[h] -= 1
        else:
            op[1].arrive()

    def step_tma(self):
        i = self.rng.randrange(len(self.tma)) if self.rng.random() < 0.3 else 0
        stage, s, unit, bar = self.tma.pop(i)
        if stage is not None:
            stage[s] = unit
        bar.arrive()

    def run(self):
        roles = [self.producer(True), self.producer(False)]
        roles += [self.issuer(h) for h in range(self.H)]
        roles += [self.softmax_warp(h, w) for h in range(self.H) for w in range(4)]
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
                    choices.append(("stop", i))  # the wait saw the abort flag
                elif (abortable and self.timeout_p and not self.timed_out
                      and self.rng.random() < self.timeout_p):
                    # its time limit ran out (the abort sequences' own waits
                    # are bounded too, but their engines always finish)
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
        # every role reached the final block barrier: TMEM is released (once)
        # and the CTA exits; nothing may still be in flight
        assert not self.pipe, "products or commits in flight at exit"
        assert not self.tma, "loads in flight at exit"
        self.tmem_frees += 1
        assert self.tmem_frees == 1
        return self


@pytest.mark.parametrize("n_halves", [1, 2])
@pytest.mark.parametrize("n_units", [1, 2, 3, 4, 7, 16])
def test_protocol_random_interleavings(n_units, n_halves):
    for seed in range(200):
        m = Model(n_units, n_halves, seed).run()
        assert not m.abort and m.o_units[:n_halves] == [n_units] * n_halves


@pytest.mark.parametrize("slip", ["no_p_full_wait", "v_empty_one_half"])
def test_planted_slips_are_caught(slip):
    caught = 0
    for n_units in (2, 3, 5):
        for seed in range(100):
            try:
                Model(n_units, 2, seed, slip).run()
            except AssertionError:
                caught += 1
    assert caught > 0


@pytest.mark.parametrize("n_halves", [1, 2])
@pytest.mark.parametrize("n_units", [1, 2, 5, 9])
def test_any_wait_may_give_up(n_units, n_halves):
    """One wait, anywhere, runs out of time: the abort flag stops the others,
    every role ends and nothing is left in flight."""
    aborted = 0
    for seed in range(300):
        m = Model(n_units, n_halves, seed, timeout_p=0.02).run()
        aborted += m.abort
    assert aborted > 50


@pytest.mark.parametrize("slip", ["producer_leaves_loads", "issuer_leaves_products",
                                  "o_full_on_abort"])
def test_abort_slips_are_caught(slip):
    caught = 0
    for n_units in (2, 3, 5):
        for seed in range(200):
            try:
                Model(n_units, 2, seed, slip, timeout_p=0.05).run()
            except AssertionError:
                caught += 1
    assert caught > 0
