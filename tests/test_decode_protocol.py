"""A model of the tensor-core decode kernel's hand-offs (16-bit caches), run on
the CPU under random schedules.

The kernel's roles -- planner, streaming warp, QK issuer, two softmax groups,
PV issuer, output warps -- pass work through mbarriers.  A waiter names the
phase it waits for only by its parity, so every barrier must never run two
phases ahead of a waiter that is about to test it: the test would then report
a completed phase as pending (and the wait would run to its bound).  The model
keeps each barrier's completed-phase count, fails the moment a role tests a
barrier that is two or more phases past the one it waits for, and fails on a
deadlock.  Tensor-core completions (commits) arrive in issue order at random
times, bulk copies land in any order.  Each role takes the same steps, in the
same order, as its code in decode_tc.cuh, the end-of-work marks included
(the planner's last record, the streamer's last stage, the QK issuer's two
metadata buffers, the softmax group whose turn the end tile is, the output
warps' last hand-off slot); the softmax warpgroups and the four output warps
are one actor each (their own barriers between warps are not modelled).  One
test plants the mistake that once went into the kernel (no wait for PV(t - 2)
before completing p_full) and checks that the model catches it."""
import random

import pytest

NS = 3       # stages
IS = 4       # items in flight between softmax and output warps (hand-off and O slots)
QS = 4       # Q slots


class Alias(AssertionError):
    pass


class Bar:
    """An mbarrier: `count` arrivals complete a phase; tests name a phase by parity."""

    def __init__(self, name, count):
        self.name, self.count, self.left, self.done = name, count, count, 0

    def arrive(self, n=1):
        self.left -= n
        assert self.left >= 0, f"{self.name}: too many arrivals"
        if self.left == 0:
            self.done += 1
            self.left = self.count

    def test(self, want):
        """try_wait.parity for phase `want` (0-based): true iff the current phase's parity differs."""
        if self.done >= want + 2:
            raise Alias(f"{self.name}: phase {want} tested with {self.done} phases completed")
        return (self.done & 1) != (want & 1)


class Model:
    def __init__(self, items, rng, pv_wait_before_p_full=True):
        self.rng = rng
        self.items = items                       # tiles per item
        self.tiles = []                          # per tile: (item, head, tail)
        for k, n in enumerate(items):
            for j in range(n):
                self.tiles.append((k, j, n - 1 - j))
        self.T = len(self.tiles)
        self.fix = pv_wait_before_p_full
        b = Bar
        self.full = [b(f"full[{i}]", 1) for i in range(NS)]
        self.empty = [b(f"empty[{i}]", 1) for i in range(NS)]
        self.s_full = [b(f"s_full[{i}]", 1) for i in range(2)]
        self.s_free = [b(f"s_free[{i}]", 1) for i in range(2)]
        self.m_full = [b(f"m_full[{i}]", 1) for i in range(2)]
        self.p_full = [b(f"p_full[{i}]", 1) for i in range(2)]
        self.pv_done = [b(f"pv_done[{i}]", 1) for i in range(2)]
        self.q_free = [b(f"q_free[{i}]", 1) for i in range(QS)]
        self.c_full = [b(f"c_full[{i}]", 2) for i in range(IS)]   # both softmax groups (one twice)
        self.c_free = [b(f"c_free[{i}]", 1) for i in range(IS)]
        self.ofin = [b(f"ofin[{i}]", 1) for i in range(2 * IS)]
        self.ofree = [b(f"ofree[{i}]", 1) for i in range(2 * IS)]
        self.rec_full = [b(f"rec_full[{i}]", 1) for i in range(2)]
        self.rec_empty = [b(f"rec_empty[{i}]", 1) for i in range(2)]
        self.tensor = []       # commits in issue order: lists of barriers to arrive on
        self.copies = []       # landing copies: stage barriers
        self.progress = 0
        self.out_items = 0
        self.end_tile = None   # set by the QK issuer when it meets the end mark

    # -- asynchronous completions
    def commit(self, bars):
        self.tensor.append(bars)

    def fire(self):
        choices = []
        if self.tensor:
            choices.append("tensor")
        if self.copies:
            choices.append("copy")
        if not choices:
            return False
        if self.rng.choice(choices) == "tensor":
            for bar in self.tensor.pop(0):
                bar.arrive()
        else:
            self.copies.pop(self.rng.randrange(len(self.copies))).arrive()
        self.progress += 1
        return True

    # -- roles (generators: `yield` gives the turn back, like one poll)
    def wait(self, bar, want):
        while not bar.test(want):
            yield

    def planner(self):
        for k in range(len(self.items)):
            if k >= QS:
                yield from self.wait(self.q_free[k % QS], k // QS - 1)
            yield                                        # Q written
            if k >= 2:
                yield from self.wait(self.rec_empty[k % 2], k // 2 - 1)
            self.rec_full[k % 2].arrive()
            self.progress += 1
        n = len(self.items)                              # the record that says "no more work"
        if n >= 2:
            yield from self.wait(self.rec_empty[n % 2], n // 2 - 1)
        self.rec_full[n % 2].arrive()
        self.progress += 1

    def streamer(self):
        t = 0
        for k, n in enumerate(self.items):
            yield from self.wait(self.rec_full[k % 2], k // 2)
            self.rec_empty[k % 2].arrive()
            for _ in range(n):
                if t >= NS:
                    yield from self.wait(self.empty[t % NS], t // NS - 1)
                self.copies.append(self.full[t % NS])    # the tile's copies, landing later
                self.progress += 1
                t += 1
                yield
        n = len(self.items)
        yield from self.wait(self.rec_full[n % 2], n // 2)   # the planner's end record
        # no more work: the next stage, once free, carries the end mark (after
        # the streamer's own copies of the last stages have landed)
        if t >= NS:
            yield from self.wait(self.empty[t % NS], t // NS - 1)
        for u in range(max(0, t - NS), t):
            yield from self.wait(self.full[u % NS], u // NS)
        self.full[t % NS].arrive()
        self.progress += 1

    def qk_issuer(self):
        for t in range(self.T + 1):
            yield from self.wait(self.full[t % NS], t // NS)
            if t == self.T:   # the end mark
                break
            if t >= 2:
                yield from self.wait(self.s_free[t & 1], (t >> 1) - 1)
            self.m_full[t & 1].arrive()
            k, head, tail = self.tiles[t]
            self.commit([self.s_full[t & 1]] + ([self.q_free[k % QS]] if tail == 0 else []))
            self.progress += 1
            yield
        T = self.T
        self.end_tile = T                                 # the PV issuer stops there
        for u in range(max(0, T - 2), T):                 # both metadata buffers read
            yield from self.wait(self.s_free[u & 1], u >> 1)
        self.m_full[0].arrive()                           # end marks (valid = T, item = n)
        self.m_full[1].arrive()
        self.progress += 1

    def softmax(self, g):
        t = g
        while True:
            yield from self.wait(self.m_full[g], t >> 1)
            if t >= self.T:   # the end mark: the group whose turn tile T is tells the output warps
                if t == self.T:
                    k = len(self.items)
                    if k >= IS:
                        yield from self.wait(self.c_free[k % IS], k // IS - 1)
                    self.c_full[k % IS].arrive(2)
                    self.progress += 1
                return
            k, head, tail = self.tiles[t]
            yield from self.wait(self.s_full[g], t >> 1)
            self.s_free[g].arrive()
            first, fin = head < 2, tail < 2
            if not first and self.rng.random() < 0.2:   # the running maximum rose: rescale O
                yield from self.wait(self.pv_done[g], (t - 2) >> 1)
            yield                                        # P^T written into the tile's stage
            if self.fix and t >= 2:
                yield from self.wait(self.pv_done[g], (t - 2) >> 1)
            self.p_full[g].arrive()
            self.progress += 1
            if fin:
                if k >= IS:
                    yield from self.wait(self.c_free[k % IS], k // IS - 1)
                self.c_full[k % IS].arrive(2 if head == 0 and tail == 0 else 1)
                self.progress += 1
            t += 2
            yield

    def pv_issuer(self):
        used = [False] * (2 * IS)
        uses = [0] * (2 * IS)
        for t in range(self.T):
            k, head, tail = self.tiles[t]
            os = (k % IS) * 2 + (t & 1)
            first, lastg = head < 2, tail < 2
            while True:   # poll P, then (a group's first tile of an item) the O slot
                if self.p_full[t & 1].test(t >> 1):
                    if not first or not used[os] or self.ofree[os].test(uses[os] - 1):
                        break
                yield
            bars = [self.pv_done[t & 1], self.empty[t % NS]] + ([self.ofin[os]] if lastg else [])
            self.commit(bars)
            if first:
                used[os] = True
                uses[os] += 1
            self.progress += 1
            yield
        while self.end_tile is None:   # polls P of tile T until the QK issuer sets the end
            self.p_full[self.T & 1].test(self.T >> 1)
            yield

    def output(self):
        reads = [0] * (2 * IS)
        t0 = 0
        for k, n in enumerate(self.items):
            q = k % IS
            yield from self.wait(self.c_full[q], k // IS)
            self.c_free[q].arrive()                       # hand-off slot read and released
            groups = {(t0 + j) & 1 for j in range(n)}
            for g in sorted(groups):
                os = q * 2 + g
                yield from self.wait(self.ofin[os], reads[os])
                reads[os] += 1
                self.ofree[os].arrive()
            for _ in range(self.rng.randrange(4)):      # the rows: a while, sometimes long
                yield
            t0 += n
            self.out_items += 1
            self.progress += 1
        n = len(self.items)
        yield from self.wait(self.c_full[n % IS], n // IS)   # the end mark

    def run(self, max_steps=200000):
        roles = [self.planner(), self.streamer(), self.qk_issuer(), self.softmax(0), self.softmax(1),
                 self.pv_issuer(), self.output()]
        live = list(roles)
        idle = 0
        for _ in range(max_steps):
            if not live and not self.tensor and not self.copies:
                break
            before = self.progress
            if (self.tensor or self.copies) and self.rng.random() < 0.3:
                self.fire()
            elif live:
                r = self.rng.choice(live)
                try:
                    next(r)
                except StopIteration:
                    live.remove(r)
            idle = 0 if self.progress != before else idle + 1
            if idle > 20000:
                raise AssertionError("deadlock: no role can move")
        assert self.out_items == len(self.items), "not every item reached the output warps"


def random_items(rng, n):
    return [rng.choice([1, 1, 1, 2, 2, 3, 4, 16]) for _ in range(n)]


def test_hand_offs_never_alias_a_phase_and_never_deadlock():
    rng = random.Random(2026)
    for _ in range(400):
        Model(random_items(rng, rng.randrange(6, 40)), rng).run()


def test_the_model_catches_p_full_running_two_phases_ahead():
    """Without the wait for PV(t - 2) before the arrive on p_full, a softmax group
    can complete p_full for tile t + 2 while PV(t) still waits for its O slot;
    the model must see that phase alias."""
    rng = random.Random(7)
    caught = 0
    for _ in range(400):
        try:
            Model(random_items(rng, rng.randrange(6, 40)), rng, pv_wait_before_p_full=False).run()
        except Alias:
            caught += 1
        except AssertionError:
            pass
    assert caught > 0
