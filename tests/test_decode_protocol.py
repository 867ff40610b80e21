"""Models of the tensor-core kernels' hand-offs (decode with 16-bit and 8-bit
caches, prefill), run on the CPU under random schedules.

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


# ---------------------------------------------------------------- 8-bit caches

ND = 4       # tile descriptors in flight (planner -> copy warp)
NRH = 2      # raw half-tile slots per half
IS8 = 2      # items in flight between softmax and output warps
QS8 = 2      # Q slots


class Model8:
    """The 8-bit cache's roles: the planner (items, Q, per-tile descriptors), the
    copy warp (each tile's chunks into a slot of both halves' raw rings), the
    converter warps of each half (raw -> operands, then the stage's `full`), the
    event-driven MMA issuer (QK and PV from one lane), one softmax group, the
    output warps."""

    def __init__(self, items, rng, drain_before_end_mark=True):
        self.rng = rng
        self.items = items
        self.tiles = []
        for k, n in enumerate(items):
            for j in range(n):
                self.tiles.append((k, j, n - 1 - j, rng.random() < 0.7))   # (item, head, tail, half 1 has bytes)
        self.T = len(self.tiles)
        self.drain_first = drain_before_end_mark
        b = Bar
        self.desc_full = [b(f"desc_full[{i}]", 1) for i in range(ND)]
        self.desc_empty = [b(f"desc_empty[{i}]", 1) for i in range(ND)]
        self.raw_full = [b(f"raw_full[{i}]", 1) for i in range(2 * NRH)]
        self.raw_empty = [b(f"raw_empty[{i}]", 1) for i in range(2 * NRH)]
        self.full = [b(f"full[{i}]", 2) for i in range(NS)]          # both halves' converters
        self.empty = [b(f"empty[{i}]", 1) for i in range(NS)]
        self.s_full = [b(f"s_full[{i}]", 1) for i in range(2)]
        self.s_free = [b(f"s_free[{i}]", 1) for i in range(2)]
        self.p_full = [b(f"p_full[{i}]", 1) for i in range(2)]
        self.pv_done = [b(f"pv_done[{i}]", 1) for i in range(2)]
        self.q_free = [b(f"q_free[{i}]", 1) for i in range(QS8)]
        self.c_full = [b(f"c_full[{i}]", 1) for i in range(IS8)]
        self.c_free = [b(f"c_free[{i}]", 1) for i in range(IS8)]
        self.ofin = [b(f"ofin[{i}]", 1) for i in range(IS8)]
        self.ofree = [b(f"ofree[{i}]", 1) for i in range(IS8)]
        self.tensor, self.copies = [], []
        self.progress = 0
        self.out_items = 0

    commit = Model.commit
    fire = Model.fire
    wait = Model.wait

    def planner(self):
        tile = 0
        for k, n in enumerate(self.items):
            if k >= QS8:
                yield from self.wait(self.q_free[k % QS8], k // QS8 - 1)
            yield                                              # Q written
            for _ in range(n):
                if tile >= ND:
                    yield from self.wait(self.desc_empty[tile % ND], tile // ND - 1)
                self.desc_full[tile % ND].arrive()
                self.progress += 1
                tile += 1
                yield
        if tile >= ND:                                         # the end descriptor
            yield from self.wait(self.desc_empty[tile % ND], tile // ND - 1)
        self.desc_full[tile % ND].arrive()
        self.progress += 1

    def copy_warp(self):
        for tile in range(self.T + 1):
            yield from self.wait(self.desc_full[tile % ND], tile // ND)
            r0, r1 = tile % NRH, NRH + tile % NRH
            if tile >= NRH:
                yield from self.wait(self.raw_empty[r0], tile // NRH - 1)
                yield from self.wait(self.raw_empty[r1], tile // NRH - 1)
            if tile == self.T:   # no more work: the mark into both halves, after the own copies landed
                drain = [(h * NRH + t % NRH, t // NRH) for h in (0, 1) for t in range(max(0, tile - NRH), tile)]
                if not self.drain_first:
                    self.raw_full[r0].arrive()
                    self.raw_full[r1].arrive()
                for r, ph in drain:
                    yield from self.wait(self.raw_full[r], ph)
                if self.drain_first:
                    self.raw_full[r0].arrive()
                    self.raw_full[r1].arrive()
                self.progress += 1
                return
            self.copies.append(self.raw_full[r0])               # half 0 always has bytes
            if self.tiles[tile][3]:
                self.copies.append(self.raw_full[r1])
            else:
                self.raw_full[r1].arrive()                       # expect_tx(0): the arrive completes it
            self.desc_empty[tile % ND].arrive()
            self.progress += 1
            yield

    def converter(self, h):
        for t in range(self.T + 1):
            r = h * NRH + t % NRH
            yield from self.wait(self.raw_full[r], t // NRH)
            if t >= NS:
                yield from self.wait(self.empty[t % NS], t // NS - 1)
            yield                                              # K into TMEM, V into the stage
            self.raw_empty[r].arrive()
            self.full[t % NS].arrive()
            self.progress += 1
            if t == self.T:
                return

    def mma_issuer(self):
        qk = pv = 0
        end = None
        used = [False] * IS8
        uses = [0] * IS8
        while end is None or pv < end:
            if end is None and self.full[qk % NS].test(qk // NS):
                if qk == self.T:
                    end = qk
                elif qk < 2 or self.s_free[qk & 1].test((qk >> 1) - 1):
                    k, head, tail, _ = self.tiles[qk]
                    self.commit([self.s_full[qk & 1]] + ([self.q_free[k % QS8]] if tail == 0 else []))
                    qk += 1
                    self.progress += 1
            if pv < qk and self.p_full[pv & 1].test(pv >> 1):
                k, head, tail, _ = self.tiles[pv]
                os = k % IS8
                first = head == 0
                if not first or not used[os] or self.ofree[os].test(uses[os] - 1):
                    self.commit([self.pv_done[pv & 1], self.empty[pv % NS]] + ([self.ofin[os]] if tail == 0 else []))
                    if first:
                        used[os] = True
                        uses[os] += 1
                    pv += 1
                    self.progress += 1
            yield

    def softmax(self):
        for t in range(self.T + 1):
            yield from self.wait(self.full[t % NS], t // NS)
            if t == self.T:   # the end mark
                n = len(self.items)
                if n >= IS8:
                    yield from self.wait(self.c_free[n % IS8], n // IS8 - 1)
                self.c_full[n % IS8].arrive()
                self.progress += 1
                return
            k, head, tail, _ = self.tiles[t]
            yield from self.wait(self.s_full[t & 1], t >> 1)
            self.s_free[t & 1].arrive()
            if head > 0 and self.rng.random() < 0.3:            # the running maximum rose: rescale O
                yield from self.wait(self.pv_done[(t - 1) & 1], (t - 1) >> 1)
            if t >= 2:                                         # the P^T buffer, last read by PV(t - 2)
                yield from self.wait(self.pv_done[t & 1], (t - 2) >> 1)
            yield                                              # P^T written
            self.p_full[t & 1].arrive()
            self.progress += 1
            if tail == 0:
                if k >= IS8:
                    yield from self.wait(self.c_free[k % IS8], k // IS8 - 1)
                self.c_full[k % IS8].arrive()
                self.progress += 1
            yield

    def output(self):
        for k in range(len(self.items)):
            q = k % IS8
            yield from self.wait(self.c_full[q], k // IS8)
            self.c_free[q].arrive()
            yield from self.wait(self.ofin[q], k // IS8)
            self.ofree[q].arrive()
            for _ in range(self.rng.randrange(4)):
                yield
            self.out_items += 1
            self.progress += 1
        n = len(self.items)
        yield from self.wait(self.c_full[n % IS8], n // IS8)

    def run(self, max_steps=200000):
        roles = [self.planner(), self.copy_warp(), self.converter(0), self.converter(1), self.mma_issuer(),
                 self.softmax(), self.output()]
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


def test_8bit_hand_offs_never_alias_a_phase_and_never_deadlock():
    rng = random.Random(2027)
    for _ in range(400):
        Model8(random_items(rng, rng.randrange(1, 40)), rng).run()


def test_the_model_catches_the_copy_warp_draining_after_its_end_mark():
    """The copy warp once drained its copies after posting its end mark into the
    raw slots; the drain's wait on a slot then named the mark's phase by the
    same parity.  The model must see that alias."""
    rng = random.Random(8)
    caught = 0
    for _ in range(200):
        try:
            Model8(random_items(rng, rng.randrange(1, 40)), rng, drain_before_end_mark=False).run()
        except Alias:
            caught += 1
        except AssertionError:
            pass
    assert caught > 0


# ---------------------------------------------------------------- prefill

class ModelPrefill:
    """The prefill kernel's roles for one query tile: the producer (KV tiles into
    two stages), the event-driven MMA issuer (QK(j) only once PV(j - 2) has been
    issued: S(j) lands in the TMEM columns that held P(j - 2); with two stages the
    refill of tile j's stage already waits for PV(j - 2), so this is belt and
    braces), the softmax warps (one actor)."""

    def __init__(self, n_kv, rng, producer_waits_empty=True):
        self.rng, self.n = rng, n_kv
        self.wait_empty = producer_waits_empty
        b = Bar
        self.full = [b(f"full[{i}]", 1) for i in range(2)]
        self.empty = [b(f"empty[{i}]", 1) for i in range(2)]
        self.s_full = [b(f"s_full[{i}]", 1) for i in range(2)]
        self.s_free = [b(f"s_free[{i}]", 1) for i in range(2)]
        self.p_full = [b(f"p_full[{i}]", 1) for i in range(2)]
        self.pv_done = [b(f"pv_done[{i}]", 1) for i in range(2)]
        self.tensor, self.copies = [], []
        self.progress = 0
        self.done = False
        self.partial = [rng.random() < 0.5 for _ in range(n_kv)]   # a tile with a ragged end

    commit = Model.commit
    fire = Model.fire
    wait = Model.wait

    def producer(self):
        for j in range(self.n):
            if j >= 2 and self.wait_empty:
                yield from self.wait(self.empty[j & 1], (j >> 1) - 1)
            self.copies.append(self.full[j & 1])
            self.progress += 1
            yield
        for j in range(max(0, self.n - 2), self.n):   # its own copies landed before the CTA ends
            yield from self.wait(self.full[j & 1], j >> 1)

    def mma_issuer(self):
        qk = pv = 0
        while pv < self.n:
            if qk < self.n and pv >= qk - 1:
                if self.full[qk & 1].test(qk >> 1) and (qk < 2 or self.s_free[qk & 1].test((qk >> 1) - 1)):
                    self.commit([self.s_full[qk & 1]])
                    qk += 1
                    self.progress += 1
            if pv < qk and self.p_full[pv & 1].test(pv >> 1):
                self.commit([self.pv_done[pv & 1], self.empty[pv & 1]])
                pv += 1
                self.progress += 1
            yield

    def softmax(self):
        for j in range(self.n):
            yield from self.wait(self.s_full[j & 1], j >> 1)
            self.s_free[j & 1].arrive()
            if j >= 1 and self.rng.random() < 0.3:           # the row maximum rose: rescale O
                yield from self.wait(self.pv_done[(j - 1) & 1], (j - 1) >> 1)
            yield                                            # P into TMEM
            if self.partial[j]:                              # zero V rows past the tile's end
                yield from self.wait(self.full[j & 1], j >> 1)
            self.p_full[j & 1].arrive()
            self.progress += 1
            yield
        if self.n:
            yield from self.wait(self.pv_done[(self.n - 1) & 1], (self.n - 1) >> 1)
        self.done = True
        self.progress += 1

    def run(self, max_steps=100000):
        live = [self.producer(), self.mma_issuer(), self.softmax()]
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
        assert self.done


def test_prefill_hand_offs_never_alias_a_phase_and_never_deadlock():
    rng = random.Random(2028)
    for _ in range(600):
        ModelPrefill(rng.randrange(0, 40), rng).run()


def test_the_model_catches_a_stage_refilled_before_its_pv_in_prefill():
    """A producer that refills a stage without waiting for the PV that last read
    it lets the stage's `full` run two phases ahead of the MMA issuer."""
    rng = random.Random(9)
    caught = 0
    for _ in range(400):
        try:
            ModelPrefill(rng.randrange(4, 40), rng, producer_waits_empty=False).run()
        except Alias:
            caught += 1
        except AssertionError:
            pass
    assert caught > 0
