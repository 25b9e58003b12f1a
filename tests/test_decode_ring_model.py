"""A randomised CPU model of the decode attention kernel's K/V ring
(csrc/attn_kernel.cu): one producer warp issues (tile, KV head) units in
order into STAGES slots; each unit is consumed by the q_len warps of its
(head, tile phase); a slot is refilled once all of them have arrived on its
empty barrier. mbarriers wait on a phase PARITY only, which is why a consumer
first waits until the slot's "issued unit" word names its own unit: a warp can
reach round r of a slot while the slot's barrier has completed only round
r - 1 (in flight) or r - 2, and the parity alone would let it through. The
model checks that no wait passes on a stale phase, no consumer reads a slot
that holds another unit, no slot is refilled before its consumers are done,
and nothing deadlocks; with the issued-word wait removed it must fail."""
import random

import pytest

WAIT = "wait"  # yielded by a role that is spinning on a barrier (not progress)


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.completed = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def ready(self, parity, phase=None):
        ok = (self.completed & 1) != (parity & 1)
        if ok and phase is not None:
            assert self.completed >= phase + 1, \
                f"{self.name}: parity wait for phase {phase} passed at {self.completed} phases"
        return ok


class Ring:
    def __init__(self, rng, stages, hpass, q_len, tph, units, check_issued=True):
        self.rng, self.S = rng, stages
        self.hpass, self.q_len, self.tph, self.N = hpass, q_len, tph, units
        self.check_issued = check_issued
        self.full = [Barrier(f"full{s}", 1) for s in range(stages)]
        self.empty = [Barrier(f"empty{s}", q_len) for s in range(stages)]
        self.issued = [None] * stages     # the issued-unit word of each slot
        self.data = [None] * stages       # unit whose tile has landed in the slot
        self.readers = {}                 # unit -> consumers still to arrive
        self.inflight = []

    def consumers(self, g):
        """Warps consuming unit g = i * hpass + hl: same head hl, tile phase
        i mod tph, every query token."""
        i, hl = divmod(g, self.hpass)
        ph = i % self.tph
        return [hl + self.hpass * (tok + self.q_len * ph) for tok in range(self.q_len)]

    def producer(self):
        for g in range(self.N):
            slot, par = g % self.S, ((g // self.S) & 1) ^ 1
            while not self.empty[slot].ready(par, phase=g // self.S - 1 if g >= self.S else None):
                yield WAIT
            old = g - self.S
            assert old < 0 or not self.readers.get(old), "slot refilled before its consumers"
            self.readers[g] = set(self.consumers(g))

            def land(slot=slot, g=g):
                self.data[slot] = g
                self.full[slot].arrive()
            self.inflight.append((self.rng.randint(1, 25), land))
            self.issued[slot] = g
            yield

    def consumer(self, w):
        mine = [g for g in range(self.N) if w in self.consumers(g)]
        for g in mine:
            slot = g % self.S
            if self.check_issued:
                while self.issued[slot] != g:
                    yield WAIT
            while not self.full[slot].ready((g // self.S) & 1, phase=g // self.S):
                yield WAIT
            assert self.data[slot] == g, "consumer read a slot holding another unit"
            for _ in range(self.rng.randint(0, 4)):
                yield
            assert self.data[slot] == g, "slot overwritten while being read"
            self.readers[g].discard(w)
            self.empty[slot].arrive()
            yield

    def run(self):
        nc = self.hpass * self.q_len * self.tph
        roles = [self.producer()] + [self.consumer(w) for w in range(nc)]
        idle = 0
        while roles or self.inflight:
            progressed = False
            nxt = []
            for t, fn in self.inflight:
                if t <= 1:
                    fn()
                    progressed = True
                else:
                    nxt.append((t - 1, fn))
            self.inflight = nxt
            self.rng.shuffle(roles)
            for r in list(roles[: self.rng.randint(1, len(roles))] if roles else []):
                try:
                    progressed |= next(r) is not WAIT
                except StopIteration:
                    roles.remove(r)
                    progressed = True
            idle = 0 if progressed or self.inflight else idle + 1
            assert idle < 500, "deadlock"


# warp layouts of the kernel (8 consumer warps): hpass KV heads per pass x
# q_len query tokens x tph tile phases
LAYOUTS = [(8, 1, 1), (4, 2, 1), (2, 4, 1), (1, 8, 1), (4, 1, 2), (1, 1, 8), (2, 2, 2), (1, 2, 4)]


@pytest.mark.parametrize("hpass,q_len,tph", LAYOUTS)
@pytest.mark.parametrize("stages", [5, 6, 10, 12])
def test_ring_random_interleavings(hpass, q_len, tph, stages):
    rng = random.Random(hash((hpass, q_len, tph, stages)) & 0xFFFF)
    for trial in range(40):
        units = rng.randint(1, 80)
        Ring(random.Random(rng.random()), stages, hpass, q_len, tph, units).run()


def test_parity_alone_is_not_enough():
    # Without the issued-unit wait a consumer can pass the parity check of a
    # round that is still in flight (the bug the issued word fixed).
    rng = random.Random(3)
    caught = False
    for trial in range(300):
        try:
            Ring(random.Random(rng.random()), 6, 1, 1, 8, 60, check_issued=False).run()
        except AssertionError:
            caught = True
            break
    assert caught


def test_ring_model_reports_a_deadlock():
    # a consumer waiting for a unit the producer never issues must end the
    # run with the deadlock report, not spin forever
    class Stuck(Ring):
        def consumer(self, w):
            while self.issued[0] != -1:
                yield WAIT
    with pytest.raises(AssertionError, match="deadlock"):
        Stuck(random.Random(1), 6, 8, 1, 1, 4).run()
