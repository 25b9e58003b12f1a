"""CPU model of the synchronisation protocol of the one-token step kernel
(paged_gqa_decode_hpc_gb300/csrc/step_kernel.cu), run under random
interleavings.

Roles of one CTA: the producer warp (publishes piece descriptors into a
4-slot queue, then issues each unit's copy into a STAGES-deep ring), 8
consumer warps (take a piece's units round-robin, deposit their states into
one shared buffer) and 1 or 2 epilogue warps (taking pieces in turn, read the
8 deposits, hand the buffer back; the kernel runs one). Barriers are modelled as the hardware's
mbarriers: an arrival count per phase and a wait that tests the parity of a
phase only -- it passes when the barrier's completed-phase count has the
other parity, so a waiter two phases ahead passes on a stale phase. Every
wait states the phase it means, and the model asserts that the phase it
passed on is that one. It also asserts that a ring slot is read only while it
holds the waited-for unit, that no deposit is overwritten before the
epilogue read it, that every piece's deposits are read exactly once, and
that nothing deadlocks. Planted mistakes (one deposit barrier shared by both
epilogue warps, a consumer that skips the ring's issued-unit word, a deposit
without waiting for the buffer) are caught.
"""
import random

import pytest

NC, Q = 8, 4


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.completed = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the phase expects"
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def passes(self, parity):
        # try_wait.parity: true once the phase with this parity has completed,
        # i.e. the count of completed phases has the other parity
        return self.completed % 2 != parity


class Violation(AssertionError):
    pass


def wait(bar, phase):
    """Generator: wait for `phase` (>= 0) of `bar` by its parity, as the
    kernel does; asserts that the phase that let it pass is `phase`."""
    while not bar.passes(phase & 1):
        yield
    if bar.completed <= phase:
        raise Violation(f"parity wait for phase {phase} passed with {bar.completed} completed")


def run_model(pieces, stages, seed, plant=None, max_steps=400000, EPI=1):
    rng = random.Random(seed)
    full = [Barrier(1) for _ in range(stages)]
    empty = [Barrier(1) for _ in range(stages)]
    issued = [None] * stages
    slot_unit = [None] * stages      # unit whose copy was issued into the slot
    landed = [False] * stages
    pfull = [Barrier(1) for _ in range(Q)]
    pfree = [Barrier(NC + 1) for _ in range(Q)]
    desc = [None] * Q
    dfull = [Barrier(NC) for _ in range(EPI)]   # piece j on barrier j % EPI
    dfree = Barrier(1)
    shared_dfull = Barrier(NC)
    deposit = [None] * NC            # piece whose state sits in warp w's deposit
    read_pieces = []
    inflight = []                    # copies not yet landed: slot

    starts, g = [], 0
    for n in pieces:
        starts.append(g)
        g += n
    items = list(range(len(pieces))) + [-1] * EPI   # -1: end marker

    def producer():
        gg = 0
        for j, it in enumerate(items):
            qs = j % Q
            if j >= Q:
                yield from wait(pfree[qs], j // Q - 1)
            desc[qs] = (it, gg if it >= 0 else 0)
            pfull[qs].arrive()
            if it < 0:
                continue
            for _ in range(pieces[it]):
                s = gg % stages
                if gg >= stages:
                    yield from wait(empty[s], gg // stages - 1)
                slot_unit[s] = gg
                landed[s] = False
                issued[s] = gg
                inflight.append(s)
                gg += 1
                yield

    def consumer(w):
        j = 0
        while True:
            qs = j % Q
            yield from wait(pfull[qs], j // Q)
            it, g0 = desc[qs]
            pfree[qs].arrive()
            if it < 0:
                return
            n = pieces[it]
            rot = (it * 3) % NC  # any fixed rotation per piece
            for i in range((w - rot) % NC, n, NC):
                gu = g0 + i
                s = gu % stages
                if plant != "no_issued_word":
                    while issued[s] != gu:
                        yield
                yield from wait(full[s], gu // stages)
                if slot_unit[s] != gu or not landed[s]:
                    raise Violation(f"warp {w} read slot {s} holding {slot_unit[s]} for unit {gu}")
                yield  # compute
                empty[s].arrive()
            if plant != "deposit_without_wait" and j > 0:
                yield from wait(dfree, j - 1)
            if deposit[w] is not None:
                raise Violation(f"warp {w} overwrote the unread deposit of piece {deposit[w]}")
            deposit[w] = it
            if plant == "one_deposit_barrier":
                shared_dfull.arrive()
            else:
                dfull[j % EPI].arrive()
            j += 1

    def epilogue(e):
        j = e
        while True:
            qs = j % Q
            yield from wait(pfull[qs], j // Q)
            it, _ = desc[qs]
            pfree[qs].arrive()
            if it < 0:
                return
            if plant == "one_deposit_barrier":
                # a single barrier shared by both epilogue warps: a warp can be
                # two phases ahead of it
                yield from wait(shared_dfull, j)
            else:
                yield from wait(dfull[j % EPI], j // EPI)
            for w in range(NC):
                if deposit[w] != it:
                    raise Violation(f"epilogue {e} read deposit {deposit[w]} of warp {w} for piece {it}")
                deposit[w] = None
            read_pieces.append(it)
            yield
            dfree.arrive()
            j += EPI

    roles = [producer()] + [consumer(w) for w in range(NC)] + [epilogue(e) for e in range(EPI)]
    live = list(range(len(roles)))
    steps = 0
    while live:
        steps += 1
        if steps > max_steps:
            raise Violation("deadlock: no role finished within the step budget")
        # a copy in flight lands at a random moment
        if inflight and rng.random() < 0.3:
            s = inflight.pop(rng.randrange(len(inflight)))
            landed[s] = True
            full[s].arrive()
        k = rng.choice(live)
        try:
            next(roles[k])
        except StopIteration:
            live.remove(k)
    while inflight:
        s = inflight.pop()
        landed[s] = True
        full[s].arrive()
    assert sorted(read_pieces) == list(range(len(pieces))), "every piece combined exactly once"


def _pieces(rng):
    return [rng.choice([1, 1, 2, 3, 7, 8, 9, rng.randint(1, 40)]) for _ in range(rng.randint(1, 12))]


@pytest.mark.parametrize("epi", [1, 2])
@pytest.mark.parametrize("stages", [5, 10, 11])
def test_protocol_random_interleavings(stages, epi):
    rng = random.Random(stages)
    for seed in range(150):
        run_model(_pieces(rng), stages, seed, EPI=epi)


@pytest.mark.parametrize("plant", ["one_deposit_barrier", "no_issued_word",
                                   "deposit_without_wait"])
def test_planted_mistakes_are_caught(plant):
    rng = random.Random(11)
    with pytest.raises(Violation):
        for seed in range(300):
            run_model(_pieces(rng), 5, seed, plant=plant, EPI=2)
