"""A randomised CPU model of the prefill / extend kernel's synchronisation
protocol (csrc/prefill_kernel.cu), checked under thousands of random
interleavings: every role of one CTA (TMA producer, e4m3 converters for FP8
caches, one MMA warp and one softmax warpgroup per query tile, the tensor
pipe) runs as a step-wise process; mbarriers have their hardware semantics
(phases, arrival counts, waits on a phase PARITY only); each MMA warp's
tcgen05 operations execute in issue order, and a commit fires once every
earlier operation of the same issuing warp has completed.

Checked: no wait ever passes on a stale phase (the parity matches but the
phase waited for has not completed), no buffer is overwritten before its
reader is done (K/V and e4m3 ring slots, the single S buffer, the two P
buffers, O during a rescale), with an FP8 cache no S MMA reads a Q tile
before its softmax warps have converted it to f16, every role finishes (no
deadlock). The model
mirrors the kernel's waits one for one; a change to either must keep them in
step."""
import random

import pytest

WAIT = "wait"  # yielded by a role that is spinning on a barrier (not progress)


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.completed = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, f"{self.name}: too many arrivals"
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def ready(self, phase):
        """try_wait.parity(phase & 1); asserts it is never fooled by parity."""
        ok = (self.completed & 1) != (phase & 1)
        if ok:
            assert self.completed >= phase + 1, \
                f"{self.name}: parity wait for phase {phase} passed at {self.completed} phases"
        return ok


class Model:
    def __init__(self, rng, qt, fp8, nkv, stages, stages8):
        self.rng, self.qt, self.fp8 = rng, qt, fp8
        self.nkv = nkv                     # K/V tiles per query tile
        self.n_kv = max(nkv)
        self.S, self.S8 = stages, stages8
        B = Barrier
        self.q_full = B("q_full", 1)
        # FP8: the softmax warps of tile g convert its Q rows to f16 in place
        self.q_ready = [B(f"q_ready{g}", 1) for g in range(qt)]
        self.q_f16 = [False] * qt
        self.kv_full = [B(f"kv_full{s}", 1) for s in range(stages)]
        self.kv_empty = [B(f"kv_empty{s}", qt) for s in range(stages)]
        self.kv8_full = [B(f"kv8_full{s}", 1) for s in range(stages8)]
        self.kv8_empty = [B(f"kv8_empty{s}", 1) for s in range(stages8)]
        self.s_full = [B(f"s_full{g}", 1) for g in range(qt)]
        self.s_free = [B(f"s_free{g}", 1) for g in range(qt)]
        self.p_full = [[B(f"p_full{g}.{i}", 1) for i in range(2)] for g in range(qt)]
        self.pv_done = [[B(f"pv_done{g}.{i}", 1) for i in range(2)] for g in range(qt)]
        # buffer states
        self.slot = [None] * stages        # K/V tile held by a bf16 slot
        self.slot8 = [None] * stages8      # tile held by an e4m3 slot
        self.readers = {}                  # tile -> set of pending MMA reads of its bf16 slot
        self.conv_reading = set()
        self.S_buf = [None] * qt           # tile whose S the S buffer holds
        self.S_read = [True] * qt          # the softmax copied it out
        self.P_buf = [[None, None] for _ in range(qt)]
        self.pv_pending = [set() for _ in range(qt)]   # PV tiles issued, not complete
        self.pv_reading_P = [[None, None] for _ in range(qt)]
        self.tma = []                      # in-flight copies: (ready_tick, action)
        self.pipe = [[] for _ in range(qt)]            # per MMA warp: ops in issue order
        self.tick = 0

    # ---------------------------------------------------------------- roles
    def producer(self):
        m = self
        m.tma.append((m.tick + m.rng.randint(1, 20), lambda: m.q_full.arrive()))
        yield
        for j in range(m.n_kv):
            if m.fp8:
                s, r = j % m.S8, j // m.S8
                if r > 0:
                    while not m.kv8_empty[s].ready(r - 1):
                        yield WAIT
                assert m.slot8[s] is None or m.slot8[s] <= j - m.S8
                assert (j - m.S8) not in m.conv_reading, "e4m3 slot overwritten while read"

                def land(s=s, j=j):
                    m.slot8[s] = j
                    m.kv8_full[s].arrive()
                m.tma.append((m.tick + m.rng.randint(1, 30), land))
            else:
                s, r = j % m.S, j // m.S
                if r > 0:
                    while not m.kv_empty[s].ready(r - 1):
                        yield WAIT
                self._check_slot_free(s, j)

                def land(s=s, j=j):
                    m.slot[s] = j
                    m.readers[j] = self._readers_of(j)
                    m.kv_full[s].arrive()
                m.tma.append((m.tick + m.rng.randint(1, 30), land))
            yield

    def _readers_of(self, j):
        return {(g, kind) for g in range(self.qt) if j < self.nkv[g] for kind in ("S", "PV")}

    def _check_slot_free(self, s, j):
        old = self.slot[s]
        if old is not None:
            assert not self.readers.get(old), f"slot {s}: tile {old} overwritten with reads pending"

    def converter(self):
        m = self
        for j in range(m.n_kv):
            s8, sb = j % m.S8, j % m.S
            while not m.kv8_full[s8].ready(j // m.S8):
                yield WAIT
            if j >= m.S:
                while not m.kv_empty[sb].ready(j // m.S - 1):
                    yield WAIT
            assert m.slot8[s8] == j
            self._check_slot_free(sb, j)
            m.conv_reading.add(j)
            for _ in range(m.rng.randint(1, 6)):
                yield
            m.conv_reading.discard(j)
            m.slot[sb] = j
            m.readers[j] = self._readers_of(j)
            m.kv8_empty[s8].arrive()
            m.kv_full[sb].arrive()
            yield

    def q_wait(self, g):
        # the MMA warp's wait for Q: as landed (BF16), or converted (FP8)
        bar = self.q_ready[g] if self.fp8 else self.q_full
        while not bar.ready(0):
            yield WAIT

    def mma(self, g):
        m = self
        nkg = m.nkv[g]
        yield from m.q_wait(g)

        def issue_s(j):
            while not m.kv_full[j % m.S].ready(j // m.S):
                yield WAIT
            if j >= 1:
                while not m.s_free[g].ready(j - 1):
                    yield WAIT
            m.pipe[g].append(("S", j))
            m.pipe[g].append(("commit", m.s_full[g]))
            yield

        def issue_pv(i):
            while not m.p_full[g][i & 1].ready(i >> 1):
                yield WAIT
            m.pipe[g].append(("PV", i))
            m.pipe[g].append(("commit", m.pv_done[g][i & 1]))
            m.pipe[g].append(("commit", m.kv_empty[i % m.S]))
            yield

        if nkg > 0:
            yield from issue_s(0)
        for j in range(nkg):
            if j + 1 < nkg:
                yield from issue_s(j + 1)
            yield from issue_pv(j)
        for j in range(nkg, m.n_kv):  # tiles this query tile does not read
            while not m.kv_full[j % m.S].ready(j // m.S):
                yield WAIT
            m.kv_empty[j % m.S].arrive()
            yield

    def softmax(self, g):
        m = self
        nk = m.nkv[g]
        if m.fp8:  # convert this tile's Q rows once they landed; arrive either way
            if nk > 0:
                while not m.q_full.ready(0):
                    yield WAIT
                for _ in range(m.rng.randint(1, 6)):
                    yield
                m.q_f16[g] = True
            m.q_ready[g].arrive()
            yield
        for j in range(nk):
            while not m.s_full[g].ready(j):
                yield WAIT
            assert m.S_buf[g] == j and not m.S_read[g], "softmax read a stale S"
            m.S_read[g] = True
            m.s_free[g].arrive()
            for _ in range(m.rng.randint(1, 8)):
                yield
            if j > 0 and m.rng.random() < 0.2:     # the row maximum moved: rescale O
                while not m.pv_done[g][(j - 1) & 1].ready((j - 1) >> 1):
                    yield WAIT
                assert not m.pv_pending[g], "O rescaled while a P*V was in flight"
            # the P buffer's previous reader, P(j-2) V, must be done (covered by s_full)
            assert m.pv_reading_P[g][j & 1] is None, "P buffer overwritten while read"
            assert (j - 2) not in m.pv_pending[g], "P buffer overwritten before its P*V ran"
            m.P_buf[g][j & 1] = j
            m.p_full[g][j & 1].arrive()
            yield
        if nk > 0:
            while not m.pv_done[g][(nk - 1) & 1].ready((nk - 1) >> 1):
                yield WAIT
            assert not m.pv_pending[g], "epilogue read O with a P*V in flight"

    # ----------------------------------------------------- the tensor pipe
    def pipe_step(self, g):
        """Run (part of) the oldest operation of MMA warp g; in-order per warp."""
        m = self
        if not m.pipe[g]:
            return False
        op = m.pipe[g][0]
        if op[0] == "commit":
            m.pipe[g].pop(0)
            op[1].arrive()    # everything this warp issued before has completed
            return True
        kind, j = op
        state = getattr(m, "_running", {}).get(g)
        if state is None:     # start: reads and hazards at issue-to-execute
            m.__dict__.setdefault("_running", {})[g] = [m.rng.randint(1, 4)]
            if kind == "S":
                assert m.slot[j % m.S] == j, "S MMA read a K slot holding another tile"
                assert m.q_f16[g] or not m.fp8, "S MMA read a Q tile not yet converted"
                assert m.S_read[g], "S buffer overwritten before the softmax copied it"
            else:
                assert m.P_buf[g][j & 1] == j, "P*V read a P buffer holding another tile"
                assert m.slot[j % m.S] == j, "P*V read a V slot holding another tile"
                m.pv_pending[g].add(j)
                m.pv_reading_P[g][j & 1] = j
            return True
        state[0] -= 1
        if state[0] > 0:
            return True
        del m._running[g]
        m.pipe[g].pop(0)
        if kind == "S":
            m.S_buf[g], m.S_read[g] = j, False
            m.readers[j].discard((g, "S"))
        else:
            m.pv_pending[g].discard(j)
            m.pv_reading_P[g][j & 1] = None
            m.readers[j].discard((g, "PV"))
        return True

    # --------------------------------------------------------------- run
    def run(self):
        m = self
        roles = [self.producer()] + [self.mma(g) for g in range(m.qt)] + \
                [self.softmax(g) for g in range(m.qt)]
        if m.fp8:
            roles.append(self.converter())
        alive = list(roles)
        idle = 0
        while alive or any(m.pipe) or m.tma:
            m.tick += 1
            progressed = False
            # land copies whose time has come
            for item in [t for t in m.tma if t[0] <= m.tick]:
                m.tma.remove(item)
                item[1]()
                progressed = True
            choices = alive + [("pipe", g) for g in range(m.qt) if m.pipe[g]]
            m.rng.shuffle(choices)
            for c in choices[:m.rng.randint(1, len(choices))] if choices else []:
                if isinstance(c, tuple):
                    progressed |= self.pipe_step(c[1])
                else:
                    try:
                        progressed |= next(c) is not WAIT
                    except StopIteration:
                        alive.remove(c)
                        progressed = True
            idle = 0 if progressed or m.tma else idle + 1
            assert idle < 1000, "deadlock: " + ", ".join(
                f"{b.name}={b.completed}" for b in m.kv_full + m.kv_empty)
        for g in range(m.qt):
            assert not m.pv_pending[g]


def tile_counts(rng, qt):
    """K/V tiles per query tile as the kernel derives them (the second tile
    of a CTA sees 16 more keys, so at most one more tile; or none if the
    sequence ends inside the first tile)."""
    n0 = rng.randint(1, 12)
    if qt == 1:
        return [n0]
    return [n0, rng.choice([0, n0, n0 + 1])]


@pytest.mark.parametrize("qt,fp8", [(1, False), (2, False), (1, True), (2, True)])
def test_protocol_random_interleavings(qt, fp8):
    rng = random.Random(1234 + 10 * qt + fp8)
    stages = (4 if fp8 else (6 if qt == 1 else 5))
    stages8 = (4 if qt == 1 else 2) if fp8 else 0
    for trial in range(300):
        nkv = tile_counts(rng, qt)
        Model(random.Random(rng.random()), qt, fp8, nkv, stages, stages8).run()


def test_model_catches_a_missing_wait():
    # Plant a mistake in the model: the softmax skips waiting for S. The model
    # must report it (a stale S read or a parity failure) in some interleaving.
    class Broken(Model):
        def softmax(self, g):
            m = self
            for j in range(m.nkv[g]):
                yield
                assert m.S_buf[g] == j and not m.S_read[g], "softmax read a stale S"
                m.S_read[g] = True
                m.s_free[g].arrive()
                m.P_buf[g][j & 1] = j
                m.p_full[g][j & 1].arrive()
                yield
    rng = random.Random(7)
    caught = False
    for trial in range(200):
        try:
            Broken(random.Random(rng.random()), 2, False, [4, 5], 5, 0).run()
        except AssertionError:
            caught = True
            break
    assert caught


def _mma_with(skip_waits_for_tile=True, wait_s_free=True):
    """The MMA warp's schedule with one of its waits optionally removed."""
    def mma(self, g):
        m = self
        nkg = m.nkv[g]
        yield from m.q_wait(g)

        def issue_s(j):
            while not m.kv_full[j % m.S].ready(j // m.S):
                yield WAIT
            if wait_s_free and j >= 1:
                while not m.s_free[g].ready(j - 1):
                    yield WAIT
            m.pipe[g].append(("S", j))
            m.pipe[g].append(("commit", m.s_full[g]))
            yield

        def issue_pv(i):
            while not m.p_full[g][i & 1].ready(i >> 1):
                yield WAIT
            m.pipe[g].append(("PV", i))
            m.pipe[g].append(("commit", m.pv_done[g][i & 1]))
            m.pipe[g].append(("commit", m.kv_empty[i % m.S]))
            yield

        if not skip_waits_for_tile:  # arrive for unread tiles right away
            for j in range(nkg, m.n_kv):
                m.kv_empty[j % m.S].arrive()
                yield
        if nkg > 0:
            yield from issue_s(0)
        for j in range(nkg):
            if j + 1 < nkg:
                yield from issue_s(j + 1)
            yield from issue_pv(j)
        if skip_waits_for_tile:
            for j in range(nkg, m.n_kv):
                while not m.kv_full[j % m.S].ready(j // m.S):
                    yield WAIT
                m.kv_empty[j % m.S].arrive()
                yield
    return mma


@pytest.mark.parametrize("mutation", ["early_skip_arrival", "no_s_free_wait"])
def test_model_catches_planted_mma_mistakes(mutation):
    # An arrival for a tile the query tile does not read, made before that tile
    # has landed, can complete the slot's previous round early and let the
    # producer overwrite a tile the other query tile still reads; an S issued
    # without s_free overwrites S before the softmax copied it.
    cls = type("Mutant", (Model,), {"mma": _mma_with(
        skip_waits_for_tile=mutation != "early_skip_arrival",
        wait_s_free=mutation != "no_s_free_wait")})
    rng = random.Random(11)
    caught = False
    for trial in range(400):
        n = rng.randint(1, 12)
        nkv = [n, 0] if rng.random() < 0.5 else [n, n + 1]
        try:
            cls(random.Random(rng.random()), 2, False, nkv, 5, 0).run()
        except AssertionError:
            caught = True
            break
    assert caught


def test_model_reports_a_deadlock():
    # a role that waits forever (a softmax that never takes its S, so the MMA
    # warp never gets s_free) must end the run with the deadlock report
    class Stuck(Model):
        def softmax(self, g):
            while True:
                yield WAIT
    with pytest.raises(AssertionError, match="deadlock"):
        Model.run(Stuck(random.Random(5), 1, False, [3], 6, 0))


def test_model_catches_an_unconverted_q_read():
    # with an FP8 cache the MMA warp waiting for the Q copy instead of the
    # softmax warps' conversion lets an S MMA read bf16 Q as f16
    class EarlyQ(Model):
        def q_wait(self, g):
            while not self.q_full.ready(0):
                yield WAIT
    rng = random.Random(13)
    caught = False
    for trial in range(300):
        qt = rng.choice([1, 2])
        try:
            EarlyQ(random.Random(rng.random()), qt, True, tile_counts(rng, qt), 3, 4).run()
        except AssertionError:
            caught = True
            break
    assert caught
