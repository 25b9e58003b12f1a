"""A randomised CPU model of the prefill / extend kernel's synchronisation
protocol (csrc/prefill_kernel.cu), checked under thousands of random
interleavings: every role of one persistent CTA (TMA producer, e4m3
converters for FP8 caches, one MMA warp and one softmax warpgroup per query
tile, the tensor pipe) runs as a step-wise process over the CTA's sequence of
work items; mbarriers have their hardware semantics (phases, arrival counts,
waits on a phase PARITY only); each MMA warp's tcgen05 operations execute in
issue order, and a commit fires once every earlier operation of the same
issuing warp has completed. The K/V ring, the S / P buffers and every
barrier's phase run on across items; the Q buffer is reloaded per item once
the previous item's S MMAs are done (q_free), and O is reused once the
previous item's epilogue has read it.

Checked: no wait ever passes on a stale phase (the parity matches but the
phase waited for has not completed), no buffer is overwritten before its
reader is done (Q, K/V and e4m3 ring slots, the single S buffer, the two P
buffers, O during a rescale or an epilogue), every role finishes (no
deadlock). The model mirrors the kernel's waits one for one; a change to
either must keep them in step."""
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
    """items: per work item of the CTA, the K/V tiles each query tile reads
    (all zero for an item with no tile, which every role skips)."""

    def __init__(self, rng, qt, fp8, items, stages, stages8):
        self.rng, self.qt, self.fp8 = rng, qt, fp8
        self.items = [list(it) for it in items]
        self.S, self.S8 = stages, stages8
        B = Barrier
        self.q_full = B("q_full", 1)
        self.q_free = B("q_free", qt)
        self.kv_full = [B(f"kv_full{s}", 1) for s in range(stages)]
        self.kv_empty = [B(f"kv_empty{s}", qt) for s in range(stages)]
        self.kv8_full = [B(f"kv8_full{s}", 1) for s in range(stages8)]
        self.kv8_empty = [B(f"kv8_empty{s}", 1) for s in range(stages8)]
        self.s_full = [B(f"s_full{g}", 1) for g in range(qt)]
        self.s_free = [B(f"s_free{g}", 1) for g in range(qt)]
        self.p_full = [[B(f"p_full{g}.{i}", 1) for i in range(2)] for g in range(qt)]
        self.pv_done = [[B(f"pv_done{g}.{i}", 1) for i in range(2)] for g in range(qt)]
        # ring positions: position -> (item, K/V tile within the item)
        self.pos = []
        for k, nkv in enumerate(self.items):
            self.pos += [(k, j) for j in range(max(nkv))]
        # buffer states
        self.Q_item, self.Q_writing = None, False
        self.S_running = [None] * qt       # item of the S MMA in progress (reads Q)
        self.slot = [None] * stages        # ring position held by a bf16 slot
        self.slot8 = [None] * stages8      # ring position held by an e4m3 slot
        self.readers = {}                  # position -> pending MMA reads of its bf16 slot
        self.conv_reading = set()
        self.S_buf = [None] * qt           # S tile index J the S buffer holds
        self.S_read = [True] * qt          # the softmax copied it out
        self.P_buf = [[None, None] for _ in range(qt)]
        self.pv_pending = [set() for _ in range(qt)]   # PV J's issued, not complete
        self.pv_reading_P = [[None, None] for _ in range(qt)]
        self.O_item = [None] * qt          # item whose accumulation O holds
        self.epi_done = [set() for _ in range(qt)]     # items whose epilogue read O
        self.O_reading = [False] * qt
        self.tma = []                      # in-flight copies: (ready_tick, action)
        self.pipe = [[] for _ in range(qt)]            # per MMA warp: ops in issue order
        self.tick = 0

    # ---------------------------------------------------------------- roles
    def producer(self, wait_q_free=True):
        m = self
        kv = qc = 0
        for k, nkv in enumerate(m.items):
            n_kv = max(nkv)
            if n_kv == 0:
                continue
            if qc > 0 and wait_q_free:
                while not m.q_free.ready(qc - 1):
                    yield WAIT
            self._q_overwrite_check()
            m.Q_writing = True

            def qland(k=k):
                self._q_overwrite_check()
                m.Q_item, m.Q_writing = k, False
                m.q_full.arrive()
            m.tma.append((m.tick + m.rng.randint(1, 20), qland))
            qc += 1
            yield
            for j in range(n_kv):
                p = kv + j
                if m.fp8:
                    s, r = p % m.S8, p // m.S8
                    if r > 0:
                        while not m.kv8_empty[s].ready(r - 1):
                            yield WAIT
                    assert m.slot8[s] is None or m.slot8[s] <= p - m.S8
                    assert (p - m.S8) not in m.conv_reading, "e4m3 slot overwritten while read"

                    def land(s=s, p=p):
                        m.slot8[s] = p
                        m.kv8_full[s].arrive()
                    m.tma.append((m.tick + m.rng.randint(1, 30), land))
                else:
                    s, r = p % m.S, p // m.S
                    if r > 0:
                        while not m.kv_empty[s].ready(r - 1):
                            yield WAIT
                    self._check_slot_free(s, p)

                    def land(s=s, p=p):
                        m.slot[s] = p
                        m.readers[p] = self._readers_of(p)
                        m.kv_full[s].arrive()
                    m.tma.append((m.tick + m.rng.randint(1, 30), land))
                yield
            kv += n_kv

    def _q_overwrite_check(self):
        assert all(r is None for r in self.S_running), "Q overwritten while an S MMA reads it"
        for g in range(self.qt):   # queued S MMAs of the item Q still holds
            assert not any(op[0] == "S" and op[2] == self.Q_item for op in self.pipe[g]), \
                "Q overwritten before a queued S MMA read it"

    def _readers_of(self, p):
        k, j = self.pos[p]
        nkv = self.items[k]
        return {(g, kind) for g in range(self.qt) if j < nkv[g] for kind in ("S", "PV")}

    def _check_slot_free(self, s, p):
        old = self.slot[s]
        if old is not None:
            assert not self.readers.get(old), \
                f"slot {s}: position {old} overwritten with reads pending"

    def converter(self):
        m = self
        for p in range(len(m.pos)):
            s8, sb = p % m.S8, p % m.S
            while not m.kv8_full[s8].ready(p // m.S8):
                yield WAIT
            if p >= m.S:
                while not m.kv_empty[sb].ready(p // m.S - 1):
                    yield WAIT
            assert m.slot8[s8] == p
            self._check_slot_free(sb, p)
            m.conv_reading.add(p)
            for _ in range(m.rng.randint(1, 6)):
                yield
            m.conv_reading.discard(p)
            m.slot[sb] = p
            m.readers[p] = self._readers_of(p)
            m.kv8_empty[s8].arrive()
            m.kv_full[sb].arrive()
            yield

    def mma(self, g):
        yield from mma_schedule(self, g)

    def softmax(self, g):
        m = self
        J = 0
        for k, nkv in enumerate(m.items):
            nk = nkv[g]
            if max(nkv) == 0 or nk == 0:
                continue
            for j in range(nk):
                JJ = J + j
                while not m.s_full[g].ready(JJ):
                    yield WAIT
                assert m.S_buf[g] == JJ and not m.S_read[g], "softmax read a stale S"
                m.S_read[g] = True
                m.s_free[g].arrive()
                for _ in range(m.rng.randint(1, 8)):
                    yield
                if j > 0 and m.rng.random() < 0.2:     # the row maximum moved: rescale O
                    while not m.pv_done[g][(JJ - 1) & 1].ready((JJ - 1) >> 1):
                        yield WAIT
                    assert not m.pv_pending[g], "O rescaled while a P*V was in flight"
                    assert m.O_item[g] == k, "O rescaled holding another item"
                # the P buffer's previous reader, P(J-2) V, must be done (covered by s_full)
                assert m.pv_reading_P[g][JJ & 1] is None, "P buffer overwritten while read"
                assert (JJ - 2) not in m.pv_pending[g], "P buffer overwritten before its P*V ran"
                m.P_buf[g][JJ & 1] = JJ
                m.p_full[g][JJ & 1].arrive()
                yield
            J += nk
            yield from self.epilogue(g, k, J)

    def epilogue(self, g, k, J):
        m = self
        while not m.pv_done[g][(J - 1) & 1].ready((J - 1) >> 1):
            yield WAIT
        assert not m.pv_pending[g], "epilogue read O with a P*V in flight"
        assert m.O_item[g] == k, "epilogue read O holding another item"
        m.O_reading[g] = True
        for _ in range(m.rng.randint(1, 6)):
            yield
            assert m.O_item[g] == k and not m.pv_pending[g], "O overwritten during the epilogue"
        m.O_reading[g] = False
        m.epi_done[g].add(k)

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
        kind, J, k, p = op[:4]
        state = getattr(m, "_running", {}).get(g)
        if state is None:     # start: reads and hazards at issue-to-execute
            m.__dict__.setdefault("_running", {})[g] = [m.rng.randint(1, 4)]
            if kind == "S":
                assert not m.Q_writing and m.Q_item == k, "S MMA read a Q holding another item"
                assert m.slot[p % m.S] == p, "S MMA read a K slot holding another tile"
                assert m.S_read[g], "S buffer overwritten before the softmax copied it"
                m.S_running[g] = k
            else:
                assert m.P_buf[g][J & 1] == J, "P*V read a P buffer holding another tile"
                assert m.slot[p % m.S] == p, "P*V read a V slot holding another tile"
                if op[4]:     # first P*V of the item overwrites O
                    prev = m.O_item[g]
                    assert prev is None or (prev in m.epi_done[g] and not m.O_reading[g]), \
                        "O overwritten before the previous item's epilogue read it"
                    m.O_item[g] = k
                else:
                    assert m.O_item[g] == k
                m.pv_pending[g].add(J)
                m.pv_reading_P[g][J & 1] = J
            return True
        state[0] -= 1
        if state[0] > 0:
            return True
        del m._running[g]
        m.pipe[g].pop(0)
        if kind == "S":
            m.S_buf[g], m.S_read[g] = J, False
            m.S_running[g] = None
            m.readers[p].discard((g, "S"))
        else:
            m.pv_pending[g].discard(J)
            m.pv_reading_P[g][J & 1] = None
            m.readers[p].discard((g, "PV"))
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
                f"{b.name}={b.completed}" for b in m.kv_full + m.kv_empty + [m.q_full, m.q_free])
        for g in range(m.qt):
            assert not m.pv_pending[g]
            done = {k for k, nkv in enumerate(m.items) if nkv[g] > 0}
            assert m.epi_done[g] == done, "an item's epilogue did not run"


def mma_schedule(m, g, skip_waits_for_tile=True, wait_s_free=True, q_free_at="last_s",
                 idle_waits_q=True):
    """The MMA warp of query tile g over the CTA's items, as the kernel runs
    it; the keyword arguments plant one mistake each (a wait removed, the
    q_free arrival moved)."""
    kv = J = qc = 0
    for k, nkv in enumerate(m.items):
        n_kv, nkg = max(nkv), nkv[g]
        if n_kv == 0:
            continue
        if nkg > 0 or idle_waits_q:
            while not m.q_full.ready(qc):
                yield WAIT
        qc += 1

        def issue_s(j):
            p, JJ = kv + j, J + j
            while not m.kv_full[p % m.S].ready(p // m.S):
                yield WAIT
            if wait_s_free and JJ >= 1:
                while not m.s_free[g].ready(JJ - 1):
                    yield WAIT
            m.pipe[g].append(("S", JJ, k, p))
            m.pipe[g].append(("commit", m.s_full[g]))
            if q_free_at == "last_s" and j == nkg - 1:   # the item's last read of Q
                m.pipe[g].append(("commit", m.q_free))
            yield

        def issue_pv(i):
            p, JJ = kv + i, J + i
            while not m.p_full[g][JJ & 1].ready(JJ >> 1):
                yield WAIT
            m.pipe[g].append(("PV", JJ, k, p, i == 0))
            m.pipe[g].append(("commit", m.pv_done[g][JJ & 1]))
            m.pipe[g].append(("commit", m.kv_empty[p % m.S]))
            yield

        if not skip_waits_for_tile:  # arrive for unread tiles right away
            for j in range(nkg, n_kv):
                m.kv_empty[(kv + j) % m.S].arrive()
                yield
        if nkg == 0 or q_free_at == "item_start":
            m.q_free.arrive()        # reads nothing of this Q (or: the planted mistake)
        if nkg > 0:
            yield from issue_s(0)
        for j in range(nkg):
            if j + 1 < nkg:
                yield from issue_s(j + 1)
            yield from issue_pv(j)
        if skip_waits_for_tile:
            for j in range(nkg, n_kv):  # tiles this query tile does not read
                p = kv + j
                while not m.kv_full[p % m.S].ready(p // m.S):
                    yield WAIT
                m.kv_empty[p % m.S].arrive()
                yield
        kv += n_kv
        J += nkg


def tile_counts(rng, qt):
    """K/V tiles per query tile as the kernel derives them (the second tile
    of a CTA sees 16 more keys, so at most one more tile; or none if the
    sequence ends inside the first tile)."""
    n0 = rng.randint(1, 12)
    if qt == 1:
        return [n0]
    return [n0, rng.choice([0, n0, n0 + 1])]


def item_list(rng, qt):
    """A persistent CTA's work items: 1 to 5, now and then one with no tile."""
    return [[0] * qt if rng.random() < 0.1 else tile_counts(rng, qt)
            for _ in range(rng.randint(1, 5))]


def rings(qt, fp8):
    return (3 if fp8 else (6 if qt == 1 else 5)), ((6 if qt == 1 else 4) if fp8 else 0)


@pytest.mark.parametrize("qt,fp8", [(1, False), (2, False), (1, True), (2, True)])
def test_protocol_random_interleavings(qt, fp8):
    rng = random.Random(1234 + 10 * qt + fp8)
    stages, stages8 = rings(qt, fp8)
    for trial in range(300):
        nkv = tile_counts(rng, qt)
        Model(random.Random(rng.random()), qt, fp8, [nkv], stages, stages8).run()


@pytest.mark.parametrize("qt,fp8", [(1, False), (2, False), (1, True), (2, True)])
def test_persistent_items_random_interleavings(qt, fp8):
    # several work items per CTA: ring, S / P buffers and barrier phases run on
    rng = random.Random(4321 + 10 * qt + fp8)
    stages, stages8 = rings(qt, fp8)
    for trial in range(250):
        Model(random.Random(rng.random()), qt, fp8, item_list(rng, qt), stages, stages8).run()


def _catches(cls, make_items, trials=400, seed=11):
    rng = random.Random(seed)
    for trial in range(trials):
        try:
            cls(random.Random(rng.random()), 2, False, make_items(rng), 5, 0).run()
        except AssertionError:
            return True
    return False


def _mutant(**kw):
    return type("Mutant", (Model,), {"mma": lambda self, g: mma_schedule(self, g, **kw)})


def test_model_catches_a_missing_wait():
    # Plant a mistake in the model: the softmax skips waiting for S. The model
    # must report it (a stale S read or a parity failure) in some interleaving.
    class Broken(Model):
        def softmax(self, g):
            m = self
            for j in range(m.items[0][g]):
                yield
                assert m.S_buf[g] == j and not m.S_read[g], "softmax read a stale S"
                m.S_read[g] = True
                m.s_free[g].arrive()
                m.P_buf[g][j & 1] = j
                m.p_full[g][j & 1].arrive()
                yield
    assert _catches(Broken, lambda rng: [[4, 5]], trials=200, seed=7)


def _single(rng):
    n = rng.randint(1, 12)
    return [[n, 0] if rng.random() < 0.5 else [n, n + 1]]


@pytest.mark.parametrize("mutation", ["early_skip_arrival", "no_s_free_wait"])
def test_model_catches_planted_mma_mistakes(mutation):
    # An arrival for a tile the query tile does not read, made before that tile
    # has landed, can complete the slot's previous round early and let the
    # producer overwrite a tile the other query tile still reads; an S issued
    # without s_free overwrites S before the softmax copied it.
    cls = _mutant(skip_waits_for_tile=mutation != "early_skip_arrival",
                  wait_s_free=mutation != "no_s_free_wait")
    assert _catches(cls, _single)


def _idle_heavy(rng):
    # items where the second query tile reads nothing, back to back
    return [[rng.randint(2, 8), 0] for _ in range(rng.randint(2, 4))]


@pytest.mark.parametrize("mutation", ["q_free_at_item_start", "idle_arrival_without_q_full"])
def test_model_catches_planted_q_reuse_mistakes(mutation):
    # q_free signalled before the item's S MMAs have read Q, or an idle query
    # tile's arrival made without first seeing this item's Q land (it can then
    # arrive twice within one phase), lets the producer reload Q under a
    # pending S MMA.
    cls = _mutant(q_free_at="item_start" if mutation == "q_free_at_item_start" else "last_s",
                  idle_waits_q=mutation != "idle_arrival_without_q_full")
    assert _catches(cls, _idle_heavy, trials=600)


def test_model_catches_q_reload_without_q_free():
    class Broken(Model):
        def producer(self):
            return Model.producer(self, wait_q_free=False)
    assert _catches(Broken, lambda rng: [tile_counts(rng, 2) for _ in range(3)])


def test_model_catches_o_reuse_before_epilogue():
    # A softmax warpgroup that publishes the P of an item's first tile before
    # its epilogue has read O of the previous item lets that item's first
    # P*V (accumulate off) overwrite O under the epilogue.
    class Reordered(Model):
        def softmax(self, g):
            m = self
            J = 0
            pending = None   # (item, J after it) whose epilogue is deferred
            for k, nkv in enumerate(m.items):
                nk = nkv[g]
                if max(nkv) == 0 or nk == 0:
                    continue
                for j in range(nk):
                    JJ = J + j
                    while not m.s_full[g].ready(JJ):
                        yield WAIT
                    m.S_read[g] = True
                    m.s_free[g].arrive()
                    m.P_buf[g][JJ & 1] = JJ
                    m.p_full[g][JJ & 1].arrive()
                    yield
                    if j == 0 and pending is not None:
                        yield from self.epilogue(g, *pending)
                        pending = None
                J += nk
                pending = (k, J)
            if pending is not None:
                yield from self.epilogue(g, *pending)
    assert _catches(Reordered, lambda rng: [[rng.randint(1, 4)] * 2 for _ in range(3)])


def test_model_reports_a_deadlock():
    # a role that waits forever (a softmax that never takes its S, so the MMA
    # warp never gets s_free) must end the run with the deadlock report
    class Stuck(Model):
        def softmax(self, g):
            while True:
                yield WAIT
    with pytest.raises(AssertionError, match="deadlock"):
        Model.run(Stuck(random.Random(5), 1, False, [[3]], 6, 0))
