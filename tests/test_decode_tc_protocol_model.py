"""A randomised CPU model of the tensor-core multi-token decode kernel's
synchronisation protocol (csrc/decode_tc_kernel.cu), checked under thousands
of random interleavings. One CTA walks a list of segments (a sequence's tile
range each); its roles (TMA producer, e4m3 converters for FP8 caches, the
MMA warp, the softmax warps -- one holding query rows and one holding only
padding rows, which keeps the barrier counts without work -- and the
in-order tensor pipe) run as step-wise processes; mbarriers have their hardware semantics (phases, arrival counts,
waits on a phase PARITY only); a commit fires once every earlier operation
of the issuing warp has completed.

Checked, across segment boundaries: no wait passes on a stale phase, no
buffer is overwritten before its reader is done (the two Q slots, K/V and
e4m3 ring slots, the single S buffer, the two P buffers), no P V reads a P
buffer that its softmax warps have not all written, with an FP8
cache no S MMA reads a Q slot before the softmax warps converted it to f16
for its segment and no Q slot is reloaded while it is being converted, the
first P V of a
segment does not overwrite O before the previous segment's epilogue read it
(the kernel has no barrier for this: that P V waits for P of the segment's
first tile, which the softmax warps write after their epilogue), each
epilogue reads an O holding exactly its own segment's P V products, and
every role finishes. The model mirrors the kernel's waits one for one; a
change to either must keep them in step."""
import random

import pytest

WAIT = "wait"  # yielded by a role that is spinning on a barrier (not progress)
NSM = 2        # softmax roles: 0 holds query rows, 1 only padding rows


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
    def __init__(self, rng, fp8, segs, stages, stages8, rescale_p=0.2):
        self.rng, self.fp8, self.segs = rng, fp8, segs
        self.S, self.S8 = stages, stages8
        self.rescale_p = rescale_p
        B = Barrier
        self.q_full = [B(f"q_full{i}", 1) for i in range(2)]
        self.q_empty = [B(f"q_empty{i}", 1) for i in range(2)]
        # FP8: the softmax warps convert a segment's Q slot to f16 in place
        self.q_ready = [B(f"q_ready{i}", NSM) for i in range(2)]
        self.q_conv = [None, None]          # segment whose Q a slot holds as f16
        self.q_converting = [False, False]
        self.kv_full = [B(f"kv_full{s}", 1) for s in range(stages)]
        self.kv_empty = [B(f"kv_empty{s}", 1) for s in range(stages)]
        self.kv8_full = [B(f"kv8_full{s}", 1) for s in range(stages8)]
        self.kv8_empty = [B(f"kv8_empty{s}", 1) for s in range(stages8)]
        self.s_full, self.s_free = B("s_full", 1), B("s_free", NSM)
        self.p_full = [B(f"p_full{i}", NSM) for i in range(2)]
        self.pv_done = [B(f"pv_done{i}", 1) for i in range(2)]
        # tile g of the CTA's stream belongs to segment seg_of[g]
        self.seg_of = [k for k, n in enumerate(segs) for _ in range(n)]
        self.first = [sum(segs[:k]) for k in range(len(segs))]
        self.G = sum(segs)
        # buffer states
        self.q_slot = [None, None]         # segment whose Q a slot holds
        self.q_reads = [0, 0]              # S MMAs issued on a slot, not complete
        self.slot = [None] * stages
        self.slot8 = [None] * stages8
        self.readers = {}                  # tile -> pending MMA reads of its bf16 slot
        self.conv_reading = set()
        self.S_buf, self.S_read_by = None, set(range(NSM))  # S's tile, roles that copied it
        self.P_buf = [None, None]
        self.pv_pending = set()
        self.pv_reading_P = [None, None]
        self.O_seg, self.O_count = None, 0   # segment whose P V products O holds, and how many
        self.O_reading = None                # segment whose epilogue is reading O
        self.tma = []
        self.pipe = []
        self.running = None
        self.epilogues = 0
        self.tick = 0

    # ---------------------------------------------------------------- roles
    def producer(self):
        m = self
        g = 0
        for k, n in enumerate(m.segs):
            if k >= 2:
                while not m.q_empty[k & 1].ready((k >> 1) - 1):
                    yield WAIT
            assert m.q_reads[k & 1] == 0, "Q slot overwritten while an S MMA reads it"
            assert not m.q_converting[k & 1], "Q slot overwritten while being converted"

            def land_q(k=k):
                m.q_slot[k & 1] = k
                m.q_conv[k & 1] = None
                m.q_full[k & 1].arrive()
            m.tma.append((m.tick + m.rng.randint(1, 20), land_q))
            yield
            for _ in range(n):
                if m.fp8:
                    s, r = g % m.S8, g // m.S8
                    if r > 0:
                        while not m.kv8_empty[s].ready(r - 1):
                            yield WAIT
                    assert (g - m.S8) not in m.conv_reading, "e4m3 slot overwritten while read"

                    def land(s=s, g=g):
                        m.slot8[s] = g
                        m.kv8_full[s].arrive()
                    m.tma.append((m.tick + m.rng.randint(1, 30), land))
                else:
                    s, r = g % m.S, g // m.S
                    if r > 0:
                        while not m.kv_empty[s].ready(r - 1):
                            yield WAIT
                    self._check_slot_free(s)

                    def land(s=s, g=g):
                        m.slot[s] = g
                        m.readers[g] = {"S", "PV"}
                        m.kv_full[s].arrive()
                    m.tma.append((m.tick + m.rng.randint(1, 30), land))
                g += 1
                yield

    def _check_slot_free(self, s):
        old = self.slot[s]
        if old is not None:
            assert not self.readers.get(old), f"slot {s}: tile {old} overwritten with reads pending"

    def converter(self):
        m = self
        for g in range(m.G):
            s8, sb = g % m.S8, g % m.S
            while not m.kv8_full[s8].ready(g // m.S8):
                yield WAIT
            if g >= m.S:
                while not m.kv_empty[sb].ready(g // m.S - 1):
                    yield WAIT
            assert m.slot8[s8] == g
            self._check_slot_free(sb)
            m.conv_reading.add(g)
            for _ in range(m.rng.randint(1, 6)):
                yield
            m.conv_reading.discard(g)
            m.slot[sb] = g
            m.readers[g] = {"S", "PV"}
            m.kv8_empty[s8].arrive()
            m.kv_full[sb].arrive()
            yield

    def issue_s(self, g, k, q_release):
        m = self
        while not m.kv_full[g % m.S].ready(g // m.S):
            yield WAIT
        if g >= 1:
            while not m.s_free.ready(g - 1):
                yield WAIT
        m.pipe.append(("S", g, k))
        m.pipe.append(("commit", m.s_full))
        if q_release is not None:
            m.pipe.append(("commit", m.q_empty[q_release]))
        yield

    def issue_pv(self, g, k, acc):
        m = self
        while not m.p_full[g & 1].ready(g >> 1):
            yield WAIT
        m.pipe.append(("PV", g, k, acc))
        m.pipe.append(("commit", m.pv_done[g & 1]))
        m.pipe.append(("commit", m.kv_empty[g % m.S]))
        yield

    def q_wait(self, k):
        # the MMA warp's wait for a segment's Q: as landed (BF16) or converted (FP8)
        bar = (self.q_ready if self.fp8 else self.q_full)[k & 1]
        while not bar.ready(k >> 1):
            yield WAIT

    def mma(self):
        m = self
        G = 0
        for k, n in enumerate(m.segs):
            yield from m.q_wait(k)
            yield from m.issue_s(G, k, (k & 1) if n == 1 else None)
            for j in range(n):
                if j + 1 < n:
                    yield from m.issue_s(G + j + 1, k, (k & 1) if j + 2 == n else None)
                yield from m.issue_pv(G + j, k, j > 0)
            G += n

    def softmax(self, role=0):
        m = self
        live = role == 0
        G = 0
        for k, n in enumerate(m.segs):
            if m.fp8:  # convert this segment's Q rows once they landed
                while not m.q_full[k & 1].ready(k >> 1):
                    yield WAIT
                assert m.q_slot[k & 1] == k, "converted a Q slot holding another segment"
                if live:
                    m.q_converting[k & 1] = True
                    for _ in range(m.rng.randint(1, 5)):
                        yield
                    m.q_converting[k & 1] = False
                    m.q_conv[k & 1] = k
                m.q_ready[k & 1].arrive()
                yield
            for j in range(n):
                g = G + j
                while not m.s_full.ready(g):
                    yield WAIT
                assert m.S_buf == g and role not in m.S_read_by, "softmax read a stale S"
                m.S_read_by.add(role)
                m.s_free.arrive()
                if not live:  # padding rows: the barrier counts only
                    yield
                    m.p_full[g & 1].arrive()
                    yield
                    continue
                for _ in range(m.rng.randint(1, 8)):
                    yield
                if j > 0 and m.rng.random() < m.rescale_p:  # the row maximum moved
                    while not m.pv_done[(g - 1) & 1].ready((g - 1) >> 1):
                        yield WAIT
                    assert not m.pv_pending, "O rescaled while a P*V was in flight"
                    assert m.O_seg == k, "O rescaled while holding another segment"
                assert m.pv_reading_P[g & 1] is None, "P buffer overwritten while read"
                assert (g - 2) not in m.pv_pending, "P buffer overwritten before its P*V ran"
                m.P_buf[g & 1] = g
                m.p_full[g & 1].arrive()
                yield
            yield from m.wait_last_pv(G + n - 1)
            if not live:
                G += n
                continue
            assert not m.pv_pending, "epilogue read O with a P*V in flight"
            assert m.O_seg == k and m.O_count == n, \
                f"epilogue of segment {k} read O of segment {m.O_seg} ({m.O_count} of {n} tiles)"
            m.O_reading = k
            for _ in range(m.rng.randint(1, 6)):
                yield
            m.O_reading = None
            m.O_count = -1  # read: the next segment's first P V may overwrite it
            m.epilogues += 1
            G += n

    def wait_last_pv(self, gl):
        while not self.pv_done[gl & 1].ready(gl >> 1):
            yield WAIT

    # ----------------------------------------------------- the tensor pipe
    def pipe_step(self):
        m = self
        if not m.pipe:
            return False
        op = m.pipe[0]
        if op[0] == "commit":
            m.pipe.pop(0)
            op[1].arrive()
            return True
        if m.running is None:  # start: operand reads and hazards
            m.running = [m.rng.randint(1, 4)]
            if op[0] == "S":
                _, g, k = op
                assert m.slot[g % m.S] == g, "S MMA read a K slot holding another tile"
                assert m.q_slot[k & 1] == k, "S MMA read a Q slot holding another segment"
                assert not m.fp8 or m.q_conv[k & 1] == k, "S MMA read a Q slot not yet converted"
                assert len(m.S_read_by) == NSM, "S buffer overwritten before the softmax copied it"
                m.q_reads[k & 1] += 1
            else:
                _, g, k, acc = op
                assert m.P_buf[g & 1] == g, "P*V read a P buffer holding another tile"
                assert m.slot[g % m.S] == g, "P*V read a V slot holding another tile"
                if not acc:
                    assert m.O_reading is None, "O overwritten while an epilogue reads it"
                    assert m.O_seg is None or m.O_seg == k - 1, "O of a segment skipped"
                    assert m.O_seg is None or m.O_count == -1, \
                        "O overwritten before the previous epilogue read it"
                m.pv_pending.add(g)
                m.pv_reading_P[g & 1] = g
            return True
        m.running[0] -= 1
        if m.running[0] > 0:
            return True
        m.running = None
        m.pipe.pop(0)
        if op[0] == "S":
            _, g, k = op
            m.S_buf, m.S_read_by = g, set()
            m.readers[g].discard("S")
            m.q_reads[k & 1] -= 1
        else:
            _, g, k, acc = op
            if not acc:
                m.O_seg, m.O_count = k, 0
            assert m.O_seg == k, "P*V accumulated into another segment's O"
            m.O_count += 1
            m.pv_pending.discard(g)
            m.pv_reading_P[g & 1] = None
            m.readers[g].discard("PV")
        return True

    # --------------------------------------------------------------- run
    def run(self):
        m = self
        roles = [self.producer(), self.mma()] + [self.softmax(r) for r in range(NSM)]
        if m.fp8:
            roles.append(self.converter())
        alive = list(roles)
        idle = 0
        while alive or m.pipe or m.tma:
            m.tick += 1
            progressed = False
            for item in [t for t in m.tma if t[0] <= m.tick]:
                m.tma.remove(item)
                item[1]()
                progressed = True
            choices = alive + (["pipe"] if m.pipe else [])
            m.rng.shuffle(choices)
            for c in choices[:m.rng.randint(1, len(choices))] if choices else []:
                if c == "pipe":
                    progressed |= self.pipe_step()
                else:
                    try:
                        progressed |= next(c) is not WAIT
                    except StopIteration:
                        alive.remove(c)
                        progressed = True
            idle = 0 if progressed or m.tma else idle + 1
            assert idle < 1000, "deadlock: " + ", ".join(
                f"{b.name}={b.completed}" for b in m.q_full + m.q_empty + [m.s_full, m.s_free])
        assert not m.pv_pending and m.epilogues == len(m.segs)


def random_segments(rng):
    """A CTA's segment list: first and last segments of a part are often
    short (a sequence cut at a part boundary), the middle ones whole short
    sequences."""
    k = rng.randint(1, 6)
    return [rng.choice([1, 1, 2, 3, rng.randint(1, 12)]) for _ in range(k)]


@pytest.mark.parametrize("fp8", [False, True])
def test_protocol_random_interleavings(fp8):
    rng = random.Random(4321 + fp8)
    stages, stages8 = (4, 4) if fp8 else (6, 0)
    for trial in range(400):
        Model(random.Random(rng.random()), fp8, random_segments(rng), stages, stages8).run()


@pytest.mark.parametrize("fp8", [False, True])
def test_protocol_single_tile_segments(fp8):
    # every segment one tile: Q slots and O turn over on every tile
    rng = random.Random(99 + fp8)
    stages, stages8 = (4, 4) if fp8 else (6, 0)
    for trial in range(200):
        Model(random.Random(rng.random()), fp8, [1] * rng.randint(2, 9), stages, stages8).run()


def _run_mutant(cls, seed, trials=400):
    rng = random.Random(seed)
    for trial in range(trials):
        try:
            cls(random.Random(rng.random()), False, random_segments(rng), 6, 0).run()
        except AssertionError:
            return True
    return False


def test_model_catches_a_missing_epilogue_wait():
    # an epilogue that does not wait for its segment's last P V reads O with
    # products missing
    class NoLastPv(Model):
        def wait_last_pv(self, gl):
            return
            yield
    assert _run_mutant(NoLastPv, 17)


def test_model_catches_a_missing_q_empty_wait():
    # the producer reloading a Q slot without waiting for the S MMAs that read it
    class NoQEmpty(Model):
        def producer(self):
            m = self
            g = 0
            for k, n in enumerate(m.segs):
                assert m.q_reads[k & 1] == 0, "Q slot overwritten while an S MMA reads it"

                def land_q(k=k):
                    m.q_slot[k & 1] = k
                    m.q_full[k & 1].arrive()
                m.tma.append((m.tick + m.rng.randint(1, 20), land_q))
                yield
                for _ in range(n):
                    s, r = g % m.S, g // m.S
                    if r > 0:
                        while not m.kv_empty[s].ready(r - 1):
                            yield WAIT
                    self._check_slot_free(s)

                    def land(s=s, g=g):
                        m.slot[s] = g
                        m.readers[g] = {"S", "PV"}
                        m.kv_full[s].arrive()
                    m.tma.append((m.tick + m.rng.randint(1, 30), land))
                    g += 1
                    yield
    assert _run_mutant(NoQEmpty, 23)


def test_model_catches_a_late_q_release():
    # releasing the Q slot after the FIRST S of a segment (not the last) lets
    # the producer overwrite Q while later S MMAs of the segment still need it
    class EarlyRelease(Model):
        def mma(self):
            m = self
            G = 0
            for k, n in enumerate(m.segs):
                while not m.q_full[k & 1].ready(k >> 1):
                    yield WAIT
                yield from m.issue_s(G, k, k & 1)
                for j in range(n):
                    if j + 1 < n:
                        yield from m.issue_s(G + j + 1, k, None)
                    yield from m.issue_pv(G + j, k, j > 0)
                G += n
    rng = random.Random(31)
    caught = False
    for trial in range(600):
        segs = [rng.randint(3, 8) for _ in range(rng.randint(3, 6))]
        try:
            EarlyRelease(random.Random(rng.random()), False, segs, 6, 0).run()
        except AssertionError:
            caught = True
            break
    assert caught


def test_model_reports_a_deadlock():
    class Stuck(Model):
        def softmax(self, role=0):
            while True:
                yield WAIT
    with pytest.raises(AssertionError, match="deadlock"):
        Stuck(random.Random(5), False, [3, 2], 6, 0).run()


def test_model_catches_an_unconverted_q_read():
    # with an FP8 cache, an MMA warp that starts a segment on the Q copy
    # instead of the softmax warps' conversion reads bf16 Q as f16
    class EarlyQ(Model):
        def q_wait(self, k):
            while not self.q_full[k & 1].ready(k >> 1):
                yield WAIT
    rng = random.Random(29)
    caught = False
    for trial in range(400):
        try:
            EarlyQ(random.Random(rng.random()), True, random_segments(rng), 4, 4).run()
        except AssertionError:
            caught = True
            break
    assert caught


def test_model_catches_an_early_p_arrival_of_the_padding_warps():
    # a padding-row warp that arrives on P buffer g % 2 before waiting for
    # S(g) can complete that buffer's phase before the query-row warp wrote
    # P(g), so P(g) V_g runs on a P buffer holding another tile
    class EarlyPad(Model):
        def softmax(self, role=0):
            if role == 0:
                yield from Model.softmax(self, role)
                return
            m = self
            G = 0
            for k, n in enumerate(m.segs):
                for j in range(n):
                    g = G + j
                    m.p_full[g & 1].arrive()
                    yield
                    while not m.s_full.ready(g):
                        yield WAIT
                    m.S_read_by.add(role)
                    m.s_free.arrive()
                    yield
                yield from m.wait_last_pv(G + n - 1)
                G += n
    assert _run_mutant(EarlyPad, 41)
