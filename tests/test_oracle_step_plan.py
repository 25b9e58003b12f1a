"""Pins for the oracle's step plan (plan_ref.step_plan): the work list of a
one-token decode step -- head-major units, a static balanced partition of
the first S units and a pool of chunks for the rest, pieces = owner range x
(sequence, KV head) pair, partial slots 2*owner (+1). Checked with
invariants any correct decomposition must satisfy, an independent unit
index and owner formula, brute force over small inputs, and hand-worked
shapes of the pages' workloads (tests/golden/step_plan_shapes.json)."""
import itertools
import json
import os

import pytest

from oracle import plan_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "step_plan_shapes.json")


def _lengths(case):
    if "lengths" in case:
        return case["lengths"]
    out = []
    for L, k in case["lengths_rle"]:
        out += [L] * k
    return out


def check_step(lengths, num_sms, H, sp):
    n = [(L + 63) // 64 for L in lengths]
    T = H * sum(n)
    assert sp.num_units == T
    W = T - sp.static_units
    assert 0 <= W and 8 * W <= T < 8 * (W + 1)          # the pool is floor(T / 8)
    S, P, C = sp.static_units, sp.num_parts, sp.chunk_units
    assert P == min(num_sms, -(-S // 8))   # at most one unit per consumer warp unless all SMs are used
    assert C >= 8 and sp.num_chunks * C >= W > (sp.num_chunks - 1) * C
    if P:
        assert 12 * P * C >= S           # a chunk is at least a twelfth of a part
    assert sp.num_chunks <= 4 * num_sms
    # independent unit index of (b, h, t): sequences in order, then head, then tile
    cu = [0]
    for nb in n:
        cu.append(cu[-1] + H * nb)
    uidx = lambda b, h, t: cu[b] + h * n[b] + t
    # every (b, h, t) exactly once; each owner's pieces tile its range in order
    seen = {}
    owners = P + sp.num_chunks
    by_owner = [[] for _ in range(owners)]
    for pc in sp.pieces:
        assert 0 <= pc.owner < owners and 0 <= pc.head < H
        assert 0 <= pc.tile_begin < pc.tile_end <= n[pc.seq]
        by_owner[pc.owner].append(pc)
        for t in range(pc.tile_begin, pc.tile_end):
            key = (pc.seq, pc.head, t)
            assert key not in seen
            seen[key] = pc.owner
    assert len(seen) == T
    sizes = []
    for o in range(owners):
        flat = [uidx(pc.seq, pc.head, t) for pc in by_owner[o]
                for t in range(pc.tile_begin, pc.tile_end)]
        assert flat, "no empty owner"
        assert flat == list(range(flat[0], flat[0] + len(flat)))
        sizes.append(len(flat))
        if o > 0:
            prev = [uidx(pc.seq, pc.head, pc.tile_end - 1) for pc in by_owner[o - 1]][-1]
            assert flat[0] == prev + 1
    # static parts balanced over S; owner of static unit x = floor(((x+1)P - 1)/S)
    if P:
        st = sizes[:P]
        assert sum(st) == S and max(st) - min(st) <= 1
        assert P == num_sms or max(st) <= 8
        for (b, h, t), o in seen.items():
            x = uidx(b, h, t)
            if x < S:
                assert o == ((x + 1) * P - 1) // S
            else:
                assert o == P + (x - S) // C
    assert all(s == C for s in sizes[P:P + sp.num_chunks - 1])
    # pieces of a pair: consecutive owners, contiguous tiles, WHOLE iff alone
    pairs = {}
    for pc in sp.pieces:
        pairs.setdefault((pc.seq, pc.head), []).append(pc)
    for (b, h), pcs in pairs.items():
        assert sp.pair_pieces[(b, h)] == len(pcs)
        assert [pc.owner for pc in pcs] == list(range(pcs[0].owner, pcs[0].owner + len(pcs)))
        assert pcs[0].tile_begin == 0 and pcs[-1].tile_end == n[b]
        for a, c in zip(pcs, pcs[1:]):
            assert a.tile_end == c.tile_begin
        assert all(pc.whole == (len(pcs) == 1) for pc in pcs)
    # slots: one per split piece, distinct, 2*owner for an owner's first piece,
    # 2*owner + 1 for its last; the lookup a merger uses from the pair's first
    # unit A: slot = 2*o + (0 if A <= owner start else 1)
    slots = [pc.slot for pc in sp.pieces if not pc.whole]
    assert len(slots) == len(set(slots))
    for o in range(owners):
        pcs = by_owner[o]
        for i, pc in enumerate(pcs):
            if pc.whole:
                assert pc.slot == -1
                continue
            assert 0 < len(pcs) and (i == 0 or i == len(pcs) - 1)
            assert pc.slot == (2 * o if i == 0 else 2 * o + 1)
            A = uidx(pc.seq, pc.head, 0)
            assert pc.slot == 2 * o + (0 if A <= sp.owner_start[o] else 1)


@pytest.mark.parametrize("H", [1, 2, 4, 8])
def test_brute_force_small(H):
    vals = [0, 1, 63, 64, 65, 130, 300, 700]
    for B in (1, 2, 3):
        for lens in itertools.product(vals, repeat=B):
            for sms in (1, 2, 3, 5, 9, 40):
                sp = plan_ref.step_plan(list(lens), sms, H)
                check_step(list(lens), sms, H, sp)


def test_random_batches():
    import random
    rng = random.Random(7)
    for _ in range(60):
        B = rng.randint(1, 24)
        lens = [rng.choice([0, 1, rng.randint(1, 5000)]) for _ in range(B)]
        H = rng.choice([1, 2, 4, 8, 16])
        sms = rng.choice([1, 7, 64, 152, 160])
        check_step(lens, sms, H, plan_ref.step_plan(lens, sms, H))


def test_pages_workload_shapes():
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        lens = _lengths(c)
        sp = plan_ref.step_plan(lens, c["num_sms"], c["num_kv_heads"])
        assert (sp.num_units, sp.static_units, sp.num_parts, sp.chunk_units, sp.num_chunks) == \
            (c["T"], c["S"], c["P"], c["C"], c["chunks"]), c["name"]
        if "whole_chunks" in c:
            chunk_pieces = [pc for pc in sp.pieces if pc.owner >= sp.num_parts]
            assert sum(pc.whole for pc in chunk_pieces) == c["whole_chunks"]
        check_step(lens, c["num_sms"], c["num_kv_heads"], sp)


def test_uniform_split_pairs_match_part_boundaries():
    """On the uniform batch the static parts (23 or 24 units) are longer than a
    pair (8 units), so each part boundary that falls strictly inside a pair
    splits that pair in two and no pair is cut twice; the pool's 64 pairs
    (sequences 56..63) are its 64 chunks, whole."""
    lens = [512] * 64
    sp = plan_ref.step_plan(lens, 152, 8)
    inside = sum(1 for p in range(1, 152) if (p * 3584 // 152) % 8 != 0)
    split = [k for k in sp.pair_pieces.values() if k > 1]
    assert len(split) == inside and set(split) == {2}


def test_empty_and_degenerate():
    sp = plan_ref.step_plan([0, 0], 152, 8)
    assert sp.num_units == 0 and sp.num_parts == 0 and sp.num_chunks == 0 and not sp.pieces
    sp = plan_ref.step_plan([1], 152, 1)       # one unit: static, no pool
    assert (sp.static_units, sp.num_parts, sp.num_chunks) == (1, 1, 0)
    assert sp.pieces[0].whole
    with pytest.raises(ValueError):
        plan_ref.step_plan([-1], 4, 1)


def test_skewed_pool_chunks_are_quarter_pairs():
    """On the skewed batch the pool (the last 4032 units) starts on a pair
    boundary (S = 441 * 64) and a chunk is a twelfth of a part rounded up,
    16 units: every pool chunk is one piece, a quarter of a 64-unit pair, and
    each of those 63 pairs is merged from exactly 4 pieces."""
    lens = [131072] + [4096] * 31
    sp = plan_ref.step_plan(lens, 152, 8)
    pool = [pc for pc in sp.pieces if pc.owner >= sp.num_parts]
    assert len(pool) == sp.num_chunks == 252
    assert all(pc.tile_end - pc.tile_begin == 16 and not pc.whole for pc in pool)
    pairs = {(pc.seq, pc.head) for pc in pool}
    assert len(pairs) == 63 and all(sp.pair_pieces[k] == 4 for k in pairs)
