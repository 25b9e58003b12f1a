"""CPU model of the order in which the one-token step kernel's producer warp
walks an owner's unit range (paged_gqa_decode_hpc_gb300/csrc/step_kernel.cu):
its first piece, then its last piece when that piece is the head of a pair
continuing past the range, then the whole pairs between them. The model
restates the kernel's index arithmetic (prefix of units per sequence, the
sequence holding a unit, pair bounds) and is checked against the oracle's
step plan: every owner publishes exactly the oracle's pieces of that owner
(sequence, KV head, tiles, whole flag, partial slot), split pieces come
before whole ones, and the pool is asked for the next chunk when two units
of the owner are left. Planted mistakes in the walk are caught."""
import random

import pytest

from oracle import plan_ref

CLAIM_AHEAD = 2


def walk(lens, H, owner_start, owner, plant=None):
    n = [(L + 63) // 64 for L in lens]
    cu = [0]
    for nb in n:
        cu.append(cu[-1] + nb * H)
    B = len(lens)

    def seq_at(x):
        l0, h0 = 0, B
        while h0 - l0 > 1:
            mid = (l0 + h0) >> 1
            if cu[mid] <= x:
                l0 = mid
            else:
                h0 = mid
        while cu[l0 + 1] <= x:
            l0 += 1
        return l0

    lo, hi = owner_start[owner], owner_start[owner + 1]
    out, asks = [], []
    ra, rb = lo, hi
    rest_a = rest_b = hi
    first = False
    b = seq_at(lo)
    nb0 = (cu[b + 1] - cu[b]) // H
    e0 = cu[b] + ((lo - cu[b]) // nb0 + 1) * nb0
    if e0 < hi:
        rb, first = e0, True
    left = hi - lo
    while True:
        u = ra
        while u < rb:
            while cu[b + 1] <= u:
                b += 1
            nb = (cu[b + 1] - cu[b]) // H
            rel = u - cu[b]
            hu = rel // nb
            t0 = rel - hu * nb
            pair_lo = cu[b] + hu * nb
            e = min(rb, pair_lo + nb)
            t1 = t0 + (e - u)
            whole = t0 == 0 and t1 == nb
            slot = -1 if whole else (2 * owner if u == lo else 2 * owner + 1)
            out.append((b, hu, t0, t1, whole, slot))
            for _ in range(e - u):
                if not asks and left <= CLAIM_AHEAD:
                    asks.append(left)
                left -= 1
            u = e
        if first:
            first = False
            e0 = rb
            b1 = seq_at(hi - 1)
            nb1 = (cu[b1 + 1] - cu[b1]) // H
            s1 = cu[b1] + ((hi - 1 - cu[b1]) // nb1) * nb1
            if s1 + nb1 > hi and s1 > e0 and plant != "unit_order":
                rest_a, rest_b, ra, b = e0, s1, s1, b1
                if plant == "middle_overlaps_last":
                    rest_b = s1 + 1
            else:
                ra = e0
            rb = hi
            continue
        if rest_a < rest_b:
            ra, rb, rest_a = rest_a, rest_b, rest_b
            b = seq_at(ra)
            continue
        break
    return out, asks, left


def check(lens, H, sms, plant=None):
    sp = plan_ref.step_plan(lens, sms, H)
    owners = sp.num_parts + sp.num_chunks
    by_owner = {}
    for pc in sp.pieces:
        by_owner.setdefault(pc.owner, []).append(
            (pc.seq, pc.head, pc.tile_begin, pc.tile_end, pc.whole, pc.slot))
    for o in range(owners):
        got, asks, left = walk(lens, H, sp.owner_start, o, plant)
        assert sorted(got) == sorted(by_owner[o]), f"owner {o}: pieces differ from the plan's"
        assert left == 0
        size = sp.owner_start[o + 1] - sp.owner_start[o]
        assert asks == [min(size, CLAIM_AHEAD)], "one pool request, two units before the end"
        rest = [w for (_, _, _, _, w, _) in got[1:]]
        k = rest.index(True) if True in rest else len(rest)
        assert all(rest[k:]), f"owner {o}: a split piece after a whole pair"
        assert rest.count(False) <= 1


def _cases(seed, count):
    rng = random.Random(seed)
    for _ in range(count):
        B = rng.randint(1, 40)
        lens = [rng.choice([0, 1, 63, 64, 65, rng.randint(1, 9000)]) for _ in range(B)]
        yield lens, rng.choice([1, 2, 4, 8]), rng.choice([1, 3, 7, 37, 152])


def test_walk_matches_plan_random():
    for lens, H, sms in _cases(3, 400):
        check(lens, H, sms)


def test_walk_pages_workloads():
    check([37, 64, 200, 1000], 1, 152)
    check([512] * 64, 8, 152)
    check([131072] + [4096] * 31, 8, 152)


@pytest.mark.parametrize("plant", ["unit_order", "middle_overlaps_last"])
def test_planted_walk_mistakes_are_caught(plant):
    with pytest.raises(AssertionError):
        for lens, H, sms in _cases(5, 400):
            check(lens, H, sms, plant)
