"""Pins for the oracle's tile plans: invariants that any correct balanced
partition must satisfy, an independent tile->part map, brute force over all
small length vectors, and the hand-worked tile counts of the pages'
workloads (tests/golden/plan_shapes.json)."""
import itertools
import json
import os

import pytest

from oracle import plan_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_shapes.json")


def _lengths(case):
    if "lengths" in case:
        return case["lengths"]
    out = []
    for L, n in case["lengths_rle"]:
        out += [L] * n
    return out


def check_dynamic(lengths, num_sms, plan, units_per_tile=1):
    n = [c * units_per_tile for c in plan_ref.tile_counts(lengths)]
    T = sum(n)
    assert plan.num_tiles == T
    assert plan.num_parts == min(num_sms, T)
    P = plan.num_parts
    starts = [0]
    for c in n:
        starts.append(starts[-1] + c)
    # every tile exactly once, and each part owns one contiguous range
    owner = {}
    for p in range(P):
        segs = plan.segments[plan.part_seg_off[p]:plan.part_seg_off[p + 1]]
        assert segs, "no empty parts"
        flat = []
        for s in segs:
            assert 0 <= s.tile_begin < s.tile_end <= n[s.seq]
            flat += [starts[s.seq] + t for t in range(s.tile_begin, s.tile_end)]
        assert flat == list(range(flat[0], flat[0] + len(flat)))
        for x in flat:
            assert x not in owner
            owner[x] = p
    assert sorted(owner) == list(range(T))
    # balance: part sizes differ by at most one tile
    sizes = [sum(s.tile_end - s.tile_begin for s in
                 plan.segments[plan.part_seg_off[p]:plan.part_seg_off[p + 1]]) for p in range(P)]
    if P:
        assert max(sizes) - min(sizes) <= 1
        assert max(sizes) == -(-T // P) and min(sizes) == T // P
    # independent owner formula: the part of tile x is floor(((x+1)P - 1)/T)
    for x, p in owner.items():
        assert p == ((x + 1) * P - 1) // T
    # per-sequence bookkeeping
    assert plan.seq_seg_off[0] == 0 and plan.seq_seg_off[-1] == len(plan.segments)
    for b in range(len(lengths)):
        segs = plan.segments[plan.seq_seg_off[b]:plan.seq_seg_off[b + 1]]
        assert all(s.seq == b for s in segs)
        if n[b] == 0:
            assert not segs
            continue
        assert segs[0].tile_begin == 0 and segs[-1].tile_end == n[b]
        for a, c in zip(segs, segs[1:]):
            assert a.tile_end == c.tile_begin
        assert all(s.whole == (len(segs) == 1) for s in segs)
    # a sequence spans ceil(n/part) + 1 parts at most
    return sizes


def test_golden_workload_shapes():
    for case in json.load(open(GOLDEN))["cases"]:
        L = _lengths(case)
        plan = plan_ref.dynamic_plan(L, case["num_sms"])
        sizes = check_dynamic(L, case["num_sms"], plan)
        assert plan.num_tiles == case["T"] and plan.num_parts == case["P"], case["name"]
        assert min(sizes) == case["part_min"] and max(sizes) == case["part_max"]
        assert sizes.count(case["part_max"]) == case["parts_at_max"]


def test_bruteforce_small_length_vectors():
    vals = [0, 1, 63, 64, 65, 128, 200]
    count = 0
    for B in range(0, 4):
        for lens in itertools.product(vals, repeat=B):
            for sms in (1, 2, 3, 5, 9):
                check_dynamic(list(lens), sms, plan_ref.dynamic_plan(list(lens), sms))
                count += 1
    assert count > 1000


def test_random_larger_vectors():
    import random
    rng = random.Random(5)
    for _ in range(200):
        B = rng.randint(1, 40)
        lens = [rng.choice([0, rng.randint(1, 64), rng.randint(1, 5000)]) for _ in range(B)]
        sms = rng.randint(1, 200)
        check_dynamic(lens, sms, plan_ref.dynamic_plan(lens, sms))


def test_empty_and_bad():
    p = plan_ref.dynamic_plan([], 10)
    assert p.num_tiles == 0 and p.num_parts == 0 and p.segments == [] and p.part_seg_off == [0]
    p = plan_ref.dynamic_plan([0, 0], 10)
    assert p.num_parts == 0 and p.seq_seg_off == [0, 0, 0]
    with pytest.raises(ValueError):
        plan_ref.dynamic_plan([-1], 4)
    with pytest.raises(ValueError):
        plan_ref.dynamic_plan([5], 0)


def test_static_plan_rule_and_coverage():
    # uniform 64 x 512 on 152 SMs, 8 kv heads: S = ceil(304/512) = 1
    L = [512] * 64
    assert plan_ref.static_split_count(L, 152, 8) == 1
    # skewed: S = ceil(304 / 256) = 2
    L = [131072] + [4096] * 31
    assert plan_ref.static_split_count(L, 152, 8) == 2
    # tiny with 1 kv head: S = ceil(304 / 4) = 76 -> clamped to max n_b = 16
    assert plan_ref.static_split_count([37, 64, 200, 1000], 152, 1) == 16
    for lens, sms, hkv, S in [([37, 64, 200, 1000], 152, 1, None), ([5000, 64, 1], 10, 2, 3),
                              ([0, 300], 4, 8, 7), ([131072] + [4096] * 31, 152, 8, None)]:
        plan = plan_ref.static_plan(lens, sms, hkv, S)
        n = plan_ref.tile_counts(lens)
        Se = plan_ref.static_split_count(lens, sms, hkv, S)
        assert plan.num_parts == len(plan.segments)
        for b, nb in enumerate(n):
            segs = plan.segments[plan.seq_seg_off[b]:plan.seq_seg_off[b + 1]]
            tiles = [t for s in segs for t in range(s.tile_begin, s.tile_end)]
            assert tiles == list(range(nb))
            assert len(segs) == min(Se, nb)
            sizes = [s.tile_end - s.tile_begin for s in segs]
            if sizes:
                assert max(sizes) - min(sizes) <= 1
            assert all(s.whole == (len(segs) == 1) for s in segs)


def test_units_per_tile_plans():
    # uniform 64 x 512 with one unit per (tile, kv head): 4096 units over 152
    # parts of 26 or 27 units (4096 = 152 * 26 + 144)
    L = [512] * 64
    plan = plan_ref.dynamic_plan(L, 152, units_per_tile=8)
    sizes = check_dynamic(L, 152, plan, units_per_tile=8)
    assert plan.num_tiles == 4096 and min(sizes) == 26 and max(sizes) == 27
    assert sizes.count(27) == 144
    import random
    rng = random.Random(9)
    for _ in range(100):
        lens = [rng.choice([0, rng.randint(1, 64), rng.randint(1, 3000)]) for _ in range(rng.randint(1, 30))]
        sms, u = rng.randint(1, 160), rng.choice([1, 2, 4, 8])
        check_dynamic(lens, sms, plan_ref.dynamic_plan(lens, sms, units_per_tile=u), units_per_tile=u)
    # U = 1 is the tile plan
    assert plan_ref.dynamic_plan([700, 3], 5, 1) == plan_ref.dynamic_plan([700, 3], 5)
