"""ORACLE (test infrastructure only): the tile plans, written plainly.

Only tests/, the smoke check and the bench's CPU-baseline leg may use it.

Dynamic plan -- the per-step load-balanced scheduler of the HPC-Ops attention
backend ("vLLM x HPC-Ops", section "Attention Backend: Dynamic Load-Balanced
Scheduling": every KV sequence is cut into uniform 64-token tiles and the
tiles are given to the CTAs of a persistent grid by actual work; the
24-ai.news page words it as tiles spread in proportion to each sequence's
length in the current step). The pages give no cost model or partition
formula; this oracle takes the plainest reading:
  * every tile costs one unit (a partial last tile included); optionally a
    tile is split into one unit per KV head (units_per_tile), a finer grain
    for batches with few tiles per CTA;
  * tiles are flattened in input sequence order, without sorting;
  * P = min(num_sms, T) parts (no parts when T == 0);
  * part p owns flattened tiles [floor(p*T/P), floor((p+1)*T/P));
  * a segment is the intersection of a part with one sequence's tiles,
    listed by part and, within a part, by sequence;
  * a segment is WHOLE when it covers every tile of its sequence.

Static plan -- the even split-KV schedule the pages compare against (same
section: "static split-KV"; the 24-ai.news page notes it assumes uniform
lengths). The split count is not given on the pages; the reading used is
S = clamp(ceil(2 * num_sms / (B * H_kv)), 1, max_b n_b), or the caller's
count; split i of a sequence with n tiles is [floor(i*n/S), floor((i+1)*n/S)),
and empty splits are dropped. Each segment is one CTA per KV head.
"""
from __future__ import annotations

from typing import List, NamedTuple, Optional

TILE = 64


class Segment(NamedTuple):
    seq: int
    tile_begin: int  # relative to the sequence's first tile
    tile_end: int
    whole: bool


class Plan(NamedTuple):
    num_tiles: int                 # T
    num_parts: int                 # P
    segments: List[Segment]
    part_seg_off: List[int]        # [P + 1]
    seq_seg_off: List[int]         # [B + 1]


def tile_counts(seq_lens: List[int]) -> List[int]:
    return [(L + TILE - 1) // TILE for L in seq_lens]


def _seq_offsets(segments: List[Segment], num_seqs: int) -> List[int]:
    count = [0] * num_seqs
    for s in segments:
        count[s.seq] += 1
    off = [0]
    for c in count:
        off.append(off[-1] + c)
    return off


def dynamic_plan(seq_lens: List[int], num_sms: int, units_per_tile: int = 1) -> Plan:
    """With units_per_tile = U > 1 every (tile, KV head) pair is one unit of
    work: sequence b has n_b * U units, unit u being head u % U of tile u // U,
    and the same partition is applied to the units (segments then hold unit
    ranges)."""
    if num_sms <= 0 or units_per_tile <= 0 or any(L < 0 for L in seq_lens):
        raise ValueError("num_sms and units_per_tile must be positive, lengths non-negative")
    n = [c * units_per_tile for c in tile_counts(seq_lens)]
    T = sum(n)
    P = min(num_sms, T)
    seq_start = [0]
    for c in n:
        seq_start.append(seq_start[-1] + c)
    segments: List[Segment] = []
    part_seg_off = [0]
    for p in range(P):
        lo_p = (p * T) // P
        hi_p = ((p + 1) * T) // P
        for b in range(len(n)):
            lo = max(lo_p, seq_start[b])
            hi = min(hi_p, seq_start[b + 1])
            if lo < hi:
                tb, te = lo - seq_start[b], hi - seq_start[b]
                segments.append(Segment(b, tb, te, tb == 0 and te == n[b]))
        part_seg_off.append(len(segments))
    return Plan(T, P, segments, part_seg_off, _seq_offsets(segments, len(n)))


def static_split_count(seq_lens: List[int], num_sms: int, num_kv_heads: int,
                       num_splits: Optional[int] = None) -> int:
    n = tile_counts(seq_lens)
    max_n = max([1] + n)
    if num_splits is not None and num_splits > 0:
        s = num_splits
    else:
        denom = len(n) * num_kv_heads
        s = -(-2 * num_sms // denom) if denom > 0 else 1
    return max(1, min(s, max_n))


def static_plan(seq_lens: List[int], num_sms: int, num_kv_heads: int,
                num_splits: Optional[int] = None) -> Plan:
    if num_sms <= 0 or num_kv_heads <= 0 or any(L < 0 for L in seq_lens):
        raise ValueError("bad arguments")
    n = tile_counts(seq_lens)
    S = static_split_count(seq_lens, num_sms, num_kv_heads, num_splits)
    segments: List[Segment] = []
    for b, nb in enumerate(n):
        splits = []
        for i in range(S):
            lo, hi = (i * nb) // S, ((i + 1) * nb) // S
            if lo < hi:
                splits.append((lo, hi))
        for lo, hi in splits:
            segments.append(Segment(b, lo, hi, len(splits) == 1))
    part_seg_off = list(range(len(segments) + 1))  # one segment per part
    return Plan(sum(n), len(segments), segments, part_seg_off,
                _seq_offsets(segments, len(n)))
