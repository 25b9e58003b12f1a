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

Step plan -- the work list of one decode step with one query token, as the
step call runs it. The same partition rule is applied to finer units, ordered
so that a part's range holds whole (sequence, KV head) pairs where it can:
  * sequence b has n_b * H_kv units; unit u of the sequence is tile u % n_b
    of KV head u // n_b (head-major: a pair's tiles are adjacent);
  * units are flattened in sequence order; T = sum_b n_b * H_kv;
  * the last W = floor(T / 8) units form a pool, S = T - W units are static;
  * P = min(num_sms, ceil(S / 8)) static parts: no more parts than it takes
    to give each CTA's 8 consumer warps one unit (they take a part's units
    round-robin, and more, smaller parts would only cut pairs into more
    pieces); part p owns units [floor(p*S/P), floor((p+1)*S/P)) (the rule
    above, over S units);
  * the pool is cut into chunks of C = max(8, ceil(S / (12 P)),
    ceil(W / (4 * num_sms))) units -- a twelfth of a static part, at least a
    unit per consumer warp, at most 4 chunks per CTA -- chunk j owning
    [S + j*C, min(S + (j+1)*C, T)); chunks are taken at run
    time by whichever CTA asks first (the pages' scheduler is static; this
    small dynamic pool absorbs the SMs' unequal streaming rates, which no
    static work estimate sees);
  * owners are the parts 0..P-1 followed by the chunks P..P+chunks-1; a piece
    is the intersection of an owner's range with one pair's units;
  * a pair held by one piece is WHOLE (its result is final); otherwise each
    of its k pieces leaves a partial state in slot 2*o if the piece is its
    owner o's first piece, else 2*o + 1 (then it is the owner's last piece:
    a piece strictly inside an owner's range is a whole pair), and the k
    states are merged.

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


POOL_DIV = 8          # the pool holds floor(T / POOL_DIV) units
MIN_CHUNK_UNITS = 8   # smallest pool chunk
CHUNKS_PER_SM = 4     # at most this many chunks per CTA of the grid
MIN_PART_UNITS = 8    # parts per 8 static units at most (one unit per consumer warp)
PART_CHUNKS = 12      # a pool chunk is at least this fraction (1/12) of a static part


class Piece(NamedTuple):
    owner: int       # static part p < P, or P + chunk index
    seq: int
    head: int        # KV head
    tile_begin: int
    tile_end: int
    whole: bool      # covers every tile of its (sequence, head) pair
    slot: int        # partial-state slot; -1 for a whole pair


class StepPlan(NamedTuple):
    num_units: int      # T
    static_units: int   # S
    num_parts: int      # P
    chunk_units: int    # C
    num_chunks: int
    owner_start: List[int]   # [P + chunks + 1] first unit of every owner, then T
    pieces: List[Piece]      # by owner, then in unit order
    pair_pieces: dict        # (seq, head) -> number of pieces (pairs with tiles only)


def step_plan(seq_lens: List[int], num_sms: int, num_kv_heads: int) -> StepPlan:
    if num_sms <= 0 or num_kv_heads <= 0 or any(L < 0 for L in seq_lens):
        raise ValueError("num_sms and num_kv_heads must be positive, lengths non-negative")
    n = tile_counts(seq_lens)
    H = num_kv_heads
    T = sum(c * H for c in n)
    W = T // POOL_DIV
    S = T - W
    P = min(num_sms, -(-S // MIN_PART_UNITS))
    C = max(MIN_CHUNK_UNITS, -(-S // (PART_CHUNKS * P)) if P else 0,
            -(-W // (CHUNKS_PER_SM * num_sms)))
    chunks = -(-W // C)
    owner_start = [(p * S) // P for p in range(P)] + [S + j * C for j in range(chunks)] + [T]
    # every unit: (sequence, head, tile), in the flattened order
    units = []
    for b, nb in enumerate(n):
        for h in range(H):
            for t in range(nb):
                units.append((b, h, t))
    assert len(units) == T
    pieces: List[Piece] = []
    for o in range(P + chunks):
        lo, hi = owner_start[o], owner_start[o + 1]
        own: List[List[int]] = []   # [seq, head, tile_begin, tile_end]
        for x in range(lo, hi):
            b, h, t = units[x]
            if own and own[-1][0] == b and own[-1][1] == h:
                own[-1][3] = t + 1
            else:
                own.append([b, h, t, t + 1])
        for i, (b, h, tb, te) in enumerate(own):
            whole = tb == 0 and te == n[b]
            slot = -1 if whole else (2 * o if i == 0 else 2 * o + 1)
            pieces.append(Piece(o, b, h, tb, te, whole, slot))
    pair_pieces: dict = {}
    for pc in pieces:
        pair_pieces[(pc.seq, pc.head)] = pair_pieces.get((pc.seq, pc.head), 0) + 1
    return StepPlan(T, S, P, C, chunks, owner_start, pieces, pair_pieces)
