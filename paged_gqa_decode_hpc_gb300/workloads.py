"""Seeded synthetic inputs for mixed-length paged GQA decode.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests. It holds none of the attention arithmetic: it only draws lengths,
block tables and tensors, and encodes the FP8 KV bytes that both sides then
read (the encoding is input preparation, the decoding is each side's job).

Workload shapes follow the pages' decode workloads ("vLLM x HPC-Ops", section
"Attention Decode under Mixed-Length Batches": uniform 64 x 0.5K and
1 x 128K + 31 x 4K mixes; Hy3 shape 64 query / 8 KV heads, head_dim 128;
"Using HPC-Ops Backends in vLLM": 64-token blocks, fp8_e4m3 KV cache).

Recipe (torch CPU generator, seed = 1000 + config index), drawn in this order:
  1. sequence lengths (fixed lists, or log-uniform draws);
  2. a permutation of the physical block ids;
  3. Q ~ N(0,1) -> bf16, [B][H_q][D];
  4. K ~ N(0,1), then V ~ N(0,1), each [num_blocks][H_kv][64][D] (bf16), or
     for FP8: fp32 values, scale = max|x| / 448 per tensor, bytes =
     (x / scale).clamp(+-448) cast to float8_e4m3fn (round to nearest even).
Sequence b's j-th logical block is physical block perm[cu_tiles[b] + j].
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

BLOCK_SIZE = 64
HEAD_DIM = 128
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Config:
    index: int
    name: str
    num_q_heads: int
    num_kv_heads: int
    kv_dtype: str  # "bf16" | "fp8_e4m3"
    lengths: Optional[List[int]] = None  # fixed lengths; None -> drawn
    num_random_seqs: int = 0  # log-uniform draw when lengths is None
    random_lo: int = 16
    random_hi: int = 65536

    @property
    def seed(self) -> int:
        return 1000 + self.index


CONFIGS = [
    Config(0, "tiny", 8, 1, "bf16", lengths=[37, 64, 200, 1000]),
    Config(1, "uniform", 64, 8, "bf16", lengths=[512] * 64),
    Config(2, "skewed", 64, 8, "bf16", lengths=[131072] + [4096] * 31),
    Config(3, "skewed_fp8", 64, 8, "fp8_e4m3", lengths=[131072] + [4096] * 31),
    Config(4, "random_mixed", 64, 8, "bf16", lengths=None, num_random_seqs=256),
]
CONFIG_BY_NAME = {c.name: c for c in CONFIGS}


@dataclasses.dataclass
class Workload:
    """Host-side (CPU) tensors of one decode step."""
    config_name: str
    seq_lens: torch.Tensor      # int32 [B]
    block_table: torch.Tensor   # int32 [B][max_blocks]; unused entries -1
    q: torch.Tensor             # bf16 [B][H_q][D]
    k_cache: torch.Tensor       # bf16 or uint8 (e4m3 bytes) [NB][H_kv][64][D]
    v_cache: torch.Tensor
    k_scale: float              # 1.0 for bf16
    v_scale: float
    kv_dtype: str
    softmax_scale: float
    num_q_heads: int
    num_kv_heads: int

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.numel())

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes: actual tokens only (not padded blocks)."""
        elt = 1 if self.kv_dtype == "fp8_e4m3" else 2
        tokens = int(self.seq_lens.to(torch.int64).sum())
        return 2 * tokens * self.num_kv_heads * HEAD_DIM * elt

    def qo_bytes(self) -> int:
        return 2 * 2 * self.num_seqs * self.num_q_heads * HEAD_DIM

    def algorithmic_bytes(self) -> int:
        return self.kv_bytes() + self.qo_bytes()


def draw_lengths(cfg: Config, gen: torch.Generator) -> List[int]:
    if cfg.lengths is not None:
        return list(cfg.lengths)
    lo, hi = math.log(cfg.random_lo), math.log(cfg.random_hi)
    u = torch.rand(cfg.num_random_seqs, generator=gen, dtype=torch.float64)
    lens = torch.round(torch.exp(lo + (hi - lo) * u)).clamp(cfg.random_lo, cfg.random_hi)
    return [int(x) for x in lens.tolist()]


def tiles_of(length: int) -> int:
    return (length + BLOCK_SIZE - 1) // BLOCK_SIZE


def _randn_chunked(shape, gen: torch.Generator, chunk: int = 1 << 26) -> torch.Tensor:
    """N(0,1) float32 drawn in fixed-size chunks (same stream as one call)."""
    n = 1
    for s in shape:
        n *= s
    out = torch.empty(n, dtype=torch.float32)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = torch.randn(hi - lo, generator=gen, dtype=torch.float32)
    return out.view(*shape)


def encode_e4m3(x: torch.Tensor):
    """Per-tensor scaled e4m3 bytes: scale = max|x| / 448 (input preparation)."""
    amax = float(x.abs().max())
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    scale = float(torch.tensor(scale, dtype=torch.float32))  # an fp32 scalar
    y = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return y.view(torch.uint8), scale


def build_block_table(lengths: List[int], perm: torch.Tensor) -> torch.Tensor:
    n = [tiles_of(L) for L in lengths]
    max_blocks = max([1] + n)
    bt = torch.full((len(lengths), max_blocks), -1, dtype=torch.int32)
    cu = 0
    for b, nb in enumerate(n):
        if nb:
            bt[b, :nb] = perm[cu:cu + nb].to(torch.int32)
        cu += nb
    return bt


def make_workload(cfg: Config | str, lengths: Optional[List[int]] = None,
                  seed: Optional[int] = None, slack_blocks: int = 0,
                  q_scale: float = 1.0) -> Workload:
    """Build the seeded workload of a config.

    `lengths` / `seed` override the config's (for small parity cases that
    keep the config's head shape and dtype). `slack_blocks` adds unused
    physical blocks. `q_scale` multiplies Q before the bf16 cast (a
    "sharp softmax" variant).
    """
    if isinstance(cfg, str):
        cfg = CONFIG_BY_NAME[cfg]
    gen = torch.Generator().manual_seed(cfg.seed if seed is None else seed)
    lens = draw_lengths(cfg, gen) if lengths is None else list(lengths)
    total_tiles = sum(tiles_of(L) for L in lens)
    num_blocks = total_tiles + slack_blocks
    perm = torch.randperm(num_blocks, generator=gen)
    bt = build_block_table(lens, perm)
    B, hq, hkv = len(lens), cfg.num_q_heads, cfg.num_kv_heads
    q = (_randn_chunked((B, hq, HEAD_DIM), gen) * q_scale).to(torch.bfloat16)
    kv_shape = (max(num_blocks, 1), hkv, BLOCK_SIZE, HEAD_DIM)
    if cfg.kv_dtype == "fp8_e4m3":
        k, ks = encode_e4m3(_randn_chunked(kv_shape, gen))
        v, vs = encode_e4m3(_randn_chunked(kv_shape, gen))
    else:
        k = _randn_chunked(kv_shape, gen).to(torch.bfloat16)
        v = _randn_chunked(kv_shape, gen).to(torch.bfloat16)
        ks = vs = 1.0
    return Workload(cfg.name, torch.tensor(lens, dtype=torch.int32), bt, q, k, v,
                    ks, vs, cfg.kv_dtype, 1.0 / math.sqrt(HEAD_DIM), hq, hkv)


@dataclasses.dataclass
class PrologueInputs:
    """The new token's projections for the fused prologue (host tensors)."""
    q_in: torch.Tensor      # bf16 [B][H_q][D]
    k_in: torch.Tensor      # bf16 [B][H_kv][D]
    v_in: torch.Tensor      # bf16 [B][H_kv][D]
    w_q: torch.Tensor       # bf16 [D] RMSNorm weight of q
    w_k: torch.Tensor       # bf16 [D]
    eps: float
    rope_base: float


def make_prologue_inputs(w: Workload, seed: int, eps: float = 1e-6,
                         rope_base: float = 10000.0) -> PrologueInputs:
    """Seeded N(0,1) q/k/v rows and weights 1 + 0.1 N(0,1) (all bf16)."""
    gen = torch.Generator().manual_seed(seed)
    B, hq, hkv = w.num_seqs, w.num_q_heads, w.num_kv_heads
    q = torch.randn(B, hq, HEAD_DIM, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, hkv, HEAD_DIM, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, hkv, HEAD_DIM, generator=gen).to(torch.bfloat16)
    wq = (1 + 0.1 * torch.randn(HEAD_DIM, generator=gen)).to(torch.bfloat16)
    wk = (1 + 0.1 * torch.randn(HEAD_DIM, generator=gen)).to(torch.bfloat16)
    return PrologueInputs(q, k, v, wq, wk, eps, rope_base)


def make_multi_query(w: Workload, q_len: int, seed: int, q_scale: float = 1.0) -> torch.Tensor:
    """Seeded N(0,1) queries of q_len new tokens per sequence: bf16 [B][q_len][H_q][D]."""
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(w.num_seqs, q_len, w.num_q_heads, HEAD_DIM, generator=gen)
            * q_scale).to(torch.bfloat16)


def make_extend_query(w: Workload, q_lens: List[int], seed: int, q_scale: float = 1.0):
    """Seeded N(0,1) queries of q_lens[b] new tokens of each sequence, packed
    ragged: (q bf16 [total_q][H_q][D], cu_q_lens int32 [B+1]). The new tokens
    are the last q_lens[b] positions of sequence b (q_lens[b] <= its length)."""
    if len(q_lens) != w.num_seqs:
        raise ValueError("one q_len per sequence")
    for n, L in zip(q_lens, w.seq_lens.tolist()):
        if n < 0 or n > L:
            raise ValueError("q_len must lie in [0, seq_len]")
    cu = [0]
    for n in q_lens:
        cu.append(cu[-1] + int(n))
    gen = torch.Generator().manual_seed(seed)
    q = (torch.randn(cu[-1], w.num_q_heads, HEAD_DIM, generator=gen) * q_scale).to(torch.bfloat16)
    return q, torch.tensor(cu, dtype=torch.int32)
