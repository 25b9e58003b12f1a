"""ORACLE (test infrastructure only): the fused decode prologue, written plainly.

Only tests/, the smoke check and the bench's CPU legs may use it.

The pages describe one kernel ahead of decode attention that applies
QK-Norm and RoPE to the new token's query and key, writes key and value into
the paged KV cache, and (in FP8) quantises the query ("vLLM x HPC-Ops",
section "Attention Backend: Dynamic Load-Balanced Scheduling", paragraph on
HpcRopeNorm; the 24-ai.news page lists RoPE, QK-Norm and the KV write). They
give no formulas. Readings taken here (all in fp64):
  * QK-Norm = RMSNorm over head_dim per head, with one learned weight vector
    for queries and one for keys: y = x / sqrt(mean(x^2) + eps) * w;
  * the norm comes before RoPE (the order of the first page);
  * RoPE rotates pairs (i, i + D/2) ("rotate half"), angle = pos * base^(-2i/D);
  * the new token sits at position pos = seq_len - 1 (seq_len counts it) and
    goes to slot pos % 64 of block block_table[b][pos // 64];
  * V is written unchanged; K and V are cast to the cache type: bf16, or
    e4m3 of (x / scale) with round-to-nearest-even and saturation to +-448;
  * the optional FP8 query is e4m3 of (q / q_scale) the same way.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x: [..., D] fp64; w: [D]."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rope_angles(pos: int, head_dim: int, base: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return pos * np.power(float(base), -2.0 * i / head_dim)


def rope(x: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotate-half RoPE of x [..., D] at one position."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    a = rope_angles(pos, D, base)
    c, s = np.cos(a), np.sin(a)
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def e4m3_decode(byte: int) -> float:
    """OCP E4M3 value of one byte (bias 7, no infinities, S.1111.111 = NaN)."""
    s = (byte >> 7) & 1
    e = (byte >> 3) & 0xF
    m = byte & 7
    if e == 0xF and m == 7:
        return math.nan
    v = math.ldexp(m / 8.0, -6) if e == 0 else math.ldexp(1.0 + m / 8.0, e - 7)
    return -v if s else v


_E4M3_MAGS = None


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code of x: round |x| to the nearest of the 127 finite
    magnitudes (ties to the even mantissa), saturating at 448, then set the
    sign bit for negative x (including -0.0). NaN maps to 0x7F."""
    global _E4M3_MAGS
    if _E4M3_MAGS is None:
        _E4M3_MAGS = [(c, e4m3_decode(c)) for c in range(0x7F)]
    if math.isnan(x):
        return 0x7F
    a = min(abs(x), E4M3_MAX)
    best, bd = 0, None
    for c, v in _E4M3_MAGS:
        d = abs(v - a)
        if bd is None or d < bd or (d == bd and (c & 1) == 0):
            best, bd = c, d
    return best | (0x80 if math.copysign(1.0, x) < 0 else 0)


def prologue(q, k, v, seq_lens, block_table, w_q, w_k, eps: float, base: float):
    """Returns (q_out [B][Hq][D], k_rows [B][Hkv][D], v_rows [B][Hkv][D],
    slots [B] as (block, slot) or None for empty sequences), all fp64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B = q.shape[0]
    q_out = np.zeros_like(q)
    k_out = np.zeros_like(k)
    slots = []
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            slots.append(None)
            continue
        pos = L - 1
        q_out[b] = rope(rms_norm(q[b], w_q, eps), pos, base)
        k_out[b] = rope(rms_norm(k[b], w_k, eps), pos, base)
        slots.append((int(block_table[b][pos // 64]), pos % 64))
    return q_out, k_out, v.copy(), slots
