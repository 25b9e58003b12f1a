"""ORACLE (test infrastructure only): split softmax states and their merge.

Only tests/, the smoke check and the bench's CPU-baseline leg may use it.

A split-KV decode computes, for each query head and each slice of a
sequence's tokens, a partial state (m, l, o): m the largest scaled score in
the slice, l = sum exp(s_t - m), o = sum exp(s_t - m) * v_t (unnormalised).
The merge pass combines the slices of one sequence by log-sum-exp rescaling:
  M = max_i m_i,  l = sum_i l_i exp(m_i - M),  out = sum_i o_i exp(m_i - M) / l,
  lse = M + ln l.
The pages name split-KV partial work ("Attention Backend: Dynamic
Load-Balanced Scheduling") but print no merge formula; the one above is the
standard identity that makes split-then-merge equal the unsplit softmax.
Everything is fp64 numpy.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np


def partial_state(scores: np.ndarray, v: np.ndarray) -> Tuple[float, float, np.ndarray]:
    """scores: [n] fp64 scaled logits of one slice; v: [n][D] fp64 rows."""
    scores = np.asarray(scores, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m = float(np.max(scores))
    w = np.exp(scores - m)
    return m, float(np.sum(w)), w @ v


def merge_states(states: List[Tuple[float, float, np.ndarray]]) -> Tuple[np.ndarray, float]:
    """Merge partial states of one (sequence, query head) -> (out, lse)."""
    if not states:
        raise ValueError("no partial states")
    M = max(s[0] for s in states)
    l = sum(s[1] * np.exp(s[0] - M) for s in states)
    o = sum(s[2] * np.exp(s[0] - M) for s in states)
    return o / l, M + float(np.log(l))
