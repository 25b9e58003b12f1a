"""ORACLE -- test infrastructure, not part of the product.

Plain, slow, obviously correct CPU implementations of what the decode path
computes, used only by tests/, the smoke check and the bench's CPU-baseline
(and `--impl reference`) legs. The CUDA library never imports, links or calls
anything here, and nothing here imports the CUDA library: the two share no
code. Only the seeded input generators are common to both sides.

Contents:
  decode_ref.c   fp64 paged GQA decode from its definition (POSIX threads);
                 __init__.py reduces multi-token decode and ragged prefill /
                 extend to it, one (sequence, new token) at a time.
  plan_ref.py    the dynamic (load-balanced) and static split-KV tile plans.
  merge_ref.py   partial softmax states and their log-sum-exp merge.

Every function here has pins in tests/ (closed forms, brute force,
invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decode_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_decode.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile decode_ref.c with gcc (plain C, -O2, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Load a compiled oracle library (the default one, or a test's variant)."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, f64 = ctypes.c_int32, ctypes.c_double
    lib.oracle_paged_decode.restype = ctypes.c_int
    lib.oracle_paged_decode.argtypes = [i32, i32, i32, i32, P, P, P, i32, f64, f64,
                                        P, i32, P, f64, P, P, i32]
    lib.oracle_bf16_to_f64.restype = f64
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_to_f64.restype = f64
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_num_cpus.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def num_cpus() -> int:
    return int(_load().oracle_num_cpus())


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(bits & 0xFFFF))


def e4m3_to_f64(byte: int) -> float:
    return float(_load().oracle_e4m3_to_f64(byte & 0xFF))


def _as_u16(x) -> np.ndarray:
    """bf16 payload as uint16 bits (accepts a torch bf16 tensor or uint16 array)."""
    if hasattr(x, "dtype") and str(getattr(x, "dtype")) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.ascontiguousarray(np.asarray(x))
    if a.dtype != np.uint16:
        raise TypeError("bf16 data must be given as uint16 bits")
    return a


def _as_np(x, dtype) -> np.ndarray:
    if hasattr(x, "numpy") and not isinstance(x, np.ndarray):
        x = x.contiguous().numpy()
    a = np.ascontiguousarray(np.asarray(x))
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, *, num_kv_heads: int,
                 softmax_scale: float, kv_is_fp8: bool = False, k_scale: float = 1.0,
                 v_scale: float = 1.0, num_threads: int = 0, lib=None):
    """fp64 decode attention. Returns (out [B][H_q][D] f64, lse [B][H_q] f64).

    q: bf16 [B][H_q][D]; k_cache/v_cache: bf16 or e4m3 bytes (uint8)
    [num_blocks][H_kv][64][D]; block_table int32 [B][max_blocks];
    seq_lens int32 [B].
    """
    lib = _load() if lib is None else lib
    qb = _as_u16(q)
    if kv_is_fp8:
        kb, vb = _as_np(k_cache, np.uint8), _as_np(v_cache, np.uint8)
    else:
        kb, vb = _as_u16(k_cache), _as_u16(v_cache)
    bt = _as_np(block_table, np.int32)
    sl = _as_np(seq_lens, np.int32)
    B, hq, D = qb.shape
    if kb.shape[1] != num_kv_heads or kb.shape[2] != 64 or kb.shape[3] != D:
        raise ValueError("k_cache must be [num_blocks][H_kv][64][D]")
    if kb.shape != vb.shape or bt.shape[0] != B or sl.shape != (B,):
        raise ValueError("shape mismatch")
    out = np.zeros((B, hq, D), dtype=np.float64)
    lse = np.zeros((B, hq), dtype=np.float64)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    rc = lib.oracle_paged_decode(B, hq, num_kv_heads, D, ptr(qb), ptr(kb), ptr(vb),
                                 1 if kv_is_fp8 else 0, float(k_scale), float(v_scale),
                                 ptr(bt), bt.shape[1], ptr(sl), float(softmax_scale),
                                 ptr(out), ptr(lse), int(num_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_paged_decode failed with code {rc}")
    return out, lse


def decode_workload(w, num_threads: int = 0, lib=None):
    """Convenience: run the oracle on a workloads.Workload-like object."""
    return paged_decode(w.q, w.k_cache, w.v_cache, w.block_table, w.seq_lens,
                        num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                        kv_is_fp8=(w.kv_dtype == "fp8_e4m3"), k_scale=w.k_scale,
                        v_scale=w.v_scale, num_threads=num_threads, lib=lib)


def paged_decode_multi(q, k_cache, v_cache, block_table, seq_lens, *, num_kv_heads: int,
                       softmax_scale: float, kv_is_fp8: bool = False, k_scale: float = 1.0,
                       v_scale: float = 1.0, num_threads: int = 0, lib=None):
    """Decode of q_len new query tokens per sequence (multi-token / draft
    verification), by its definition: the q_len tokens are the last q_len
    positions of the sequence, and token t attends causally to the positions
    before L - q_len + 1 + t. Each (sequence, token) is therefore a plain decode
    of that length over the same block table.

    q: bf16 [B][q_len][H_q][D]. Returns (out [B][q_len][H_q][D], lse [B][q_len][H_q]).
    """
    import torch
    qt = q if hasattr(q, "shape") else np.asarray(q)
    B, T = int(qt.shape[0]), int(qt.shape[1])
    lens = _as_np(seq_lens, np.int32)
    vlen = np.array([max(0, int(lens[b]) - T + 1 + t) for b in range(B) for t in range(T)],
                    dtype=np.int32)
    bt = np.repeat(_as_np(block_table, np.int32), T, axis=0)
    qv = qt.reshape(B * T, qt.shape[2], qt.shape[3])
    out, lse = paged_decode(qv, k_cache, v_cache, bt, vlen, num_kv_heads=num_kv_heads,
                            softmax_scale=softmax_scale, kv_is_fp8=kv_is_fp8, k_scale=k_scale,
                            v_scale=v_scale, num_threads=num_threads, lib=lib)
    return out.reshape(B, T, qt.shape[2], -1), lse.reshape(B, T, -1)


def paged_extend(q, k_cache, v_cache, block_table, seq_lens, cu_q_lens, *, num_kv_heads: int,
                 softmax_scale: float, kv_is_fp8: bool = False, k_scale: float = 1.0,
                 v_scale: float = 1.0, num_threads: int = 0, lib=None, rows=None):
    """Prefill / extend attention over the paged cache ("vLLM x HPC-Ops",
    section "Attention Across Prefill, Extend and Decode Shapes"), by its
    definition. Sequence b brings n_b = cu_q_lens[b+1] - cu_q_lens[b] new
    tokens, already written to its cache, so they are its last n_b positions
    of L_b = seq_lens[b]; new token i (0-based) attends causally to the
    positions before L_b - n_b + 1 + i. Prefill is the case n_b = L_b.
    Each (sequence, new token) is a plain decode of that length over the
    sequence's block table, computed by the fp64 decode oracle.

    q: bf16 [total_q][H_q][D] (rows of sequence b at cu_q_lens[b]..);
    cu_q_lens int32 [B+1], non-decreasing from 0 to total_q.
    Returns (out [total_q][H_q][D] f64, lse [total_q][H_q] f64); with `rows`
    (indices into total_q) only those rows, in that order.
    """
    qt = q if hasattr(q, "shape") else np.asarray(q)
    cu = _as_np(cu_q_lens, np.int32).astype(np.int64)
    lens = _as_np(seq_lens, np.int32)
    bt = _as_np(block_table, np.int32)
    B = int(lens.shape[0])
    total = int(qt.shape[0])
    if cu.shape != (B + 1,) or cu[0] != 0 or cu[-1] != total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_q_lens must run from 0 to total_q without decreasing")
    seq_rows, vlen = [], []
    for b in range(B):
        n = int(cu[b + 1] - cu[b])
        if n > int(lens[b]):
            raise ValueError("a sequence has more new tokens than positions")
        for i in range(n):
            seq_rows.append(b)
            vlen.append(int(lens[b]) - n + 1 + i)
    seq_of = np.array(seq_rows, dtype=np.int64)
    vlen = np.array(vlen, dtype=np.int32)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        qt = qt[rows]
        seq_of, vlen = seq_of[rows], vlen[rows]
    if len(vlen) == 0:
        return (np.zeros((0,) + tuple(qt.shape[1:]), dtype=np.float64),
                np.zeros((0, qt.shape[1]), dtype=np.float64))
    return paged_decode(qt, k_cache, v_cache, bt[seq_of], vlen, num_kv_heads=num_kv_heads,
                        softmax_scale=softmax_scale, kv_is_fp8=kv_is_fp8, k_scale=k_scale,
                        v_scale=v_scale, num_threads=num_threads, lib=lib)
