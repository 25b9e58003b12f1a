"""Mixed-length paged GQA decode attention for GB300 (sm_103a).

A thin ctypes binding over libhpc_decode.so (see include/hpc_decode.h). Each
function here has the C entry point's name and only marshals arguments:
torch tensors become `hpc_tensor` descriptors, torch streams become
cudaStream_t handles. Every step of the computation runs in the library's
CUDA kernels; there is no Python or CPU fallback, and a missing library is
an error (build it with `paged_gqa_decode_hpc_gb300.build()`).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import numpy as np

from . import _build

__all__ = [
    "build", "load_library", "HpcError", "Plan",
    "hpc_decode_plan", "hpc_decode_plan_ex", "hpc_decode_plan_compute_ex", "hpc_decode_plan_static", "hpc_decode_plan_create",
    "hpc_decode_plan_device", "hpc_decode_plan_update", "hpc_decode_plan_export",
    "hpc_decode_plan_compute", "hpc_decode_plan_static_compute", "hpc_decode_plan_status",
    "hpc_decode_plan_destroy", "hpc_decode_attn", "hpc_device_sm_count", "hpc_last_error",
    "hpc_decode_plan_set_timing_events", "hpc_decode_attn_noalloc", "hpc_decode_step",
    "hpc_decode_step_host",
    "hpc_rope_norm_kv_write", "hpc_extend_attn", "hpc_decode_tc_min_q_len",
    "HPC_OK", "HPC_ERR_INVALID_ARG", "HPC_ERR_UNSUPPORTED", "HPC_ERR_CUDA", "HPC_ERR_OOM",
    "HPC_ERR_DEVICE_CHECK",
]

HPC_OK, HPC_ERR_INVALID_ARG, HPC_ERR_UNSUPPORTED, HPC_ERR_CUDA, HPC_ERR_OOM, \
    HPC_ERR_DEVICE_CHECK = range(6)
HPC_BF16, HPC_FP8_E4M3, HPC_F32, HPC_I32 = range(4)
HPC_PLAN_DYNAMIC, HPC_PLAN_STATIC, HPC_PLAN_STEP = 0, 1, 2
HPC_SEG_WHOLE = 1
HPC_DEVCHK_BAD_LENGTH, HPC_DEVCHK_BAD_BLOCK, HPC_DEVCHK_TABLE_TOO_SHORT, \
    HPC_DEVCHK_TIMEOUT, HPC_DEVCHK_CAPACITY = 1, 2, 4, 8, 16

_STATUS_NAMES = {0: "HPC_OK", 1: "HPC_ERR_INVALID_ARG", 2: "HPC_ERR_UNSUPPORTED",
                 3: "HPC_ERR_CUDA", 4: "HPC_ERR_OOM", 5: "HPC_ERR_DEVICE_CHECK"}


class HpcError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class HpcTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4),
                ("scale", ctypes.c_float)]


_lib = None
_lock = threading.Lock()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libhpc_decode.so for sm_103a in-tree (nvcc); returns its path."""
    return _build.build(force=force, verbose=verbose)


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load libhpc_decode.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run paged_gqa_decode_hpc_gb300.build() "
                               "(the CUDA library is required; there is no fallback)")
        try:  # share torch's CUDA runtime when torch is present
            import torch  # noqa: F401
        except Exception:
            pass
        lib = ctypes.CDLL(path)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        pi32, pi64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
        T = ctypes.POINTER(HpcTensor)
        sigs = {
            "hpc_decode_plan": [pi32, i32, i32, ctypes.POINTER(P)],
            "hpc_decode_plan_ex": [pi32, i32, i32, i32, ctypes.POINTER(P)],
            "hpc_decode_plan_compute_ex": [pi32, i32, i32, i32, pi32, i64, pi64],
            "hpc_decode_plan_create": [i32, i32, i32, ctypes.POINTER(P)],
            "hpc_decode_plan_device": [P, i32, i32, P, P],
            "hpc_decode_plan_update": [pi32, i32, i32, P, P],
            "hpc_decode_plan_static": [pi32, i32, i32, i32, i32, ctypes.POINTER(P)],
            "hpc_decode_plan_export": [P, pi32, i64, pi64],
            "hpc_decode_plan_compute": [pi32, i32, i32, pi32, i64, pi64],
            "hpc_decode_plan_static_compute": [pi32, i32, i32, i32, i32, pi32, i64, pi64],
            "hpc_decode_plan_status": [P, pi32],
            "hpc_decode_attn": [T, T, T, T, T, P, T, T, P],
            "hpc_decode_attn_ex": [T, T, T, T, T, P, T, T, ctypes.c_float, P],
            "hpc_device_sm_count": [pi32],
            "hpc_decode_plan_set_timing_events": [P, P, P, P],
            "hpc_decode_attn_noalloc": [T, T, T, T, T, i32, T, T, P, P],
            "hpc_decode_step": [T, T, T, T, T, P, i32, T, T, P],
            "hpc_decode_step_host": [T, T, T, T, T, P, i32, T, T, P],
            "hpc_decode_tc_min_q_len": [i32, pi32],
            "hpc_rope_norm_kv_write": [T, T, T, T, T, T, T, ctypes.c_float, ctypes.c_float,
                                       T, T, T, T, P, P],
            "hpc_extend_attn": [T, T, T, T, T, T, T, T, ctypes.c_float, P, P],
            "hpc_extend_attn_ex": [T, T, T, T, T, T, T, T, ctypes.c_float, i32, P, P],
        }
        for name, args in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.hpc_decode_plan_destroy.argtypes = [P]
        lib.hpc_decode_plan_destroy.restype = None
        lib.hpc_last_error.argtypes = []
        lib.hpc_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def hpc_last_error() -> str:
    return load_library().hpc_last_error().decode()


def _check(status: int):
    if status != HPC_OK:
        raise HpcError(status, hpc_last_error())


def _i32_array(values) -> np.ndarray:
    if hasattr(values, "detach"):
        values = values.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(values, dtype=np.int32))


def _p_i32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    if hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


class Plan:
    """Owner of an hpc_plan_t handle (freed by destroy() or garbage collection)."""

    def __init__(self, handle: ctypes.c_void_p, kind: int):
        self.handle = handle
        self.kind = kind

    def destroy(self):
        if self.handle:
            load_library().hpc_decode_plan_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()


def hpc_decode_plan(seq_lens: Sequence[int], num_sms: int) -> Plan:
    a = _i32_array(seq_lens)
    h = ctypes.c_void_p()
    _check(load_library().hpc_decode_plan(_p_i32(a), a.size, int(num_sms), ctypes.byref(h)))
    return Plan(h, HPC_PLAN_DYNAMIC)


def hpc_decode_plan_ex(seq_lens: Sequence[int], num_sms: int, units_per_tile: int) -> Plan:
    """Balanced plan over (tile, KV head) units when units_per_tile = H_kv."""
    a = _i32_array(seq_lens)
    h = ctypes.c_void_p()
    _check(load_library().hpc_decode_plan_ex(_p_i32(a), a.size, int(num_sms),
                                             int(units_per_tile), ctypes.byref(h)))
    return Plan(h, HPC_PLAN_DYNAMIC)


def hpc_decode_plan_static(seq_lens: Sequence[int], num_sms: int, num_kv_heads: int,
                           num_splits: int = 0) -> Plan:
    a = _i32_array(seq_lens)
    h = ctypes.c_void_p()
    _check(load_library().hpc_decode_plan_static(_p_i32(a), a.size, int(num_sms),
                                                 int(num_kv_heads), int(num_splits),
                                                 ctypes.byref(h)))
    return Plan(h, HPC_PLAN_STATIC)


def hpc_decode_plan_create(max_seqs: int, num_sms: int, num_q_heads: int) -> Plan:
    h = ctypes.c_void_p()
    _check(load_library().hpc_decode_plan_create(int(max_seqs), int(num_sms), int(num_q_heads),
                                                 ctypes.byref(h)))
    return Plan(h, HPC_PLAN_DYNAMIC)


def hpc_decode_plan_device(seq_lens_dev, num_sms: int, plan: Plan, stream=None):
    """seq_lens_dev: int32 CUDA tensor [B]."""
    import torch
    if not seq_lens_dev.is_cuda or seq_lens_dev.dtype != torch.int32 or \
            not seq_lens_dev.is_contiguous():
        raise HpcError(HPC_ERR_INVALID_ARG, "seq_lens_dev must be a contiguous int32 CUDA tensor")
    _check(load_library().hpc_decode_plan_device(
        ctypes.c_void_p(seq_lens_dev.data_ptr()), seq_lens_dev.numel(), int(num_sms),
        plan.handle, _stream_ptr(stream)))


def hpc_decode_plan_update(seq_lens: Sequence[int], num_sms: int, plan: Plan, stream=None):
    a = _i32_array(seq_lens)
    _check(load_library().hpc_decode_plan_update(_p_i32(a), a.size, int(num_sms), plan.handle,
                                                 _stream_ptr(stream)))


def _canonical(fn, *args) -> np.ndarray:
    n = ctypes.c_int64()
    _check(fn(*args, None, 0, ctypes.byref(n)))
    buf = np.zeros(n.value, dtype=np.int32)
    _check(fn(*args, _p_i32(buf), buf.size, ctypes.byref(n)))
    return buf


def hpc_decode_plan_export(plan: Plan) -> np.ndarray:
    return _canonical(load_library().hpc_decode_plan_export, plan.handle)


def hpc_decode_plan_compute(seq_lens: Sequence[int], num_sms: int) -> np.ndarray:
    a = _i32_array(seq_lens)
    return _canonical(load_library().hpc_decode_plan_compute, _p_i32(a), a.size, int(num_sms))


def hpc_decode_plan_compute_ex(seq_lens: Sequence[int], num_sms: int,
                               units_per_tile: int) -> np.ndarray:
    a = _i32_array(seq_lens)
    return _canonical(load_library().hpc_decode_plan_compute_ex, _p_i32(a), a.size, int(num_sms),
                      int(units_per_tile))


def hpc_decode_plan_static_compute(seq_lens: Sequence[int], num_sms: int, num_kv_heads: int,
                                   num_splits: int = 0) -> np.ndarray:
    a = _i32_array(seq_lens)
    return _canonical(load_library().hpc_decode_plan_static_compute, _p_i32(a), a.size,
                      int(num_sms), int(num_kv_heads), int(num_splits))


def hpc_decode_plan_status(plan: Plan) -> int:
    """Device error bits since the last call (0 = none); never raises for them."""
    v = ctypes.c_int32()
    st = load_library().hpc_decode_plan_status(plan.handle, ctypes.byref(v))
    if st not in (HPC_OK, HPC_ERR_DEVICE_CHECK):
        _check(st)
    return int(v.value)


def hpc_decode_plan_destroy(plan: Plan):
    plan.destroy()


def hpc_decode_plan_set_timing_events(plan: Plan, ev_start=None, ev_attn_done=None,
                                      ev_end=None):
    """Record torch.cuda.Event objects (or raw cudaEvent_t ints) around the
    attention and merge kernels of later hpc_decode_attn calls on `plan`."""
    def h(e):
        if e is None:
            return None
        return ctypes.c_void_p(int(e.cuda_event if hasattr(e, "cuda_event") else e))
    _check(load_library().hpc_decode_plan_set_timing_events(plan.handle, h(ev_start),
                                                            h(ev_attn_done), h(ev_end)))


def hpc_decode_tc_min_q_len(q_len: int = -1) -> int:
    """Set the smallest q_len that runs on the tensor-core decode kernel
    (>= 2; above 8: never; 0: the per-dtype defaults, 4 for bf16 and 3 for
    fp8_e4m3 caches; < 0: no change) and return the previous setting."""
    prev = ctypes.c_int32()
    _check(load_library().hpc_decode_tc_min_q_len(int(q_len), ctypes.byref(prev)))
    return int(prev.value)


def hpc_device_sm_count() -> int:
    v = ctypes.c_int32()
    _check(load_library().hpc_device_sm_count(ctypes.byref(v)))
    return int(v.value)


_DTYPES = None


def _dtype_code(t) -> int:
    global _DTYPES
    if _DTYPES is None:
        import torch
        _DTYPES = {torch.bfloat16: HPC_BF16, torch.uint8: HPC_FP8_E4M3,
                   torch.float8_e4m3fn: HPC_FP8_E4M3, torch.float32: HPC_F32,
                   torch.int32: HPC_I32}
    if t.dtype not in _DTYPES:
        raise HpcError(HPC_ERR_INVALID_ARG, f"unsupported tensor dtype {t.dtype}")
    return _DTYPES[t.dtype]


def make_tensor(t, scale: float = 1.0) -> Optional[HpcTensor]:
    """hpc_tensor descriptor of a torch tensor (None -> None)."""
    if t is None:
        return None
    if t.dim() > 4:
        raise HpcError(HPC_ERR_INVALID_ARG, "tensors have at most 4 dimensions")
    d = HpcTensor()
    d.data = ctypes.c_void_p(t.data_ptr())
    d.dtype = _dtype_code(t)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    d.scale = float(scale)
    return d


def hpc_rope_norm_kv_write(q_in, k_in, v_in, seq_lens, block_table, q_norm_weight,
                           k_norm_weight, q_out, k_cache, v_cache, eps: float = 1e-6,
                           rope_base: float = 10000.0, q_out_fp8=None, q_fp8_scale: float = 1.0,
                           k_scale: float = 1.0, v_scale: float = 1.0, device_error=None,
                           stream=None):
    """Fused decode prologue: QK-Norm + RoPE of the new token's q and k, the
    paged KV-cache write of k and v, and optionally an FP8 copy of q."""
    lib = load_library()
    d = [make_tensor(q_in), make_tensor(k_in), make_tensor(v_in), make_tensor(seq_lens),
         make_tensor(block_table), make_tensor(q_norm_weight), make_tensor(k_norm_weight)]
    qo, qf = make_tensor(q_out), make_tensor(q_out_fp8, q_fp8_scale)
    kc, vc = make_tensor(k_cache, k_scale), make_tensor(v_cache, v_scale)
    ref = lambda t: ctypes.byref(t) if t is not None else None
    err = ctypes.c_void_p(device_error.data_ptr()) if device_error is not None else None
    _check(lib.hpc_rope_norm_kv_write(*[ref(t) for t in d], ctypes.c_float(eps),
                                      ctypes.c_float(rope_base), ref(qo), ref(qf), ref(kc),
                                      ref(vc), err, _stream_ptr(stream)))


def hpc_extend_attn(q, k_cache, v_cache, block_table, seq_lens, cu_q_lens, out, lse=None,
                    softmax_scale: Optional[float] = None, device_error=None, stream=None,
                    tiles_per_cta: int = 0, k_scale: float = 1.0, v_scale: float = 1.0):
    """Prefill / extend attention on the tensor cores: q and out are bf16
    [total_q][H_q][128] with the new tokens of sequence b in rows
    cu_q_lens[b] .. cu_q_lens[b+1]-1 (the last positions of its cache);
    lse f32 [total_q][H_q] or None; device_error an int32 CUDA tensor
    receiving HPC_DEVCHK_* bits, or None; tiles_per_cta 0 (automatic), 1 or 2
    query tiles of 128 rows per CTA; k_scale / v_scale the per-tensor scales of
    an e4m3 cache (uint8 / float8_e4m3fn bytes)."""
    lib = load_library()
    tq, tk, tv = make_tensor(q), make_tensor(k_cache, k_scale), make_tensor(v_cache, v_scale)
    tb, ts, tc = make_tensor(block_table), make_tensor(seq_lens), make_tensor(cu_q_lens)
    to, tl = make_tensor(out), make_tensor(lse)
    ref = lambda d: ctypes.byref(d) if d is not None else None
    err = ctypes.c_void_p(device_error.data_ptr()) if device_error is not None else None
    _check(lib.hpc_extend_attn_ex(ref(tq), ref(tk), ref(tv), ref(tb), ref(ts), ref(tc),
                                  ref(to), ref(tl), ctypes.c_float(softmax_scale or -1.0),
                                  int(tiles_per_cta), err, _stream_ptr(stream)))


def hpc_decode_step(q, k_cache, v_cache, block_table, seq_lens, plan: Plan, num_sms: int, out,
                    lse=None, stream=None, k_scale: float = 1.0, v_scale: float = 1.0):
    """One decode step planned on the device (one step-kernel launch for one
    query token per sequence and at most 3072 sequences); `plan` from
    hpc_decode_plan_create, `seq_lens` an int32 CUDA tensor."""
    lib = load_library()
    tq, tk, tv = make_tensor(q), make_tensor(k_cache, k_scale), make_tensor(v_cache, v_scale)
    tb, ts, to = make_tensor(block_table), make_tensor(seq_lens), make_tensor(out)
    tl = make_tensor(lse)
    ref = lambda d: ctypes.byref(d) if d is not None else None
    _check(lib.hpc_decode_step(ref(tq), ref(tk), ref(tv), ref(tb), ref(ts), plan.handle,
                               int(num_sms), ref(to), ref(tl), _stream_ptr(stream)))


def hpc_decode_step_host(q, k_cache, v_cache, block_table, seq_lens, plan: Plan, num_sms: int,
                         out, lse=None, stream=None, k_scale: float = 1.0, v_scale: float = 1.0):
    """hpc_decode_step with q, block_table, seq_lens, out and lse in host
    memory (contiguous CPU tensors; pinned ones make the copies
    asynchronous): the library enqueues the copies in, the step and the
    copies out on `stream`. The caches are CUDA tensors. `out` / `lse` hold
    the result once the stream has passed the copies out."""
    lib = load_library()
    tq, tk, tv = make_tensor(q), make_tensor(k_cache, k_scale), make_tensor(v_cache, v_scale)
    tb, ts, to = make_tensor(block_table), make_tensor(seq_lens), make_tensor(out)
    tl = make_tensor(lse)
    ref = lambda d: ctypes.byref(d) if d is not None else None
    _check(lib.hpc_decode_step_host(ref(tq), ref(tk), ref(tv), ref(tb), ref(ts), plan.handle,
                                    int(num_sms), ref(to), ref(tl), _stream_ptr(stream)))


def hpc_decode_attn(q, k_cache, v_cache, block_table, seq_lens, plan: Plan, out, lse=None,
                    stream=None, k_scale: float = 1.0, v_scale: float = 1.0,
                    softmax_scale: Optional[float] = None):
    """Decode attention into `out` (bf16 [B][H_q][128]) and `lse` (f32 [B][H_q]).

    k_cache/v_cache: bf16, or e4m3 bytes (uint8 / float8_e4m3fn) with
    per-tensor k_scale / v_scale; [num_blocks][H_kv][64][128] (or a permuted
    view of a [num_blocks][64][H_kv][128] cache).
    """
    lib = load_library()
    tq, tk, tv = make_tensor(q), make_tensor(k_cache, k_scale), make_tensor(v_cache, v_scale)
    tb, ts, to = make_tensor(block_table), make_tensor(seq_lens), make_tensor(out)
    tl = make_tensor(lse)
    ref = lambda d: ctypes.byref(d) if d is not None else None
    st = lib.hpc_decode_attn_ex(ref(tq), ref(tk), ref(tv), ref(tb), ref(ts), plan.handle,
                                ref(to), ref(tl),
                                ctypes.c_float(-1.0 if softmax_scale is None else softmax_scale),
                                _stream_ptr(stream))
    _check(st)


def hpc_decode_attn_noalloc(q, k_cache, v_cache, block_table, seq_lens, out, lse=None,
                            num_sms: int = 0, device_error=None, stream=None,
                            k_scale: float = 1.0, v_scale: float = 1.0):
    """One decode step (planner, attention, merge) that allocates nothing.

    For callers that may not call cudaMalloc/cudaFree at this point -- an
    engine's enqueue step or a plugin whose contract forbids allocation, or
    code whose device memory is all owned by a caching allocator. The step's
    scratch is a fixed device array inside the library (limits:
    HPC_NOALLOC_MAX_SEQS sequences, HPC_NOALLOC_MAX_CTAS CTAs,
    HPC_NOALLOC_MAX_Q_HEADS query heads). Calls that overlap on the GPU race
    on that array; keep them on one stream. `device_error`: optional int32
    CUDA tensor of one element receiving device-check bits (zero it first).
    """
    lib = load_library()
    tq, tk, tv = make_tensor(q), make_tensor(k_cache, k_scale), make_tensor(v_cache, v_scale)
    tb, ts, to = make_tensor(block_table), make_tensor(seq_lens), make_tensor(out)
    tl = make_tensor(lse)
    ref = lambda d: ctypes.byref(d) if d is not None else None
    err = ctypes.c_void_p(device_error.data_ptr()) if device_error is not None else None
    _check(lib.hpc_decode_attn_noalloc(ref(tq), ref(tk), ref(tv), ref(tb), ref(ts), int(num_sms),
                                       ref(to), ref(tl), err, _stream_ptr(stream)))
