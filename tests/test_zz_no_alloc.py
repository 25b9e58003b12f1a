"""The allocation-free decode entry point (hpc_decode_attn_noalloc).

Some callers may not allocate device memory when they run a decode step: an
inference engine's enqueue step or a plugin whose contract forbids it, or a
framework whose device memory all belongs to a caching allocator, where a
cudaMalloc/cudaFree would synchronise the device or fail under memory
pressure. This entry point keeps its plan and partial results in a fixed
device array inside the library instead.

These tests call it through the C ABI. It runs the same plan rule (the
device planner with one unit per tile) and the same attention and merge
kernels as hpc_decode_attn with a host-built plan for the same CTA count, so
its output must be bit-identical to that call's, on consecutive calls, with
and without a caller-supplied error word, below the device's SM count, and
for a small batch after a larger one (stale plan or partial words left in
the shared array must not leak into a later call). One call is also
compared with the fp64 oracle at the parity tolerances. The file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import assert_parity, device_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hpc.load_library()


def _workload(kv_dtype, lens, seed):
    return W.make_workload(W.Config(95, "noalloc", 64, 8, kv_dtype), lengths=lens, seed=seed)


def _reference(w, d, num_sms):
    """hpc_decode_attn with a host-built plan for num_sms CTAs."""
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    with hpc.hpc_decode_plan(w.seq_lens.tolist(), num_sms) as p:
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, lse,
                            k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        assert hpc.hpc_decode_plan_status(p) == 0
    return out, lse


def _noalloc(w, d, num_sms=0, with_err=True):
    out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(w.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda") if with_err else None
    hpc.hpc_decode_attn_noalloc(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, lse,
                                num_sms=num_sms, device_error=err, k_scale=w.k_scale,
                                v_scale=w.v_scale)
    torch.cuda.synchronize()
    if err is not None:
        assert int(err.item()) == 0, f"device check bits {int(err.item())}"
    return out, lse


def _identical(got, ref, label):
    assert torch.equal(got[0], ref[0]), f"{label}: out differs from hpc_decode_attn"
    assert torch.equal(got[1], ref[1]), f"{label}: lse differs from hpc_decode_attn"


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_noalloc_is_bit_identical_to_hpc_decode_attn_on_two_calls(kv_dtype):
    lens = [9000, 0, 1, 64, 65, 700, 3001] + [130] * 33
    w = _workload(kv_dtype, lens, 31)
    d = device_workload(w)
    sms = hpc.hpc_device_sm_count()
    ref = _reference(w, d, sms)
    for call in range(2):
        _identical(_noalloc(w, d), ref, f"call {call}")
    # the first call also against the fp64 oracle
    ref_out, ref_lse = oracle.decode_workload(w)
    got = _noalloc(w, d)
    assert_parity(got[0].double().cpu().numpy(), got[1].double().cpu().numpy(), ref_out, ref_lse,
                  label=f"noalloc {kv_dtype} vs oracle")


def test_noalloc_without_error_word_and_below_the_sm_count():
    w = _workload("bf16", [4097, 5, 640, 1, 0, 2000, 64, 77] * 4, 33)
    d = device_workload(w)
    # device_error=None: the library's own error word, cleared on the stream
    _identical(_noalloc(w, d, with_err=False), _reference(w, d, hpc.hpc_device_sm_count()),
               "no error word")
    # 37 CTAs: fewer parts than the scratch's fixed 160, so the part and
    # segment offsets of the plan words differ from a full-size plan's
    _identical(_noalloc(w, d, num_sms=37), _reference(w, d, 37), "37 CTAs")
    _identical(_noalloc(w, d, num_sms=1), _reference(w, d, 1), "1 CTA")


def test_noalloc_small_batch_after_a_large_one():
    big = _workload("bf16", [50 + 211 * i for i in range(40)], 34)
    small = _workload("bf16", [3000, 1, 64, 129, 700], 35)
    db, ds = device_workload(big), device_workload(small)
    sms = hpc.hpc_device_sm_count()
    ref_big, ref_small = _reference(big, db, sms), _reference(small, ds, sms)
    _identical(_noalloc(big, db), ref_big, "40 sequences")
    _identical(_noalloc(small, ds), ref_small, "5 sequences after 40")
    _identical(_noalloc(big, db), ref_big, "40 sequences after 5")


def test_noalloc_rejects_sizes_beyond_its_limit():
    cfg = W.Config(96, "noalloc", 8, 1, "bf16")
    w = W.make_workload(cfg, lengths=[3] * 257, seed=32)
    d = device_workload(w)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hpc.HpcError) as ei:
        hpc.hpc_decode_attn_noalloc(d["q"], d["k"], d["v"], d["bt"], d["sl"], out)
    assert ei.value.status == hpc.HPC_ERR_INVALID_ARG and "limit" in str(ei.value)
    with pytest.raises(hpc.HpcError) as ei:
        hpc.hpc_decode_attn_noalloc(d["q"][:4], d["k"], d["v"], d["bt"][:4], d["sl"][:4],
                                    out[:4], num_sms=161)
    assert ei.value.status == hpc.HPC_ERR_INVALID_ARG and "limit" in str(ei.value)


def test_noalloc_rejected_call_enqueues_nothing():
    """A call refused by an argument check (a strided seq_lens, a multi-token
    q) launches nothing: the caller's error word stays untouched and the
    next valid call is still bit-identical to hpc_decode_attn."""
    w = _workload("bf16", [300, 40, 2000, 1], 36)
    d = device_workload(w)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    err = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    sl2 = torch.stack([d["sl"], d["sl"]], dim=1)[:, 0]  # stride 2
    with pytest.raises(hpc.HpcError) as ei:
        hpc.hpc_decode_attn_noalloc(d["q"], d["k"], d["v"], d["bt"], sl2, out,
                                    device_error=err)
    assert ei.value.status == hpc.HPC_ERR_INVALID_ARG
    q4 = d["q"].unsqueeze(1).contiguous()
    with pytest.raises(hpc.HpcError) as ei:
        hpc.hpc_decode_attn_noalloc(q4, d["k"], d["v"], d["bt"], d["sl"], out.unsqueeze(1),
                                    device_error=err)
    assert ei.value.status == hpc.HPC_ERR_INVALID_ARG and "one query token" in str(ei.value)
    torch.cuda.synchronize()
    assert int(err.item()) == 12345
    _identical(_noalloc(w, d), _reference(w, d, hpc.hpc_device_sm_count()), "after refusals")
