"""The allocation-free decode entry point (hpc_decode_attn_noalloc).

Some callers may not allocate device memory when they run a decode step: an
inference engine's enqueue step or a plugin whose contract forbids it, or a
framework whose device memory all belongs to a caching allocator, where a
cudaMalloc/cudaFree would synchronise the device or fail under memory
pressure. This entry point keeps its plan and partial results in a fixed
device array inside the library instead. These tests call it through the C
ABI and compare it with the ordinary entry point (hpc_decode_attn with a
host-built plan), twice in a row, within the parity tolerances used for the
oracle comparisons. The file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import LSE_ATOL, OUT_ATOL, OUT_RTOL, device_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hpc.load_library()


def _reference(w, d):
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    with hpc.hpc_decode_plan(w.seq_lens.tolist(), hpc.hpc_device_sm_count()) as p:
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, lse,
                            k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        assert hpc.hpc_decode_plan_status(p) == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def _close(out, lse, ref_out, ref_lse):
    assert np.all(np.abs(out - ref_out) <= OUT_ATOL + OUT_RTOL * np.abs(ref_out))
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(np.abs(lse[fin] - ref_lse[fin]) <= LSE_ATOL)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_noalloc_matches_hpc_decode_attn_on_two_calls(kv_dtype):
    cfg = W.Config(95, "noalloc", 64, 8, kv_dtype)
    lens = [9000, 0, 1, 64, 65, 700, 3001] + [130] * 33
    w = W.make_workload(cfg, lengths=lens, seed=31)
    d = device_workload(w)
    ref_out, ref_lse = _reference(w, d)
    for call in range(2):
        out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full(w.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        hpc.hpc_decode_attn_noalloc(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, lse,
                                    device_error=err, k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device check bits {int(err.item())}"
        _close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse)


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
