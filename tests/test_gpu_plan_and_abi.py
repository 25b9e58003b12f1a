"""GPU checks of the planner and the ABI: the device planner equals the host
planner word for word, outputs are bit-identical under a permutation of the
physical blocks and across repeated calls, bad inputs become error statuses
or device-check bits (never a fault), and the capacity plan works under
host updates and CUDA-graph capture."""
import ctypes
import random

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import assert_parity, check_against_oracle, device_workload, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hpc.load_library()


def _cfg(hq=64, hkv=8, fp8=False):
    return W.Config(91, "case", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


def _length_vectors():
    rng = random.Random(4)
    out = [[], [0], [0, 0, 3], [37, 64, 200, 1000], [512] * 64, [131072] + [4096] * 31,
           [1] * 2000]
    for _ in range(40):
        B = rng.randint(1, 300)
        out.append([rng.choice([0, rng.randint(1, 64), rng.randint(1, 20000)]) for _ in range(B)])
    return out


def test_device_plan_equals_host_plan_bitwise():
    sms_full = hpc.hpc_device_sm_count()
    for lens in _length_vectors():
        for sms in (1, 7, 64, sms_full):
            B = len(lens)
            p = hpc.hpc_decode_plan_create(max(B, 1), sms_full, 64)
            sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
            hpc.hpc_decode_plan_device(sl, sms, p)
            got = hpc.hpc_decode_plan_export(p)
            ref = hpc.hpc_decode_plan_compute(lens, sms)
            assert np.array_equal(got, ref), (B, sms)
            assert hpc.hpc_decode_plan_status(p) == 0
            p.destroy()
            if B:
                with hpc.hpc_decode_plan(lens, sms) as ph:
                    assert np.array_equal(hpc.hpc_decode_plan_export(ph), ref)


def test_device_plan_negative_length_sets_check():
    p = hpc.hpc_decode_plan_create(4, 8, 64)
    hpc.hpc_decode_plan_device(torch.tensor([5, -3, 7], dtype=torch.int32, device="cuda"), 8, p)
    assert hpc.hpc_decode_plan_status(p) & hpc.HPC_DEVCHK_BAD_LENGTH
    words = hpc.hpc_decode_plan_export(p)
    assert words[3] == 0 and words[5] == 0  # empty plan
    p.destroy()


def test_block_permutation_gives_bit_identical_output():
    w = W.make_workload(_cfg(), lengths=[700, 64, 3001, 129, 5], seed=12, slack_blocks=5)
    out1, lse1 = run_cuda(w)
    nb = w.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(99))
    k2 = torch.empty_like(w.k_cache); v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache; v2[perm] = w.v_cache
    bt2 = w.block_table.clone()
    m = bt2 >= 0
    bt2[m] = perm[bt2[m].long()].to(torch.int32)
    w.k_cache, w.v_cache, w.block_table = k2, v2, bt2
    out2, lse2 = run_cuda(w)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_repeated_calls_are_deterministic():
    w = W.make_workload(_cfg(fp8=True), lengths=[5000, 3, 640], seed=13)
    d = device_workload(w)
    a = run_cuda(w, d=d, plan="device")
    b = run_cuda(w, d=d, plan="device")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_skewed_config():
    check_against_oracle(W.make_workload("skewed"))


def test_skewed_fp8_config():
    check_against_oracle(W.make_workload("skewed_fp8"))


def test_skewed_config_static_rule():
    check_against_oracle(W.make_workload("skewed"), plan="static")


@pytest.mark.slow
def test_random_mixed_config():
    check_against_oracle(W.make_workload("random_mixed"), plan="device")


def test_permuted_view_cache_layout():
    # a [blocks][64][H_kv][128] cache passed as a [blocks][H_kv][64][128] view
    w = W.make_workload(_cfg(), lengths=[300, 64, 1000], seed=14)
    ref = run_cuda(w)
    d = device_workload(w)
    kt = d["k"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    vt = d["v"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert kt.stride(1) == 128 and kt.stride(2) == 8 * 128
    d["k"], d["v"] = kt, vt
    got = run_cuda(w, d=d)
    assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])


def test_lse_is_optional():
    w = W.make_workload(_cfg(), lengths=[300, 5000], seed=15)
    d = device_workload(w)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    with hpc.hpc_decode_plan(w.seq_lens.tolist(), hpc.hpc_device_sm_count()) as p:
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, None)
        torch.cuda.synchronize()
    ref_out, _ = oracle.decode_workload(w)
    assert np.allclose(out.double().cpu().numpy(), ref_out, atol=1e-2, rtol=1e-2)


def test_bad_block_id_sets_device_check_not_fault():
    w = W.make_workload(_cfg(), lengths=[300, 200], seed=16)
    d = device_workload(w)
    d["bt"][1, 2] = w.k_cache.shape[0] + 5  # out of range
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    with hpc.hpc_decode_plan(w.seq_lens.tolist(), 16) as p:
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, None)
        assert hpc.hpc_decode_plan_status(p) & hpc.HPC_DEVCHK_BAD_BLOCK
    torch.cuda.synchronize()  # the context is still usable


def test_lengths_differing_from_plan_set_device_check():
    w = W.make_workload(_cfg(), lengths=[300, 200], seed=17)
    d = device_workload(w)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    with hpc.hpc_decode_plan([300, 100], 16) as p:  # plan built from other lengths
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, None)
        assert hpc.hpc_decode_plan_status(p) & hpc.HPC_DEVCHK_BAD_LENGTH


def _expect_status(status, fn):
    with pytest.raises(hpc.HpcError) as ei:
        fn()
    assert ei.value.status == status, str(ei.value)


def test_abi_rejects_bad_arguments():
    w = W.make_workload(_cfg(), lengths=[100, 70], seed=18)
    d = device_workload(w)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    with hpc.hpc_decode_plan(w.seq_lens.tolist(), 16) as p:
        call = lambda **kw: hpc.hpc_decode_attn(kw.get("q", d["q"]), kw.get("k", d["k"]),
                                                kw.get("v", d["v"]), kw.get("bt", d["bt"]),
                                                kw.get("sl", d["sl"]), kw.get("p", p),
                                                kw.get("out", out), kw.get("lse", lse))
        _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: call(q=d["q"].float()))
        _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: call(out=out[:1]))
        _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: call(lse=lse[:, :5]))
        _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: call(v=d["v"][:-1]))
        _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: call(bt=d["bt"].to(torch.int64).to(torch.float32)))
        _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: call(sl=d["sl"][:1]))
        _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: call(v=d["v"].to(torch.uint8)))
        _expect_status(hpc.HPC_ERR_UNSUPPORTED, lambda: call(q=d["q"][:, :, :64].contiguous(),
                                                             out=out[:, :, :64].contiguous(),
                                                             k=d["k"][..., :64].contiguous(),
                                                             v=d["v"][..., :64].contiguous()))
        _expect_status(hpc.HPC_ERR_UNSUPPORTED, lambda: call(q=d["q"][:, :32].contiguous(),
                                                             out=out[:, :32].contiguous(),
                                                             lse=lse[:, :32].contiguous()))
        _expect_status(hpc.HPC_ERR_UNSUPPORTED, lambda: call(k=d["k"][:, :, :32].contiguous(),
                                                             v=d["v"][:, :, :32].contiguous()))
    with hpc.hpc_decode_plan([100, 70, 5], 16) as p3:
        _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: hpc.hpc_decode_attn(
            d["q"], d["k"], d["v"], d["bt"], d["sl"], p3, out, lse))
    _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: hpc.hpc_decode_plan([5, -1], 8))
    _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: hpc.hpc_decode_plan([5], 0))
    _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: hpc.hpc_decode_plan_create(-1, 8, 64))
    small = hpc.hpc_decode_plan_create(2, 8, 64)
    _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: hpc.hpc_decode_plan_update([1, 2, 3], 8, small))
    _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: hpc.hpc_decode_plan_update([1, 2], 9, small))
    _expect_status(hpc.HPC_ERR_INVALID_ARG, lambda: hpc.hpc_decode_plan_device(
        torch.zeros(3, dtype=torch.int32, device="cuda"), 8, small))
    small.destroy()


def test_capacity_plan_with_host_updates():
    sms = hpc.hpc_device_sm_count()
    p = hpc.hpc_decode_plan_create(8, sms, 64)
    for seed, lens in [(20, [300, 5, 4096]), (21, [64] * 8), (22, [1, 2, 3])]:
        w = W.make_workload(_cfg(), lengths=lens, seed=seed)
        d = device_workload(w)
        out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
        hpc.hpc_decode_plan_update(lens, sms, p)
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, lse)
        torch.cuda.synchronize()
        assert hpc.hpc_decode_plan_status(p) == 0
        ref_out, ref_lse = oracle.decode_workload(w)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse)
    p.destroy()


def test_cuda_graph_capture_of_a_step():
    sms = hpc.hpc_device_sm_count()
    w = W.make_workload(_cfg(), lengths=[2000, 64, 700], seed=23)
    d = device_workload(w)
    out = torch.zeros(w.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(w.q.shape[:2], dtype=torch.float32, device="cuda")
    p = hpc.hpc_decode_plan_create(3, sms, 64)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        hpc.hpc_decode_plan_device(d["sl"], sms, p, s)  # first call outside capture
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, lse, stream=s)
    torch.cuda.synchronize()
    out.zero_(); lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hpc.hpc_decode_plan_device(d["sl"], sms, p, s)
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, lse, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert hpc.hpc_decode_plan_status(p) == 0
    ref_out, ref_lse = oracle.decode_workload(w)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse)
    p.destroy()
