"""GPU parity of multi-token decode (q_len new query tokens per sequence,
causal among themselves, one KV read shared by all of them) against the
fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import assert_parity, device_workload, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hpc.load_library()


def _cfg(hq, hkv, fp8=False):
    return W.Config(98, "mtp", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


def _oracle(w, q):
    return oracle.paged_decode_multi(q, w.k_cache, w.v_cache, w.block_table, w.seq_lens,
                                     num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                                     kv_is_fp8=w.kv_dtype == "fp8_e4m3", k_scale=w.k_scale,
                                     v_scale=w.v_scale)


def run_multi(w, q, plan="step", num_sms=None, splits=0):
    d = device_workload(w)
    qd = q.to("cuda")
    B, T, hq = q.shape[0], q.shape[1], q.shape[2]
    sms = hpc.hpc_device_sm_count()
    num_sms = num_sms or sms
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    if plan == "step":
        p = hpc.hpc_decode_plan_create(max(B, 1), sms, T * hq)
        hpc.hpc_decode_step(qd, d["k"], d["v"], d["bt"], d["sl"], p, num_sms, out, lse,
                            k_scale=w.k_scale, v_scale=w.v_scale)
    else:
        if plan == "host":
            p = hpc.hpc_decode_plan(w.seq_lens.tolist(), num_sms)
        elif plan == "static":
            p = hpc.hpc_decode_plan_static(w.seq_lens.tolist(), num_sms, w.num_kv_heads, splits)
        hpc.hpc_decode_attn(qd, d["k"], d["v"], d["bt"], d["sl"], p, out, lse,
                            k_scale=w.k_scale, v_scale=w.v_scale)
    torch.cuda.synchronize()
    err = hpc.hpc_decode_plan_status(p)
    p.destroy()
    assert err == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


LENS = [1, 2, 3, 63, 64, 65, 130, 700, 3001]


@pytest.mark.parametrize("T,hq,hkv,fp8,plan,sms", [
    (2, 64, 8, False, "step", None),
    (2, 64, 8, True, "step", 7),
    (3, 64, 8, False, "host", None),
    (4, 64, 8, False, "step", None),
    (4, 64, 8, True, "host", 3),
    (8, 64, 8, False, "step", None),
    (2, 8, 1, False, "step", None),
    (3, 8, 1, True, "step", 1),
    (4, 16, 2, False, "host", None),
    (2, 64, 8, False, "static", None),
    (4, 8, 1, False, "static", None),
    (1, 64, 8, False, "step", None),
])
def test_multitoken_parity(T, hq, hkv, fp8, plan, sms):
    w = W.make_workload(_cfg(hq, hkv, fp8), lengths=LENS, seed=61, slack_blocks=2)
    q = W.make_multi_query(w, T, seed=62)
    ref_out, ref_lse = _oracle(w, q)
    out, lse = run_multi(w, q, plan=plan, num_sms=sms)
    assert_parity(out, lse, ref_out, ref_lse, label=f"T={T} hkv={hkv} fp8={fp8} {plan}")


def test_single_token_4d_equals_3d_bitwise():
    w = W.make_workload(_cfg(64, 8), lengths=[5000, 64, 129], seed=63)
    out4, lse4 = run_multi(w, w.q[:, None], plan="host")
    out3, lse3 = run_cuda(w, plan="host")
    assert np.array_equal(out4[:, 0], out3) and np.array_equal(lse4[:, 0], lse3)


def test_skewed_config_two_tokens():
    w = W.make_workload("skewed")
    q = W.make_multi_query(w, 2, seed=64)
    ref_out, ref_lse = _oracle(w, q)
    out, lse = run_multi(w, q)
    assert_parity(out, lse, ref_out, ref_lse, label="skewed q_len 2")


def test_rejects_too_many_tokens():
    w = W.make_workload(_cfg(64, 8), lengths=[100], seed=65)
    d = device_workload(w)
    q = W.make_multi_query(w, 9, seed=66).cuda()
    out = torch.empty_like(q)
    with hpc.hpc_decode_plan([100], 8) as p:
        with pytest.raises(hpc.HpcError) as ei:
            hpc.hpc_decode_attn(q, d["k"], d["v"], d["bt"], d["sl"], p, out)
    assert ei.value.status == hpc.HPC_ERR_UNSUPPORTED
