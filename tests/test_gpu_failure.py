"""Failure detection on the GPU without a fault: the bounded waits of the
attention, tensor-core decode and extend kernels must end a call whose data
never arrives with an
error status, and leave the context usable.

A child process sets HPC_DECODE_TEST_WITHHOLD_COPIES=1 (the producer warp
issues no copies, so every consumer waits on a word nothing sets) and a
200 ms wait limit, runs one step, and reports the device-check bits, the
time the step took and whether CUDA still works afterwards. No trap, no bad
address, no endless loop is involved."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import assert_parity, device_workload

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import oracle
import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import assert_parity, device_workload
hpc.load_library()
res = {}
for hkv, hq in ((8, 64), (1, 8)):  # one-token steps: the step kernel
    w = W.make_workload(W.Config(99, "fail", hq, hkv, "bf16"), lengths=[3000, 64, 700], seed=71)
    d = device_workload(w)
    sms = hpc.hpc_device_sm_count()
    plan = hpc.hpc_decode_plan_create(3, sms, hq)
    out = torch.zeros(w.q.shape, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    hpc.hpc_decode_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], plan, sms, out)
    bits = hpc.hpc_decode_plan_status(plan)  # synchronises
    res[str(hkv)] = {"bits": bits, "seconds": time.time() - t0}
    # the failed step left the plan's arrival counters and pool at zero: a
    # normal step on the same plan is right
    os.environ["HPC_DECODE_TEST_WITHHOLD_COPIES"] = "0"
    lse = torch.zeros(w.q.shape[:2], dtype=torch.float32, device="cuda")
    hpc.hpc_decode_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], plan, sms, out, lse)
    ok_bits = hpc.hpc_decode_plan_status(plan)
    ref_out, ref_lse = oracle.decode_workload(w)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse)
    res[str(hkv)]["recovered"] = ok_bits == 0
    os.environ["HPC_DECODE_TEST_WITHHOLD_COPIES"] = "1"
    plan.destroy()
# the tensor-core multi-token decode kernel (q_len 4), BF16 and FP8 caches
for kvd in ("bf16", "fp8_e4m3"):
    w = W.make_workload(W.Config(99, "fail", 64, 8, kvd), lengths=[3000, 64, 700], seed=74)
    d = device_workload(w)
    q = W.make_multi_query(w, 4, seed=75).cuda()
    sms = hpc.hpc_device_sm_count()
    plan = hpc.hpc_decode_plan_create(3, sms, 4 * 64)
    out = torch.zeros(q.shape, dtype=torch.bfloat16, device="cuda")
    prev = hpc.hpc_decode_tc_min_q_len(2)
    torch.cuda.synchronize()
    t0 = time.time()
    hpc.hpc_decode_step(q, d["k"], d["v"], d["bt"], d["sl"], plan, sms, out,
                        k_scale=w.k_scale, v_scale=w.v_scale)
    bits = hpc.hpc_decode_plan_status(plan)  # synchronises
    hpc.hpc_decode_tc_min_q_len(prev)
    res[f"tc_{kvd}"] = {"bits": bits, "seconds": time.time() - t0}
    plan.destroy()
# the extend kernel (tcgen05, TMA), BF16 and FP8 caches, one and two query tiles per CTA
for kvd in ("bf16", "fp8_e4m3"):
    w = W.make_workload(W.Config(99, "fail", 64, 8, kvd), lengths=[600, 70], seed=72)
    q, cu = W.make_extend_query(w, [600, 33], seed=73)
    for tpc in (1, 2):
        out = torch.zeros(q.shape, dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        t0 = time.time()
        hpc.hpc_extend_attn(q.cuda(), w.k_cache.cuda(), w.v_cache.cuda(), w.block_table.cuda(),
                            w.seq_lens.cuda(), cu.cuda(), out, device_error=err, tiles_per_cta=tpc,
                            k_scale=w.k_scale, v_scale=w.v_scale)
        bits = int(err.item())  # synchronises
        res[f"extend_{kvd}_{tpc}"] = {"bits": bits, "seconds": time.time() - t0}
# the context still works
res["usable"] = float(torch.arange(1000, device="cuda", dtype=torch.float32).sum().item()) == 499500.0
print(json.dumps(res))
"""


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hpc.load_library()


def test_withheld_copies_end_in_a_timeout_status_and_a_usable_context():
    env = dict(os.environ, HPC_DECODE_TEST_WITHHOLD_COPIES="1", HPC_DECODE_WAIT_LIMIT_MS="200")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("8", "1", "tc_bf16", "tc_fp8_e4m3", "extend_bf16_1", "extend_bf16_2",
                "extend_fp8_e4m3_1", "extend_fp8_e4m3_2"):
        assert res[key]["bits"] & hpc.HPC_DEVCHK_TIMEOUT, res
        assert res[key]["seconds"] < 30, res
    assert res["8"]["recovered"] and res["1"]["recovered"], res
    assert res["usable"]
    # and this process, without the switch, still computes the right answer
    w = W.make_workload(W.Config(99, "fail", 64, 8, "bf16"), lengths=[3000, 64, 700], seed=71)
    d = device_workload(w)
    sms = hpc.hpc_device_sm_count()
    plan = hpc.hpc_decode_plan_create(3, sms, 64)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    hpc.hpc_decode_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], plan, sms, out, lse)
    assert hpc.hpc_decode_plan_status(plan) == 0
    plan.destroy()
    ref_out, ref_lse = oracle.decode_workload(w)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse)
