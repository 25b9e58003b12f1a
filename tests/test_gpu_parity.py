"""GPU parity: the CUDA path (planner + persistent split-KV attention + LSE
merge, called through the C ABI) against the fp64 oracle, element by
element, on seeded inputs with the pages' workload shapes."""
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


def _cfg(hq, hkv, fp8=False):
    return W.Config(90, "case", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


RAGGED = [1, 63, 64, 65, 127, 129, 700, 3001]


def test_tiny_config():
    check_against_oracle(W.make_workload("tiny"))


@pytest.mark.parametrize("num_sms", [1, 7, 64, None])
def test_tiny_config_num_sms_sweep(num_sms):
    check_against_oracle(W.make_workload("tiny"), num_sms=num_sms)


@pytest.mark.parametrize("hq,hkv,fp8", [(64, 8, False), (64, 8, True), (8, 1, False), (8, 1, True),
                                        (16, 2, False), (32, 4, True), (128, 16, False)])
def test_ragged_shapes(hq, hkv, fp8):
    w = W.make_workload(_cfg(hq, hkv, fp8), lengths=RAGGED, seed=5, slack_blocks=7)
    check_against_oracle(w)


@pytest.mark.parametrize("plan", ["host", "device", "static"])
def test_plan_kinds(plan):
    w = W.make_workload(_cfg(64, 8), lengths=[3000, 5, 640, 64, 1999], seed=8)
    check_against_oracle(w, plan=plan)


@pytest.mark.parametrize("splits", [1, 2, 3, 8, 64])
def test_static_split_counts(splits):
    w = W.make_workload(_cfg(64, 8), lengths=[4096, 100, 900], seed=9)
    check_against_oracle(w, plan="static", splits=splits)


def test_sharp_softmax_variant():
    # q scaled x8: peaked attention weights, where errors in the max/rescale path show
    w = W.make_workload(_cfg(64, 8), lengths=[512] * 6 + [37], seed=10, q_scale=8.0)
    check_against_oracle(w)
    w = W.make_workload("tiny", q_scale=8.0)
    check_against_oracle(w)


def test_uniform_config():
    check_against_oracle(W.make_workload("uniform"))


def test_empty_sequences():
    w = W.make_workload(_cfg(64, 8), lengths=[0, 70, 0, 1], seed=3)
    out, lse = check_against_oracle(w)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    w = W.make_workload(_cfg(64, 8), lengths=[0, 0], seed=3)
    out, lse = check_against_oracle(w)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("ns", [2, 7, 8, 9, 16])
def test_merge_at_the_one_warp_path_boundary(ns):
    # a sequence split into exactly ns segments: up to 8 partials are merged
    # by one warp per head, more by four warps per head; next to it a second
    # sequence split into 3
    w = W.make_workload(_cfg(64, 8), lengths=[64 * ns], seed=11)
    check_against_oracle(w, num_sms=ns)
    w = W.make_workload(_cfg(64, 8), lengths=[64 * ns - 5, 192], seed=12)
    check_against_oracle(w, num_sms=ns + 3)
