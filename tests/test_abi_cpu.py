"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every entry point include/hpc_decode.h declares, and its host
planners reproduce the oracle's plans word for word."""
import ctypes
import os
import random
import re

import numpy as np
import pytest

import paged_gqa_decode_hpc_gb300 as hpc
from oracle import plan_ref

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "hpc_decode.h")


@pytest.fixture(scope="module")
def lib():
    hpc.build()
    return hpc.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hpc_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_plan_and_attention_calls():
    names = declared_functions()
    assert "hpc_decode_plan" in names and "hpc_decode_attn" in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def oracle_words(plan, lengths, num_sms, kind, splits=0):
    """Canonical words of an oracle plan (word 7: static split count, or the
    units per tile of a unit plan)."""
    w = [0x48504344, kind, len(lengths), plan.num_parts, plan.num_tiles, len(plan.segments),
         num_sms, splits]
    w += plan.part_seg_off + plan.seq_seg_off
    for s in plan.segments:
        w += [s.seq, s.tile_begin, s.tile_end, 1 if s.whole else 0]
    return np.array(w, dtype=np.int32)


def _cases():
    rng = random.Random(11)
    cases = [([], 4), ([0], 3), ([0, 0, 5], 2), ([37, 64, 200, 1000], 152), ([512] * 64, 152),
             ([131072] + [4096] * 31, 152), ([131072] + [4096] * 31, 148), ([1] * 300, 7),
             ([65] * 3, 1)]
    for _ in range(150):
        B = rng.randint(1, 50)
        lens = [rng.choice([0, rng.randint(1, 64), rng.randint(1, 9000)]) for _ in range(B)]
        cases.append((lens, rng.randint(1, 300)))
    return cases


def test_host_dynamic_plan_matches_oracle(lib):
    for lens, sms in _cases():
        got = hpc.hpc_decode_plan_compute(lens, sms)
        ref = oracle_words(plan_ref.dynamic_plan(lens, sms), lens, sms, 0)
        assert np.array_equal(got, ref), (lens[:8], sms)


def test_host_static_plan_matches_oracle(lib):
    rng = random.Random(3)
    for lens, sms in _cases()[:80]:
        for hkv, splits in [(8, 0), (1, 0), (2, 3), (4, 1), (8, 32)]:
            got = hpc.hpc_decode_plan_static_compute(lens, sms, hkv, splits)
            S = plan_ref.static_split_count(lens, sms, hkv, splits or None)
            ref = oracle_words(plan_ref.static_plan(lens, sms, hkv, splits or None), lens, sms, 1, S)
            assert np.array_equal(got, ref), (lens[:8], sms, hkv, splits)


def test_random_mixed_workload_plan_matches_oracle(lib):
    from paged_gqa_decode_hpc_gb300 import workloads as W
    import torch
    cfg = W.CONFIG_BY_NAME["random_mixed"]
    lens = W.draw_lengths(cfg, torch.Generator().manual_seed(cfg.seed))
    assert len(lens) == 256 and min(lens) >= 16 and max(lens) <= 65536
    got = hpc.hpc_decode_plan_compute(lens, 152)
    assert np.array_equal(got, oracle_words(plan_ref.dynamic_plan(lens, 152), lens, 152, 0))


def test_host_planner_error_statuses(lib):
    n = ctypes.c_int64()
    a = np.array([5, -1], dtype=np.int32)
    p = a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    assert lib.hpc_decode_plan_compute(p, 2, 4, None, 0, ctypes.byref(n)) == hpc.HPC_ERR_INVALID_ARG
    assert "negative" in hpc.hpc_last_error()
    a = np.array([5, 7], dtype=np.int32)
    p = a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    assert lib.hpc_decode_plan_compute(p, 2, 0, None, 0, ctypes.byref(n)) == hpc.HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_plan_compute(None, 2, 4, None, 0, ctypes.byref(n)) == hpc.HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_plan_compute(p, 2, 4, None, 0, None) == hpc.HPC_ERR_INVALID_ARG
    # size query, then a too-small buffer
    assert lib.hpc_decode_plan_compute(p, 2, 4, None, 0, ctypes.byref(n)) == hpc.HPC_OK
    small = np.zeros(n.value - 1, dtype=np.int32)
    assert lib.hpc_decode_plan_compute(p, 2, 4, small.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       small.size, ctypes.byref(n)) == hpc.HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_plan_static_compute(p, 2, 4, 0, 0, None, 0, ctypes.byref(n)) == \
        hpc.HPC_ERR_INVALID_ARG
    # the device-facing calls reject null handles before touching any device
    assert lib.hpc_decode_plan(p, 2, 4, None) == hpc.HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_plan_export(None, None, 0, ctypes.byref(n)) == hpc.HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_attn(None, None, None, None, None, None, None, None, None) == \
        hpc.HPC_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import paged_gqa_decode_hpc_gb300._build as B
    monkeypatch.setattr(hpc, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        hpc.load_library()


def test_host_unit_plans_match_oracle(lib):
    for lens, sms in _cases()[:60]:
        for u in (2, 4, 8):
            got = hpc.hpc_decode_plan_compute_ex(lens, sms, u)
            ref = oracle_words(plan_ref.dynamic_plan(lens, sms, units_per_tile=u), lens, sms, 0, u)
            assert np.array_equal(got, ref), (lens[:8], sms, u)
        assert np.array_equal(hpc.hpc_decode_plan_compute_ex(lens, sms, 1),
                              hpc.hpc_decode_plan_compute(lens, sms))


def test_extend_argument_statuses(lib):
    # hpc_extend_attn validates shapes, dtypes and strides before it touches a
    # device, so host tensors (never dereferenced) exercise every refusal here
    import torch

    def args(hq=16, hkv=2, d=128, kv_dtype=torch.bfloat16, cu_len=3, total=10):
        q = torch.zeros(total, hq, d, dtype=torch.bfloat16)
        kc = torch.zeros(4, hkv, 64, d, dtype=kv_dtype)
        return [q, kc, kc.clone(), torch.zeros(2, 4, dtype=torch.int32),
                torch.tensor([8, 6], dtype=torch.int32),
                torch.tensor([0, 4, 10][:cu_len] + [10] * max(0, cu_len - 3), dtype=torch.int32),
                torch.zeros(total, hq, d, dtype=torch.bfloat16)]

    def status(a, **kw):
        try:
            hpc.hpc_extend_attn(*a, stream=0, **kw)  # an explicit null stream: no torch.cuda
        except hpc.HpcError as e:
            return e.status
        return hpc.HPC_OK

    assert status(args(), tiles_per_cta=3) == hpc.HPC_ERR_INVALID_ARG
    assert status(args(kv_dtype=torch.uint8), k_scale=float("inf")) == hpc.HPC_ERR_INVALID_ARG
    assert "FP8 scales" in hpc.hpc_last_error()
    assert status(args(hq=12, hkv=2)) == hpc.HPC_ERR_UNSUPPORTED           # group != 8
    assert status(args(d=64)) == hpc.HPC_ERR_UNSUPPORTED                   # head_dim
    assert status(args(cu_len=2)) == hpc.HPC_ERR_INVALID_ARG               # cu_q_lens [B+1]
    a = args()
    a[6] = torch.zeros(10, 16, 64, dtype=torch.bfloat16)                    # out shape
    assert status(a) == hpc.HPC_ERR_INVALID_ARG
    a = args()
    a[0] = a[0].float()                                                     # q dtype
    assert status(a) == hpc.HPC_ERR_INVALID_ARG
    assert lib.hpc_extend_attn(None, None, None, None, None, None, None, None,
                               ctypes.c_float(-1.0), None, None) == hpc.HPC_ERR_INVALID_ARG


def test_tensor_core_threshold_setting(lib):
    # process-wide kernel choice for multi-token decode; no device involved
    prev = hpc.hpc_decode_tc_min_q_len(-1)
    try:
        assert hpc.hpc_decode_tc_min_q_len(0) == prev      # 0: the per-dtype defaults
        assert hpc.hpc_decode_tc_min_q_len(-1) == 0
        assert hpc.hpc_decode_tc_min_q_len(6) == 0
        assert hpc.hpc_decode_tc_min_q_len(-5) == 6         # negative: query only
        assert hpc.hpc_decode_tc_min_q_len(9) == 6          # above 8: never
        assert hpc.hpc_decode_tc_min_q_len(-1) == 9
        with pytest.raises(hpc.HpcError) as ei:
            hpc.hpc_decode_tc_min_q_len(1)
        assert ei.value.status == hpc.HPC_ERR_INVALID_ARG
        assert hpc.hpc_decode_tc_min_q_len(-1) == 9         # a refused call changes nothing
        assert lib.hpc_decode_tc_min_q_len(-1, None) == hpc.HPC_OK  # previous may be NULL
    finally:
        hpc.hpc_decode_tc_min_q_len(prev)
