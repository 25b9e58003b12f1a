"""GPU parity of the tensor-core multi-token decode kernel
(csrc/decode_tc_kernel.cu: one CTA per (KV head, plan part), the q_len x 8
query rows of a KV head on tcgen05) against the fp64 oracle. The kernel
choice is pinned with hpc_decode_tc_min_q_len, so these cases run the
tensor-core path for every q_len >= 2 whatever the default threshold; the
multi-token tests in test_gpu_multitoken.py cover the default choice."""
import contextlib

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


@contextlib.contextmanager
def tc_threshold(q_len):
    prev = hpc.hpc_decode_tc_min_q_len(q_len)
    try:
        yield
    finally:
        hpc.hpc_decode_tc_min_q_len(prev)


def _cfg(hq, hkv, fp8=False):
    return W.Config(97, "mtp-tc", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


def _oracle(w, q):
    return oracle.paged_decode_multi(q, w.k_cache, w.v_cache, w.block_table, w.seq_lens,
                                     num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                                     kv_is_fp8=w.kv_dtype == "fp8_e4m3", k_scale=w.k_scale,
                                     v_scale=w.v_scale)


def run(w, q, plan="step", num_sms=None, threshold=2, d=None):
    d = d or device_workload(w)
    qd = q.to("cuda")
    B, T, hq = q.shape[0], q.shape[1], q.shape[2]
    sms = hpc.hpc_device_sm_count()
    num_sms = num_sms or sms
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    with tc_threshold(threshold):
        if plan == "step":
            p = hpc.hpc_decode_plan_create(max(B, 1), sms, T * hq)
            hpc.hpc_decode_step(qd, d["k"], d["v"], d["bt"], d["sl"], p, num_sms, out, lse,
                                k_scale=w.k_scale, v_scale=w.v_scale)
        else:
            p = hpc.hpc_decode_plan(w.seq_lens.tolist(), num_sms)
            hpc.hpc_decode_attn(qd, d["k"], d["v"], d["bt"], d["sl"], p, out, lse,
                                k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
    err = hpc.hpc_decode_plan_status(p)
    p.destroy()
    assert err == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


# short sequences (fewer positions than new tokens: early tokens see
# nothing), one-block edges, several tiles and a ragged tail
LENS = [1, 2, 3, 5, 63, 64, 65, 127, 129, 700, 3001]


@pytest.mark.parametrize("T,hq,hkv,fp8,plan,sms", [
    (2, 64, 8, False, "step", None),
    (3, 64, 8, True, "step", None),
    (4, 64, 8, False, "host", 19),
    (5, 64, 8, True, "host", 7),
    (6, 8, 1, False, "step", None),
    (7, 16, 2, True, "step", 5),
    (8, 32, 4, False, "host", 1),
    (8, 64, 8, True, "step", None),
    (4, 128, 16, False, "step", None),
    (8, 8, 1, True, "host", 152),
])
def test_tc_parity(T, hq, hkv, fp8, plan, sms):
    w = W.make_workload(_cfg(hq, hkv, fp8), lengths=LENS, seed=71, slack_blocks=2)
    q = W.make_multi_query(w, T, seed=72)
    ref_out, ref_lse = _oracle(w, q)
    out, lse = run(w, q, plan=plan, num_sms=sms)
    assert_parity(out, lse, ref_out, ref_lse, label=f"tc T={T} hkv={hkv} fp8={fp8} {plan}")


@pytest.mark.parametrize("T", [4, 8])
def test_tc_fp8_query_rows_of_any_scale(T):
    # with an e4m3 cache each query row is converted to f16 with its own power
    # of two at the start of each segment; rows scaled by 2^-40 .. 2^3 (a flat
    # to a sharp softmax) must match the oracle under both plans
    w = W.make_workload(_cfg(64, 8, True), lengths=LENS, seed=73, slack_blocks=2)
    q = W.make_multi_query(w, T, seed=74)
    gen = torch.Generator().manual_seed(75)
    pw = torch.randint(-40, 4, q.shape[:3], generator=gen).to(torch.float32)
    q = (q.float() * 4.0 * torch.exp2(pw)[..., None]).to(torch.bfloat16)
    ref_out, ref_lse = _oracle(w, q)
    for plan, sms in (("step", None), ("host", 7)):
        out, lse = run(w, q, plan=plan, num_sms=sms)
        assert_parity(out, lse, ref_out, ref_lse, label=f"tc fp8 T={T} rows 2^-40..2^3 {plan}")


@pytest.mark.parametrize("fp8", [False, True])
def test_tc_one_tile_per_part(fp8):
    # every part one tile: each CTA walks one-tile segments, so Q slots turn
    # over on every tile, and the last tile of a sequence is a segment of its
    # own in which the early tokens see no key (m = -inf partials)
    lens = [129, 65, 2, 191, 64]
    w = W.make_workload(_cfg(64, 8, fp8), lengths=lens, seed=73)
    q = W.make_multi_query(w, 8, seed=74)
    tiles = sum((L + 63) // 64 for L in lens)
    ref_out, ref_lse = _oracle(w, q)
    out, lse = run(w, q, plan="host", num_sms=tiles)
    assert_parity(out, lse, ref_out, ref_lse, label=f"one tile per part fp8={fp8}")


def test_tc_many_segments_per_part():
    # few parts over many short sequences: a CTA walks dozens of segments
    lens = [int(x) for x in np.random.default_rng(75).integers(1, 400, size=120)]
    w = W.make_workload(_cfg(64, 8), lengths=lens, seed=76)
    q = W.make_multi_query(w, 4, seed=77)
    ref_out, ref_lse = _oracle(w, q)
    out, lse = run(w, q, plan="host", num_sms=3)
    assert_parity(out, lse, ref_out, ref_lse, label="many segments per part")


def test_tc_empty_sequences():
    # sequences of length 0 have no tile and no segment: the merge writes
    # out = 0 and lse = -inf
    w = W.make_workload(_cfg(64, 8), lengths=[0, 300, 0, 70], seed=78)
    q = W.make_multi_query(w, 4, seed=79)
    ref_out, ref_lse = _oracle(w, q)
    out, lse = run(w, q, plan="step")
    assert_parity(out, lse, ref_out, ref_lse, label="empty sequences")
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))


def test_threshold_selects_the_tensor_core_plan():
    # hpc_decode_step sizes its plan for the kernel it runs: num_sms / H_kv
    # parts (one CTA per (KV head, part)) for the tensor-core kernel, num_sms
    # for the one-warp-per-token kernel. Plan words: 3 = parts, 6 = the CTA
    # count the plan was sized for.
    w = W.make_workload(_cfg(64, 8), lengths=[12000, 65], seed=80)
    q = W.make_multi_query(w, 4, seed=81).cuda()
    d = device_workload(w)
    sms = hpc.hpc_device_sm_count()
    tiles = (12000 + 63) // 64 + (65 + 63) // 64
    words = {}
    for threshold in (2, 9):
        out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
        p = hpc.hpc_decode_plan_create(2, sms, 4 * 64)
        with tc_threshold(threshold):
            hpc.hpc_decode_step(q, d["k"], d["v"], d["bt"], d["sl"], p, sms, out, lse)
            torch.cuda.synchronize()
        assert hpc.hpc_decode_plan_status(p) == 0
        words[threshold] = hpc.hpc_decode_plan_export(p)
        p.destroy()
    assert words[2][6] == sms // 8 and words[2][3] == min(sms // 8, tiles)
    assert words[9][6] == sms and words[9][3] == min(sms, tiles)


def test_threshold_argument_statuses():
    prev = hpc.hpc_decode_tc_min_q_len(-1)
    try:
        with pytest.raises(hpc.HpcError) as ei:
            hpc.hpc_decode_tc_min_q_len(1)
        assert ei.value.status == hpc.HPC_ERR_INVALID_ARG
        hpc.hpc_decode_tc_min_q_len(5)
        assert hpc.hpc_decode_tc_min_q_len(0) == 5
        assert hpc.hpc_decode_tc_min_q_len(-1) == 0  # the per-dtype defaults
    finally:
        hpc.hpc_decode_tc_min_q_len(prev)


def _subset(w, q, seqs):
    idx = torch.tensor(seqs, dtype=torch.long)
    sub = W.Workload(w.config_name, w.seq_lens[idx].clone(), w.block_table[idx].clone(),
                     w.q[idx].clone(), w.k_cache, w.v_cache, w.k_scale, w.v_scale, w.kv_dtype,
                     w.softmax_scale, w.num_q_heads, w.num_kv_heads)
    return sub, q[idx]


@pytest.mark.parametrize("name,T", [("skewed", 8), ("skewed_fp8", 4)])
def test_tc_full_size_step_sampled(name, T):
    # the full-size skewed batch through hpc_decode_step (the launch the bench
    # times), sampled: the long sequence and two short ones against the oracle
    w = W.make_workload(name)
    q = W.make_multi_query(w, T, seed=82)
    out, lse = run(w, q, plan="step", threshold=0)  # the default choice
    seqs = [0, 1, w.num_seqs - 1]
    sub, qs = _subset(w, q, seqs)
    ref_out, ref_lse = _oracle(sub, qs)
    assert_parity(out[seqs], lse[seqs], ref_out, ref_lse, label=f"{name} q_len {T} sampled")


def test_tc_block_permutation_gives_bit_identical_output():
    # the block table is the only link between positions and physical blocks
    w = W.make_workload(_cfg(64, 8, True), lengths=[700, 64, 3001, 129, 5], seed=83,
                        slack_blocks=5)
    q = W.make_multi_query(w, 4, seed=84)
    out1, lse1 = run(w, q, plan="host", num_sms=19)
    nb = w.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(85))
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt2 = w.block_table.clone()
    m = bt2 >= 0
    bt2[m] = perm[bt2[m].long()].to(torch.int32)
    w.k_cache, w.v_cache, w.block_table = k2, v2, bt2
    out2, lse2 = run(w, q, plan="host", num_sms=19)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


@pytest.mark.parametrize("fp8", [False, True])
def test_tc_permuted_view_cache_layout(fp8):
    # a [blocks][64][H_kv][128] cache passed as a [blocks][H_kv][64][128] view
    w = W.make_workload(_cfg(64, 8, fp8), lengths=[300, 64, 1000], seed=86)
    q = W.make_multi_query(w, 8, seed=87)
    ref = run(w, q)
    d = device_workload(w)
    kt = d["k"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    vt = d["v"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert kt.stride(1) == 128 and kt.stride(2) == 8 * 128
    d["k"], d["v"] = kt, vt
    got = run(w, q, d=d)
    assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])


def test_tc_cuda_graph_capture_of_a_step():
    # planner kernel, tensor-core kernel and merge captured once, replayed
    sms = hpc.hpc_device_sm_count()
    w = W.make_workload(_cfg(64, 8), lengths=[2000, 64, 700], seed=88)
    q = W.make_multi_query(w, 4, seed=89)
    d = device_workload(w)
    qd = q.cuda()
    out = torch.zeros(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(q.shape[:3], dtype=torch.float32, device="cuda")
    p = hpc.hpc_decode_plan_create(3, sms, 4 * 64)
    s = torch.cuda.Stream()
    with tc_threshold(2):
        with torch.cuda.stream(s):  # first call outside the capture
            hpc.hpc_decode_step(qd, d["k"], d["v"], d["bt"], d["sl"], p, sms, out, lse, stream=s)
        torch.cuda.synchronize()
        out.zero_()
        lse.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            hpc.hpc_decode_step(qd, d["k"], d["v"], d["bt"], d["sl"], p, sms, out, lse, stream=s)
        g.replay()
        torch.cuda.synchronize()
    assert hpc.hpc_decode_plan_status(p) == 0
    p.destroy()
    ref_out, ref_lse = _oracle(w, q)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                  label="tc graph replay")
