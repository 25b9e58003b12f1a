"""hpc_decode_step: the kernels plan the step themselves. With one query token
per sequence the step kernel runs alone (head-major units, static parts plus a
pool of chunks, in-kernel merges of split pairs): its output must match the
oracle, repeat bit for bit although pool chunks go to whichever CTA asks first,
and its per-owner records must equal the oracle's step plan. Batches above the
in-kernel limit run the planner kernel, the attention kernel and the merge,
whose plan words equal the host planner's."""
import numpy as np
import pytest
import torch

import oracle
from oracle import plan_ref
import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import assert_parity, device_workload, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hpc.load_library()


def _cfg(hq=64, hkv=8, fp8=False):
    return W.Config(92, "step", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


def run_plan_ex(w, units, num_sms):
    d = device_workload(w)
    B, hq = w.q.shape[0], w.q.shape[1]
    out = torch.full((B, hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
    with hpc.hpc_decode_plan_ex(w.seq_lens.tolist(), num_sms, units) as p:
        hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, lse,
                            k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        assert hpc.hpc_decode_plan_status(p) == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def run_step(w, d=None, num_sms=None, plan=None):
    d = d or device_workload(w)
    sms_all = hpc.hpc_device_sm_count()
    num_sms = num_sms or sms_all
    B, hq = w.q.shape[0], w.q.shape[1]
    own = plan is None
    if own:
        plan = hpc.hpc_decode_plan_create(max(B, 1), sms_all, hq)
    out = torch.full((B, hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
    hpc.hpc_decode_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], plan, num_sms, out, lse,
                        k_scale=w.k_scale, v_scale=w.v_scale)
    torch.cuda.synchronize()
    err = hpc.hpc_decode_plan_status(plan)
    words = hpc.hpc_decode_plan_export(plan)
    if own:
        plan.destroy()
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), words, err


def check_step_records(words, lens, num_sms, hkv, runs=1):
    """The step's exported work list against the oracle's step plan: header,
    then per owner (static parts, then pool chunks) its unit range, its number
    of pieces and how many times a CTA ran it since the plan was created."""
    sp = plan_ref.step_plan(list(lens), num_sms, hkv)
    assert words[1] == hpc.HPC_PLAN_STEP
    assert list(words[2:8]) == [len(lens), sp.num_parts, sp.num_units, sp.num_chunks, num_sms,
                                hkv]
    rec = np.asarray(words[8:]).reshape(-1, 4)
    owners = sp.num_parts + sp.num_chunks
    assert rec.shape[0] == owners
    pieces = np.zeros(owners, dtype=np.int64)
    for pc in sp.pieces:
        pieces[pc.owner] += 1
    assert np.array_equal(rec[:, 0], sp.owner_start[:-1])
    assert np.array_equal(rec[:, 1], sp.owner_start[1:])
    assert np.array_equal(rec[:, 2], pieces)
    assert np.all(rec[:, 3] == runs), "every part and every pool chunk runs exactly once per step"


@pytest.mark.parametrize("lens,hq,hkv,fp8,sms", [
    ([37, 64, 200, 1000], 8, 1, False, None),
    ([37, 64, 200, 1000], 8, 1, False, 1),
    ([1, 63, 64, 65, 127, 129, 700, 3001], 64, 8, False, 7),
    ([1, 63, 64, 65, 127, 129, 700, 3001], 64, 8, True, None),
    ([0, 5, 0, 300, 4096, 0], 16, 2, False, 3),
    ([700, 65, 3001], 128, 16, False, None),
    ([9000, 1, 2, 130], 32, 4, True, 2),
    ([64] * 40 + [6400], 64, 8, False, 37),
])
def test_step_parity_and_plan_records(lens, hq, hkv, fp8, sms):
    w = W.make_workload(_cfg(hq, hkv, fp8), lengths=lens, seed=41)
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse, words, err = run_step(w, num_sms=sms)
    assert err == 0
    assert_parity(out, lse, ref_out, ref_lse, label=f"step {lens[:4]}")
    n = sms or hpc.hpc_device_sm_count()
    check_step_records(words, lens, n, hkv)
    # pool chunks go to whichever CTA asks first, yet every piece's arithmetic
    # is fixed, so a second step gives the same bits
    out2, lse2, _, err2 = run_step(w, num_sms=sms)
    assert err2 == 0
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_step_skewed_config():
    w = W.make_workload("skewed")
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse, words, err = run_step(w)
    assert err == 0
    assert_parity(out, lse, ref_out, ref_lse, label="step skewed")
    check_step_records(words, w.seq_lens.tolist(), hpc.hpc_device_sm_count(), 8)


@pytest.mark.parametrize("fp8", [False, True])
def test_step_bit_identical_under_block_permutation(fp8):
    """The same logical cache stored under another permutation of physical
    blocks gives the same bits (the step reads tiles only through the table)."""
    lens = [3000, 65, 1, 640, 129]
    w = W.make_workload(_cfg(64, 8, fp8), lengths=lens, seed=52)
    out, lse, _, err = run_step(w, num_sms=19)
    assert err == 0
    nb = w.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(53))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    bt2 = torch.where(w.block_table >= 0, inv[w.block_table.clamp(min=0).long()],
                      w.block_table.long()).to(torch.int32)
    w2 = W.Workload(w.config_name, w.seq_lens, bt2,
                    w.q, w.k_cache[perm], w.v_cache[perm], w.k_scale, w.v_scale, w.kv_dtype,
                    w.softmax_scale, w.num_q_heads, w.num_kv_heads)
    out2, lse2, _, err2 = run_step(w2, num_sms=19)
    assert err2 == 0
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("fp8", [False, True])
def test_step_token_major_cache_layout(fp8):
    """A [blocks][64][H_kv][128] (token-major) cache passed as a
    [blocks][H_kv][64][128] view: the step kernel's copies take the other
    coordinate order and give the same bits as the head-major cache."""
    w = W.make_workload(_cfg(64, 8, fp8), lengths=[300, 64, 1000, 0, 4097], seed=54)
    out, lse, _, err = run_step(w, num_sms=23)
    assert err == 0
    d = device_workload(w)
    for k in ("k", "v"):
        d[k] = d[k].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert d["k"].stride(1) == 128 and d["k"].stride(2) == 8 * 128
    out2, lse2, _, err2 = run_step(w, d=d, num_sms=23)
    assert err2 == 0
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    ref_out, ref_lse = oracle.decode_workload(w)
    assert_parity(out2, lse2, ref_out, ref_lse, label="step, token-major cache")


def test_step_without_lse():
    """lse is optional: the output bits are those of a step that writes it."""
    w = W.make_workload(_cfg(64, 8), lengths=[2000, 7, 640, 0, 129], seed=55)
    out, _, _, err = run_step(w, num_sms=11)
    assert err == 0
    d = device_workload(w)
    plan = hpc.hpc_decode_plan_create(8, hpc.hpc_device_sm_count(), 64)
    o2 = torch.full((5, 64, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    hpc.hpc_decode_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], plan, 11, o2, None)
    torch.cuda.synchronize()
    assert hpc.hpc_decode_plan_status(plan) == 0
    plan.destroy()
    assert np.array_equal(out, o2.double().cpu().numpy())


def test_step_records_count_every_run():
    lens = [4096] * 6 + [70]
    w = W.make_workload(_cfg(64, 8), lengths=lens, seed=54)
    d = device_workload(w)
    sms = hpc.hpc_device_sm_count()
    plan = hpc.hpc_decode_plan_create(len(lens), sms, 64)
    for _ in range(3):
        run_step(w, d=d, plan=plan)
    check_step_records(hpc.hpc_decode_plan_export(plan), lens, sms, 8, runs=3)
    plan.destroy()


def test_step_at_the_in_kernel_sequence_limit():
    # 3072 sequences, the most the step kernel plans in shared memory (its
    # prefix array fills the dynamic shared memory it is configured for),
    # with empty sequences among them: parity, the oracle's work list, and
    # the same bits on a second step
    lens = [(i * 53) % 300 for i in range(3072)]
    w = W.make_workload(_cfg(8, 1), lengths=lens, seed=44)
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse, words, err = run_step(w)
    assert err == 0
    assert_parity(out, lse, ref_out, ref_lse, label="step 3072 seqs")
    check_step_records(words, lens, hpc.hpc_device_sm_count(), 1)
    out2, lse2, _, err2 = run_step(w)
    assert err2 == 0 and np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_step_many_sequences_uses_the_planner_kernel():
    lens = [(i * 37) % 150 + 1 for i in range(3500)]  # above the in-kernel limit
    w = W.make_workload(_cfg(8, 1), lengths=lens, seed=42)
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse, words, err = run_step(w)
    assert err == 0
    assert_parity(out, lse, ref_out, ref_lse, label="step 3500 seqs")
    assert np.array_equal(words, hpc.hpc_decode_plan_compute(lens, hpc.hpc_device_sm_count()))


def test_step_negative_length_sets_check():
    w = W.make_workload(_cfg(), lengths=[100, 50], seed=43)
    d = device_workload(w)
    d["sl"][1] = -5
    out, lse, words, err = run_step(w, d=d)
    assert err & hpc.HPC_DEVCHK_BAD_LENGTH
    assert words[3] == 0 and words[5] == 0  # empty plan
    # a length whose (tile, KV head) units could wrap the plan's 32-bit scan
    # (2^30 tokens x 8 KV heads) is refused the same way, before any copy:
    # every output row is 0 and every lse -inf
    d["sl"][1] = 1 << 30
    out, lse, words, err = run_step(w, d=d)
    assert err & hpc.HPC_DEVCHK_BAD_LENGTH
    assert words[3] == 0 and words[5] == 0
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_step_reuses_one_plan_across_batches_and_graph_capture():
    sms = hpc.hpc_device_sm_count()
    plan = hpc.hpc_decode_plan_create(16, sms, 64)
    for seed, lens in [(44, [3000, 64, 1]), (45, [512] * 16), (46, [9000])]:
        w = W.make_workload(_cfg(), lengths=lens, seed=seed)
        ref_out, ref_lse = oracle.decode_workload(w)
        out, lse, words, err = run_step(w, plan=plan)
        assert err == 0
        assert_parity(out, lse, ref_out, ref_lse)
    w = W.make_workload(_cfg(), lengths=[2000, 640, 7], seed=47)
    d = device_workload(w)
    out = torch.zeros(w.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(w.q.shape[:2], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        hpc.hpc_decode_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], plan, sms, out, lse, stream=s)
    torch.cuda.synchronize()
    out.zero_(); lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hpc.hpc_decode_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], plan, sms, out, lse, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert hpc.hpc_decode_plan_status(plan) == 0
    ref_out, ref_lse = oracle.decode_workload(w)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse)
    plan.destroy()


@pytest.mark.parametrize("lens,fp8,sms", [
    ([512] * 64, False, None), ([512] * 64, True, 7), ([1, 63, 64, 65, 700, 3001, 0], False, 3),
    ([131072] + [4096] * 31, False, None)])
def test_unit_plans_parity(lens, fp8, sms):
    w = W.make_workload(_cfg(64, 8, fp8), lengths=lens, seed=48)
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse = run_plan_ex(w, 8, sms or hpc.hpc_device_sm_count())
    assert_parity(out, lse, ref_out, ref_lse, label=f"unit plan {lens[:3]}")


def test_unit_plan_rejected_for_other_layouts():
    w = W.make_workload(_cfg(16, 2), lengths=[100, 300], seed=49)
    with pytest.raises(hpc.HpcError) as ei:
        run_plan_ex(w, 2, 16)  # 2 KV heads: warps split tiles, unit plans unsupported
    assert ei.value.status == hpc.HPC_ERR_UNSUPPORTED


def test_step_many_sequences_unit_plan_through_the_planner_kernel():
    lens = [(i * 53) % 200 + 1 for i in range(3300)]
    w = W.make_workload(_cfg(64, 8), lengths=lens, seed=50)
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse, words, err = run_step(w)
    assert err == 0
    assert_parity(out, lse, ref_out, ref_lse, label="step 3300 seqs, unit plan")
    assert np.array_equal(words, hpc.hpc_decode_plan_compute_ex(lens, hpc.hpc_device_sm_count(), 8))


@pytest.mark.parametrize("sms", [5, 8, 9, 13])
def test_unit_plan_merges_with_partial_head_segments(sms):
    # 24 (tile, KV head) units over sms parts: segments start and end inside a
    # tile, so some heads have empty partials, on both sides of the 8-partial
    # boundary between the merge's one-warp and four-warp paths
    w = W.make_workload(_cfg(64, 8), lengths=[192], seed=51)
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse = run_plan_ex(w, 8, sms)
    assert_parity(out, lse, ref_out, ref_lse, label=f"unit plan over {sms} parts")


@pytest.mark.parametrize("name", ["tiny", "uniform", "skewed_fp8", "random_mixed"])
def test_step_full_size_configs(name):
    # the launch configuration bench.py times (hpc_decode_step: one launch of
    # the step kernel, which plans, computes and merges the step), at each
    # config's full size, element by element against the fp64 oracle
    w = W.make_workload(name)
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse, words, err = run_step(w)
    assert err == 0
    assert_parity(out, lse, ref_out, ref_lse, label=f"step {name}")


@pytest.mark.parametrize("fp8", [False, True])
def test_step_host_entry_matches_the_device_step(fp8):
    # hpc_decode_step_host: the batch and the results in pinned host memory,
    # copied by the library around the same step -- the same bits as
    # hpc_decode_step, and the oracle's values; a larger batch regrows the
    # plan's staging area, a smaller one reuses it
    sms = hpc.hpc_device_sm_count()
    plan = hpc.hpc_decode_plan_create(16, sms, 64)
    for lens in ([300, 5, 0, 2000, 64], [1, 63, 64, 65, 127, 129, 700, 3001, 40, 9000], [77]):
        w = W.make_workload(_cfg(64, 8, fp8), lengths=lens, seed=45)
        d = device_workload(w)
        out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
        hpc.hpc_decode_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], plan, sms, out, lse,
                            k_scale=w.k_scale, v_scale=w.v_scale)
        pin = lambda t: t.clone().pin_memory()
        q_h, bt_h, sl_h = pin(w.q), pin(w.block_table), pin(w.seq_lens)
        out_h = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
        lse_h = torch.full(w.q.shape[:2], float("nan"), dtype=torch.float32).pin_memory()
        hpc.hpc_decode_step_host(q_h, d["k"], d["v"], bt_h, sl_h, plan, sms, out_h, lse_h,
                                 k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        assert torch.equal(out_h, out.cpu()) and torch.equal(lse_h, lse.cpu())
        ref_out, ref_lse = oracle.decode_workload(w)
        assert_parity(out_h.double().numpy(), lse_h.double().numpy(), ref_out, ref_lse,
                      label=f"host entry {lens[:3]}")
    # a strided (non-dense) host tensor is refused before any copy
    with pytest.raises(hpc.HpcError) as e:
        hpc.hpc_decode_step_host(q_h[:, ::2], d["k"], d["v"], bt_h, sl_h, plan, sms,
                                 out_h[:, ::2], lse_h)
    assert e.value.status == hpc.HPC_ERR_INVALID_ARG
    plan.destroy()
