"""GPU parity of prefill / extend attention (hpc_extend_attn, the tcgen05
kernel) against the fp64 oracle: ragged batches, prefill from an empty
cache, extends over long contexts, sharp softmax, block-permutation and
cache-layout invariance, sampled rows of a large prefill, and the argument
and device checks."""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hpc.load_library()


def _cfg(hq, hkv, fp8=False):
    return W.Config(95, "extend", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


def run_extend(w, q, cu, k=None, v=None, bt=None, softmax_scale=None, expect_err=0, tpc=0):
    dev = "cuda"
    qd = q.to(dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    hpc.hpc_extend_attn(qd, w.k_cache.to(dev) if k is None else k,
                        w.v_cache.to(dev) if v is None else v,
                        w.block_table.to(dev) if bt is None else bt, w.seq_lens.to(dev),
                        cu.to(dev), out, lse, softmax_scale=softmax_scale, device_error=err,
                        tiles_per_cta=tpc, k_scale=w.k_scale, v_scale=w.v_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == expect_err, f"device check bits {int(err.item())}"
    return out, lse


def _oracle(w, q, cu, rows=None, softmax_scale=None):
    return oracle.paged_extend(q, w.k_cache, w.v_cache, w.block_table, w.seq_lens, cu,
                               num_kv_heads=w.num_kv_heads,
                               softmax_scale=softmax_scale or w.softmax_scale,
                               kv_is_fp8=w.kv_dtype == "fp8_e4m3", k_scale=w.k_scale,
                               v_scale=w.v_scale, rows=rows)


CASES = [
    # (H_q, H_kv, lengths, new tokens per sequence, fp8_e4m3 cache)
    (8, 1, [64], [64], False),                                   # one prefill tile row block
    (16, 2, [100], [100], False),                                # prefill with a ragged tail
    (64, 8, [512], [512], False),                                # q512 prefill
    (64, 8, [70, 9, 130, 64, 1000], [70, 3, 66, 1, 17], False),  # ragged prefill / extend mix
    (64, 8, [4096], [100], False),                               # extend over a long context
    (32, 4, [50, 300, 17], [0, 20, 17], False),                  # a sequence with no new token
    (128, 16, [200, 65], [33, 65], False),
    (64, 8, [512], [512], True),                                 # q512 prefill, e4m3 cache
    (16, 2, [70, 9, 130, 1000], [70, 3, 66, 17], True),          # ragged mix, e4m3 cache
    (64, 8, [4096], [100], True),                                # long extend, e4m3 cache
]


@pytest.mark.parametrize("hq,hkv,lens,qn,fp8", CASES)
def test_matches_oracle(hq, hkv, lens, qn, fp8):
    w = W.make_workload(_cfg(hq, hkv, fp8), lengths=lens, seed=40 + len(lens))
    q, cu = W.make_extend_query(w, qn, seed=41)
    ref_out, ref_lse = _oracle(w, q, cu)
    outs = []
    for tpc in (1, 2):  # one or two 128-row query tiles per CTA
        out, lse = run_extend(w, q, cu, tpc=tpc)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      label=f"extend {lens} {qn} fp8={fp8} tiles/CTA {tpc}")
        outs.append((out, lse))
    # the CTA shape changes which rows share a CTA, not any row's arithmetic
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_sharp_softmax_and_explicit_scale():
    # q x 8 makes the softmax peaked, so row maxima jump between tiles and the
    # O rescale path runs; a second scale checks the scale argument
    w = W.make_workload(_cfg(64, 8), lengths=[700, 129], seed=42)
    q, cu = W.make_extend_query(w, [300, 129], seed=43, q_scale=8.0)
    for scale, tpc in ((None, 1), (None, 2), (0.05, 2)):
        out, lse = run_extend(w, q, cu, softmax_scale=scale, tpc=tpc)
        ref_out, ref_lse = _oracle(w, q, cu, softmax_scale=scale)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      label=f"sharp scale={scale} tiles/CTA {tpc}")


def test_fp8_cache_query_rows_of_any_scale():
    # with an e4m3 cache each query row is converted to f16 with its own power
    # of two; rows scaled by 2^-40 .. 2^3 (a flat to a sharp softmax; larger
    # logits would put the lse beyond fp32's absolute 1e-3) must still match
    # the oracle, and a whole q scaled by a power of two gives the same bits as
    # the same scale in the softmax scale argument
    w = W.make_workload(_cfg(64, 8, True), lengths=[700, 129], seed=48)
    q, cu = W.make_extend_query(w, [300, 129], seed=49, q_scale=4.0)
    gen = torch.Generator().manual_seed(50)
    pw = torch.randint(-40, 4, q.shape[:2], generator=gen).to(torch.float32)
    qs = (q.float() * torch.exp2(pw)[..., None]).to(torch.bfloat16)
    for tpc in (1, 2):
        out, lse = run_extend(w, qs, cu, tpc=tpc)
        ref_out, ref_lse = _oracle(w, qs, cu)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      label=f"fp8 cache, rows scaled 2^-40..2^3, tiles/CTA {tpc}")
    q3 = (q.float() * 8.0).to(torch.bfloat16)  # exact: a power of two
    out1, _ = run_extend(w, q, cu, softmax_scale=w.softmax_scale * 8.0)
    out2, _ = run_extend(w, q3, cu)
    assert torch.equal(out1, out2)


def test_block_permutation_and_layout_invariance():
    w = W.make_workload(_cfg(64, 8), lengths=[300, 77], seed=44, slack_blocks=5)
    q, cu = W.make_extend_query(w, [120, 40], seed=45)
    out1, lse1 = run_extend(w, q, cu)
    # same logical cache under another physical placement
    nb = w.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(46))
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt2 = torch.where(w.block_table >= 0, perm[w.block_table.clamp(min=0).long()].int(),
                      w.block_table)
    out2, lse2 = run_extend(w, q, cu, k=k2.cuda(), v=v2.cuda(), bt=bt2.cuda())
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    # [blocks][64][kv heads][128] storage passed as a permuted view
    ks = w.k_cache.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    vs = w.v_cache.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    out3, lse3 = run_extend(w, q, cu, k=ks, v=vs)
    assert torch.equal(out1, out3) and torch.equal(lse1, lse3)


@pytest.mark.parametrize("fp8", [False, True])
def test_large_prefill_sampled_rows(fp8):
    # 4 x 4096-token prefill at the decode configs' head shape: every row finite,
    # 64 sampled rows (first, last and tile edges included) against the oracle
    lens = [4096] * 4
    w = W.make_workload(_cfg(64, 8, fp8), lengths=lens, seed=47)
    q, cu = W.make_extend_query(w, lens, seed=48)
    out, lse = run_extend(w, q, cu)   # automatic: two query tiles per CTA at this size
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    out1, lse1 = run_extend(w, q, cu, tpc=1)
    assert torch.equal(out, out1) and torch.equal(lse, lse1)
    g = torch.Generator().manual_seed(49)
    rows = sorted(set([0, 15, 16, 4095, 4096, 8191, 12287, 16383] +
                      torch.randint(0, 16384, (56,), generator=g).tolist()))
    ref_out, ref_lse = _oracle(w, q, cu, rows=rows)
    assert_parity(out[rows].double().cpu().numpy(), lse[rows].double().cpu().numpy(), ref_out,
                  ref_lse, label=f"prefill 4 x 4096 sampled fp8={fp8}")


def test_decode_shape_equals_decode_kernel():
    # one new token per sequence is a decode: same answer as the decode path
    w = W.make_workload(_cfg(64, 8), lengths=[1, 64, 65, 3000], seed=50)
    cu = torch.arange(5, dtype=torch.int32)
    out, lse = run_extend(w, w.q, cu)
    ref_out, ref_lse = oracle.decode_workload(w)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                  label="extend as decode")


def test_argument_and_device_checks():
    w = W.make_workload(_cfg(16, 2), lengths=[40, 80], seed=51)
    q, cu = W.make_extend_query(w, [10, 20], seed=52)
    dev = "cuda"
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    args = [q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_table.to(dev),
            w.seq_lens.to(dev), cu.to(dev), out]
    # an fp8 cache needs finite per-tensor scales
    k8 = torch.zeros(w.k_cache.shape, dtype=torch.uint8, device=dev)
    with pytest.raises(hpc.HpcError) as e:
        hpc.hpc_extend_attn(args[0], k8, k8, *args[3:], k_scale=float("inf"))
    assert e.value.status == hpc.HPC_ERR_INVALID_ARG
    with pytest.raises(hpc.HpcError) as e:
        hpc.hpc_extend_attn(*args, tiles_per_cta=3)
    assert e.value.status == hpc.HPC_ERR_INVALID_ARG
    # cu_q_lens of the wrong length
    with pytest.raises(hpc.HpcError) as e:
        hpc.hpc_extend_attn(*args[:5], cu[:2].to(dev), out)
    assert e.value.status == hpc.HPC_ERR_INVALID_ARG
    # more new tokens than positions: flagged on the device, rows left alone
    sl = torch.tensor([40, 15], dtype=torch.int32)
    w_bad = W.Workload(w.config_name, sl, w.block_table, w.q, w.k_cache, w.v_cache, 1.0, 1.0,
                       "bf16", w.softmax_scale, 16, 2)
    run_extend(w_bad, q, cu, expect_err=hpc.HPC_DEVCHK_BAD_LENGTH)
    # a block id out of range reads zeros and is flagged
    bt = w.block_table.clone()
    bt[1, 0] = 10_000
    run_extend(w, q, cu, bt=bt.to(dev), expect_err=hpc.HPC_DEVCHK_BAD_BLOCK)


def test_many_ragged_sequences():
    # 100 sequences (the tile lookup scans cu_q_lens in chunks of 32), new-token
    # counts 0..40 with contexts up to 3000, both CTA shapes
    g = torch.Generator().manual_seed(53)
    qn = torch.randint(0, 41, (100,), generator=g).tolist()
    lens = [n + int(torch.randint(0, 3000, (1,), generator=g)) for n in qn]
    lens = [max(L, 1) for L in lens]
    w = W.make_workload(_cfg(16, 2), lengths=lens, seed=54)
    q, cu = W.make_extend_query(w, qn, seed=55)
    ref_out, ref_lse = _oracle(w, q, cu)
    for tpc in (1, 2):
        out, lse = run_extend(w, q, cu, tpc=tpc)
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      label=f"100 ragged sequences tiles/CTA {tpc}")


def test_extend_over_long_context():
    # 16 new tokens after 65520 cached ones: 1024 K/V tiles per CTA
    w = W.make_workload(_cfg(64, 8), lengths=[65536], seed=56)
    q, cu = W.make_extend_query(w, [16], seed=57)
    out, lse = run_extend(w, q, cu)
    ref_out, ref_lse = _oracle(w, q, cu)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                  label="extend 16 over 65536")


def test_bench_extend_shape_sampled_rows():
    # the bench's 8 x (8192 context + 512 new tokens) extend, in the launch
    # configuration the bench times (automatic CTA shape): 48 sampled rows
    lens, qn = [8704] * 8, [512] * 8
    w = W.make_workload(_cfg(64, 8), lengths=lens, seed=9000)
    q, cu = W.make_extend_query(w, qn, seed=9001)
    out, lse = run_extend(w, q, cu)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    g = torch.Generator().manual_seed(58)
    rows = sorted(set([0, 511, 512, 4095, 4096 - 15] +
                      torch.randint(0, 4096, (43,), generator=g).tolist()))
    ref_out, ref_lse = _oracle(w, q, cu, rows=rows)
    assert_parity(out[rows].double().cpu().numpy(), lse[rows].double().cpu().numpy(), ref_out,
                  ref_lse, label="extend 8 x (8192 + 512) sampled")


@pytest.mark.parametrize("fp8", [False, True])
def test_strided_outputs_and_untouched_neighbours(fp8):
    # out and lse as views with padded heads: a full 16-token tile leaves
    # through a TMA store over out's own strides, a partial tile row by row,
    # and nothing outside the views changes (a full tile's box never reaches
    # the next sequence's rows, a partial tile's rows are never stored as a box)
    w = W.make_workload(_cfg(64, 8, fp8), lengths=[70, 512, 40], seed=52)
    q, cu = W.make_extend_query(w, [70, 512, 33], seed=53)
    ref_out, ref_lse = _oracle(w, q, cu)
    total, hq = q.shape[0], q.shape[1]
    dev = "cuda"
    big = torch.full((total, hq + 8, 128), 7.0, dtype=torch.bfloat16, device=dev)
    lse_big = torch.full((total, hq + 8), 7.0, dtype=torch.float32, device=dev)
    out, lse = big[:, 4:4 + hq, :], lse_big[:, 4:4 + hq]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for tpc in (1, 2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        hpc.hpc_extend_attn(q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev),
                            w.block_table.to(dev), w.seq_lens.to(dev), cu.to(dev), out, lse,
                            device_error=err, tiles_per_cta=tpc, k_scale=w.k_scale,
                            v_scale=w.v_scale)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                      label=f"strided out, tiles/CTA {tpc}")
        assert torch.all(big[:, :4] == 7) and torch.all(big[:, 4 + hq:] == 7)
        assert torch.all(lse_big[:, :4] == 7) and torch.all(lse_big[:, 4 + hq:] == 7)
