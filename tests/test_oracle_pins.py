"""Pins for the fp64 oracle: checks against facts fixed by the format
definitions, closed forms, invariants and an independent brute force.

Each pin is chosen so that a plausible slip in the oracle (a wrong kv-head
map, a dropped scale, a mis-indexed block/slot, k paired with the wrong v,
a wrong FP8 exponent bias) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_hpc_gb300 import workloads as W

D = 128


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _mk(lengths, hq, hkv, seed=0, fp8=False, slack=0):
    cfg = W.Config(99, "t", hq, hkv, "fp8_e4m3" if fp8 else "bf16", lengths=list(lengths))
    return W.make_workload(cfg, seed=seed, slack_blocks=slack)


def _run(w, **kw):
    return oracle.decode_workload(w, **kw)


# ---------------------------------------------------------------- formats
def test_bf16_decode_all_codes_match_torch():
    codes = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(c) for c in range(1 << 16)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7F and 0xFF only
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0xB8, -1.0), (0x7E, 448.0), (0xFE, -448.0),
    (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x40, 2.0), (0x3C, 1.5)])
def test_e4m3_format_definition_values(code, value):
    # OCP 8-bit floating point spec, E4M3: bias 7, max normal 448, min subnormal 2^-9
    assert oracle.e4m3_to_f64(code) == value


# ------------------------------------------------------- brute force
def _brute(w):
    """Dense gather + naive softmax (no max shift) in long double."""
    q = w.q.to(torch.float64).numpy()
    if w.kv_dtype == "fp8_e4m3":
        kf = w.k_cache.view(torch.float8_e4m3fn).to(torch.float64).numpy() * w.k_scale
        vf = w.v_cache.view(torch.float8_e4m3fn).to(torch.float64).numpy() * w.v_scale
    else:
        kf = w.k_cache.to(torch.float64).numpy()
        vf = w.v_cache.to(torch.float64).numpy()
    B, hq, _ = q.shape
    G = hq // w.num_kv_heads
    out = np.zeros((B, hq, D), dtype=np.longdouble)
    lse = np.zeros((B, hq), dtype=np.longdouble)
    for b in range(B):
        L = int(w.seq_lens[b])
        t = np.arange(L)
        blk = w.block_table[b].numpy()[t // 64]
        for j in range(hq):
            h = j // G
            K = kf[blk, h, t % 64, :].astype(np.longdouble)
            V = vf[blk, h, t % 64, :].astype(np.longdouble)
            s = (K @ q[b, j].astype(np.longdouble)) * np.longdouble(w.softmax_scale)
            e = np.exp(s)
            out[b, j] = (e[:, None] * V).sum(0) / e.sum()
            lse[b, j] = np.log(e.sum())
    return out.astype(np.float64), lse.astype(np.float64)


@pytest.mark.parametrize("lengths,hq,hkv,fp8", [
    ([1, 2, 63, 64, 65, 130], 8, 1, False),
    ([37, 64, 200], 16, 2, False),
    ([5, 129, 300], 8, 4, True),
    ([70, 1], 32, 4, True),
])
def test_oracle_matches_bruteforce(lengths, hq, hkv, fp8):
    w = _mk(lengths, hq, hkv, seed=7, fp8=fp8, slack=3)
    out, lse = _run(w, num_threads=3)
    bo, bl = _brute(w)
    np.testing.assert_allclose(out, bo, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- closed forms
def test_identical_v_rows_per_kv_head_give_that_row():
    # V rows are constant per kv head, distinct across kv heads: catches a
    # wrong query-head -> kv-head map (h = j // G).
    w = _mk([1, 77, 640], 16, 4, seed=3)
    rows = torch.randn(4, D, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    w.v_cache[:] = rows[None, :, None, :]
    out, _ = _run(w)
    G = 4
    for j in range(16):
        np.testing.assert_allclose(out[:, j, :], np.broadcast_to(
            rows[j // G].to(torch.float64).numpy(), (3, D)), rtol=1e-14, atol=1e-14)


def test_length_one_gives_its_v_and_scaled_score():
    w = _mk([1, 1], 8, 2, seed=11)
    out, lse = _run(w)
    G = 4
    for b in range(2):
        blk = int(w.block_table[b, 0])
        for j in range(8):
            k0 = w.k_cache[blk, j // G, 0].to(torch.float64).numpy()
            v0 = w.v_cache[blk, j // G, 0].to(torch.float64).numpy()
            qv = w.q[b, j].to(torch.float64).numpy()
            np.testing.assert_array_equal(out[b, j], v0)
            assert lse[b, j] == pytest.approx(w.softmax_scale * float(qv @ k0), rel=1e-13, abs=1e-13)


def test_zero_query_gives_mean_of_v_and_log_length():
    w = _mk([3, 64, 65, 1000], 8, 1, seed=2)
    w.q.zero_()
    # v_t = logical token index (exact in bf16 up to 256): mean = (L - 1) / 2
    for b, L in enumerate(w.seq_lens.tolist()):
        for t in range(L):
            w.v_cache[int(w.block_table[b, t // 64]), 0, t % 64, :] = float(t % 256)
    out, lse = _run(w)
    for b, L in enumerate(w.seq_lens.tolist()):
        expect = np.mean([t % 256 for t in range(L)])
        np.testing.assert_allclose(out[b], expect, rtol=1e-13)
        np.testing.assert_allclose(lse[b], math.log(L), rtol=1e-14)


def test_sharp_query_closed_form():
    # K rows one-hot (k_t = c * e_t), q = a * e_{t*}: only token t* scores
    # a*c*scale, the others score 0, so
    #   out = (e^x v_{t*} + sum_{t != t*} v_t) / (e^x + L - 1),  lse = ln(e^x + L - 1).
    L, tstar, a, c = 100, 41, 16.0, 4.0
    w = _mk([L], 8, 1, seed=9)
    w.k_cache.zero_()
    blk = [int(w.block_table[0, i]) for i in range(2)]
    for t in range(L):
        w.k_cache[blk[t // 64], 0, t % 64, t] = c
    w.q.zero_()
    w.q[0, :, tstar] = a
    out, lse = _run(w)
    x = a * c * w.softmax_scale
    V = np.stack([w.v_cache[blk[t // 64], 0, t % 64].to(torch.float64).numpy() for t in range(L)])
    expect = (math.exp(x) * V[tstar] + V.sum(0) - V[tstar]) / (math.exp(x) + L - 1)
    for j in range(8):
        np.testing.assert_allclose(out[0, j], expect, rtol=1e-12, atol=1e-14)
        assert lse[0, j] == pytest.approx(math.log(math.exp(x) + L - 1), rel=1e-14)


def test_two_token_hand_value():
    # q = e_0, k_0 = 2 e_0, k_1 = -1 e_0, v_0 = e_1, v_1 = 3 e_1, scale 1/sqrt(128):
    # s = (2, -1) / sqrt(128); out[1] = (e^{s0} + 3 e^{s1}) / (e^{s0} + e^{s1}).
    w = _mk([2], 8, 1, seed=1)
    w.q.zero_(); w.k_cache.zero_(); w.v_cache.zero_()
    blk = int(w.block_table[0, 0])
    w.q[0, :, 0] = 1.0
    w.k_cache[blk, 0, 0, 0] = 2.0
    w.k_cache[blk, 0, 1, 0] = -1.0
    w.v_cache[blk, 0, 0, 1] = 1.0
    w.v_cache[blk, 0, 1, 1] = 3.0
    out, lse = _run(w)
    s0, s1 = 2 / math.sqrt(128), -1 / math.sqrt(128)
    assert out[0, 0, 1] == pytest.approx((math.exp(s0) + 3 * math.exp(s1)) / (math.exp(s0) + math.exp(s1)), rel=1e-15)
    assert out[0, 0, 0] == 0.0 and out[0, 0, 2] == 0.0
    assert lse[0, 0] == pytest.approx(math.log(math.exp(s0) + math.exp(s1)), rel=1e-15)


def test_block_permutation_invariance_is_exact():
    w = _mk([37, 64, 200, 1000], 8, 1, seed=4)
    out1, lse1 = _run(w)
    # move every logical block to a new physical id under a second permutation
    nb = w.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(77))
    k2 = torch.empty_like(w.k_cache); v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache; v2[perm] = w.v_cache
    bt2 = w.block_table.clone()
    valid = bt2 >= 0
    bt2[valid] = perm[bt2[valid].long()].to(torch.int32)
    w.k_cache, w.v_cache, w.block_table = k2, v2, bt2
    out2, lse2 = _run(w)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_fp8_constant_v_and_scale():
    w = _mk([50, 300], 8, 2, seed=6, fp8=True)
    w.v_cache[:] = 0x3C  # 1.5
    w.v_scale = 0.25
    out, _ = _run(w)
    np.testing.assert_allclose(out, np.full_like(out, 1.5 * 0.25), rtol=1e-14)


def test_fp8_key_scale_enters_logits():
    # identical K bytes scaled by k_scale: lse = ln(L) + scale*k_scale*q.k
    w = _mk([10], 8, 1, seed=6, fp8=True)
    w.k_cache[:] = 0x38  # 1.0
    w.k_scale = 0.5
    out, lse = _run(w)
    for j in range(8):
        qsum = float(w.q[0, j].to(torch.float64).sum())
        assert lse[0, j] == pytest.approx(math.log(10) + w.softmax_scale * 0.5 * qsum, rel=1e-13, abs=1e-13)


def test_empty_sequence():
    w = _mk([0, 5, 0], 8, 1, seed=8)
    out, lse = _run(w)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    assert np.all(np.isfinite(lse[1]))


def test_thread_count_does_not_change_result():
    w = _mk([100, 3, 900, 64], 16, 2, seed=12)
    a = _run(w, num_threads=1)
    b = _run(w, num_threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rejects_bad_arguments():
    w = _mk([10], 8, 1)
    w.seq_lens[0] = -1
    with pytest.raises(RuntimeError):
        _run(w)
    w.seq_lens[0] = 65  # needs 2 blocks, table has 1 column
    with pytest.raises(RuntimeError):
        _run(w)
