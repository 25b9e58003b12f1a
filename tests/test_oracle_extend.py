"""Pins for the prefill / extend oracle (ragged new tokens per sequence over
the paged cache, causal among themselves): a dense masked-softmax brute force
over whole score matrices, the first token of a prefill returns v_0 exactly,
keys after a token's causal limit never reach it, one new token is a plain
decode, and ragged packing equals the uniform multi-token form."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_hpc_gb300 import workloads as W


def _cfg(hq, hkv, fp8=False):
    return W.Config(96, "extend", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


def _extend(w, q, cu):
    return oracle.paged_extend(q, w.k_cache, w.v_cache, w.block_table, w.seq_lens, cu,
                               num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                               kv_is_fp8=w.kv_dtype == "fp8_e4m3", k_scale=w.k_scale,
                               v_scale=w.v_scale)


def _kv_f64(w):
    if w.kv_dtype == "fp8_e4m3":
        return (w.k_cache.view(torch.float8_e4m3fn).to(torch.float64).numpy() * w.k_scale,
                w.v_cache.view(torch.float8_e4m3fn).to(torch.float64).numpy() * w.v_scale)
    return w.k_cache.to(torch.float64).numpy(), w.v_cache.to(torch.float64).numpy()


@pytest.mark.parametrize("fp8", [False, True])
def test_matches_dense_score_matrix(fp8):
    # whole (new tokens x positions) score matrices with a triangular mask
    lens, qn = [70, 9, 130, 64], [70, 3, 66, 0]
    w = W.make_workload(_cfg(16, 2, fp8), lengths=lens, seed=21)
    q, cu = W.make_extend_query(w, qn, seed=22)
    out, lse = _extend(w, q, cu)
    kf, vf = _kv_f64(w)
    qf = q.to(torch.float64).numpy()
    assert out.shape == (sum(qn), 16, 128) and lse.shape == (sum(qn), 16)
    for b, (L, n) in enumerate(zip(lens, qn)):
        if n == 0:
            continue
        pos = np.arange(L)
        blk = w.block_table[b].numpy()[pos // 64]
        rows = slice(int(cu[b]), int(cu[b + 1]))
        allowed = pos[None, :] <= (L - n + np.arange(n))[:, None]   # [n][L]
        for j in range(16):
            h = j // 8
            K = kf[blk, h, pos % 64].astype(np.longdouble)          # [L][D]
            V = vf[blk, h, pos % 64].astype(np.longdouble)
            S = qf[rows, j].astype(np.longdouble) @ K.T * w.softmax_scale
            E = np.where(allowed, np.exp(S), 0.0)
            ref = (E @ V) / E.sum(1, keepdims=True)
            np.testing.assert_allclose(out[rows, j], ref.astype(float), rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse[rows, j], np.log(E.sum(1)).astype(float),
                                       rtol=0, atol=1e-12)


def test_prefill_first_token_is_v0():
    w = W.make_workload(_cfg(8, 1), lengths=[200, 65], seed=23)
    q, cu = W.make_extend_query(w, [200, 65], seed=24)
    out, lse = _extend(w, q, cu)
    kf, vf = _kv_f64(w)
    qf = q.to(torch.float64).numpy()
    for b in range(2):
        r = int(cu[b])
        blk0 = int(w.block_table[b, 0])
        for j in range(8):
            assert np.array_equal(out[r, j], vf[blk0, 0, 0])
            assert abs(lse[r, j] - w.softmax_scale * float(qf[r, j] @ kf[blk0, 0, 0])) < 1e-12


def test_keys_after_the_causal_limit_are_invisible():
    lens, qn = [150, 40], [20, 40]
    w = W.make_workload(_cfg(8, 1), lengths=lens, seed=25)
    q, cu = W.make_extend_query(w, qn, seed=26)
    out1, lse1 = _extend(w, q, cu)
    # position 140 of sequence 0 is new token 10's own position
    blk = int(w.block_table[0, 140 // 64])
    w.k_cache[blk, :, 140 % 64] += 3.0
    w.v_cache[blk, :, 140 % 64] -= 1.0
    out2, lse2 = _extend(w, q, cu)
    assert np.array_equal(out1[:10], out2[:10]) and np.array_equal(lse1[:10], lse2[:10])
    assert not np.allclose(out1[10:20], out2[10:20])
    assert np.array_equal(out1[20:], out2[20:])  # the other sequence


def test_one_new_token_is_decode_and_ragged_equals_uniform():
    w = W.make_workload(_cfg(16, 2), lengths=[1, 70, 300], seed=27)
    cu1 = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    out, lse = _extend(w, w.q, cu1)
    ref_out, ref_lse = oracle.decode_workload(w)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)
    T = 1
    qm = W.make_multi_query(w, T, seed=28)
    om, lm = oracle.paged_decode_multi(qm, w.k_cache, w.v_cache, w.block_table, w.seq_lens,
                                       num_kv_heads=2, softmax_scale=w.softmax_scale)
    oe, le = _extend(w, qm.reshape(3, 16, 128), cu1)
    assert np.array_equal(oe, om.reshape(3, 16, 128)) and np.array_equal(le, lm.reshape(3, 16))


def test_rejects_bad_cu_q_lens():
    w = W.make_workload(_cfg(8, 1), lengths=[10, 5], seed=29)
    q = torch.zeros(8, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _extend(w, q, torch.tensor([0, 2, 8], dtype=torch.int32))   # 6 new tokens > 5 positions
    with pytest.raises(ValueError):
        _extend(w, q, torch.tensor([0, 5, 4], dtype=torch.int32))


def test_row_subset_equals_full_rows():
    w = W.make_workload(_cfg(16, 2), lengths=[90, 200], seed=30)
    q, cu = W.make_extend_query(w, [40, 70], seed=31)
    out, lse = _extend(w, q, cu)
    rows = [0, 39, 40, 77, 109]
    so, sl = oracle.paged_extend(q, w.k_cache, w.v_cache, w.block_table, w.seq_lens, cu,
                                 num_kv_heads=2, softmax_scale=w.softmax_scale, rows=rows)
    assert np.array_equal(so, out[rows]) and np.array_equal(sl, lse[rows])
