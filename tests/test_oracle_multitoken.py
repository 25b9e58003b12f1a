"""Pins for the multi-token decode oracle (q_len new tokens per sequence,
causal among themselves): it reduces to the single-token oracle for q_len 1,
token t ignores every key after its own position, it matches a dense
masked-softmax brute force, and tokens that see no key give 0 / -inf."""
import numpy as np
import torch

import oracle
from paged_gqa_decode_hpc_gb300 import workloads as W

D = 128


def _cfg(hq, hkv, fp8=False):
    return W.Config(97, "mtp", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


def _multi(w, q):
    return oracle.paged_decode_multi(q, w.k_cache, w.v_cache, w.block_table, w.seq_lens,
                                     num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                                     kv_is_fp8=w.kv_dtype == "fp8_e4m3", k_scale=w.k_scale,
                                     v_scale=w.v_scale)


def test_single_token_reduces_to_decode():
    w = W.make_workload(_cfg(16, 2), lengths=[1, 70, 300], seed=5)
    out, lse = _multi(w, w.q[:, None])
    ref_out, ref_lse = oracle.decode_workload(w)
    assert np.array_equal(out[:, 0], ref_out) and np.array_equal(lse[:, 0], ref_lse)


def test_causality_and_last_token():
    w = W.make_workload(_cfg(8, 1), lengths=[130, 64], seed=6)
    T = 3
    q = W.make_multi_query(w, T, seed=7)
    out1, lse1 = _multi(w, q)
    # perturb the key/value of sequence 0 at its last position (129): only token 2 sees it
    blk = int(w.block_table[0, 129 // 64])
    w.k_cache[blk, :, 129 % 64] += 1.0
    w.v_cache[blk, :, 129 % 64] -= 2.0
    out2, lse2 = _multi(w, q)
    assert np.array_equal(out1[0, :2], out2[0, :2]) and np.array_equal(lse1[0, :2], lse2[0, :2])
    assert not np.allclose(out1[0, 2], out2[0, 2])
    assert np.array_equal(out1[1], out2[1])
    # the last token is an ordinary decode over the whole sequence
    w.q = q[:, T - 1].contiguous()
    ref_out, ref_lse = oracle.decode_workload(w)
    assert np.array_equal(out2[:, T - 1], ref_out)


def test_matches_dense_masked_brute_force():
    w = W.make_workload(_cfg(16, 2, fp8=True), lengths=[5, 67, 2], seed=8)
    T = 4
    q = W.make_multi_query(w, T, seed=9)
    out, lse = _multi(w, q)
    qf = q.to(torch.float64).numpy()
    kf = w.k_cache.view(torch.float8_e4m3fn).to(torch.float64).numpy() * w.k_scale
    vf = w.v_cache.view(torch.float8_e4m3fn).to(torch.float64).numpy() * w.v_scale
    for b, L in enumerate(w.seq_lens.tolist()):
        pos = np.arange(L)
        blk = w.block_table[b].numpy()[pos // 64]
        for t in range(T):
            vis = pos < L - T + 1 + t  # causal mask of token t
            for j in range(16):
                h = j // 8
                if not vis.any():
                    assert np.all(out[b, t, j] == 0) and np.isneginf(lse[b, t, j])
                    continue
                K = kf[blk, h, pos % 64][vis].astype(np.longdouble)
                V = vf[blk, h, pos % 64][vis].astype(np.longdouble)
                s = K @ qf[b, t, j].astype(np.longdouble) * w.softmax_scale
                e = np.exp(s)
                np.testing.assert_allclose(out[b, t, j], ((e[:, None] * V).sum(0) / e.sum()).astype(float),
                                           rtol=1e-10, atol=1e-12)
                assert abs(lse[b, t, j] - float(np.log(e.sum()))) < 1e-12
