"""GPU parity of the fused prologue (QK-Norm + RoPE + paged KV write + FP8
query copy) against the fp64 oracle, and of prologue -> decode step against
the chained oracles."""
import numpy as np
import pytest
import torch

import oracle
from oracle import prologue_ref as PR
import paged_gqa_decode_hpc_gb300 as hpc
from paged_gqa_decode_hpc_gb300 import workloads as W
from tests.gpu_util import OUT_ATOL, OUT_RTOL, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hpc.load_library()


def _cfg(hq=64, hkv=8, fp8=False):
    return W.Config(93, "prologue", hq, hkv, "fp8_e4m3" if fp8 else "bf16")


def _f64(t):
    return t.to(torch.float64).numpy()


def _run(w, pin, q_fp8_scale=None, inplace=False, bt=None, err=None):
    dev = "cuda"
    q_in = pin.q_in.to(dev)
    kc, vc = w.k_cache.clone().to(dev), w.v_cache.clone().to(dev)
    q_out = q_in if inplace else torch.empty_like(q_in)
    q8 = torch.zeros(q_in.shape, dtype=torch.uint8, device=dev) if q_fp8_scale else None
    hpc.hpc_rope_norm_kv_write(q_in, pin.k_in.to(dev), pin.v_in.to(dev), w.seq_lens.to(dev),
                               (w.block_table if bt is None else bt).to(dev), pin.w_q.to(dev),
                               pin.w_k.to(dev), q_out, kc, vc, eps=pin.eps,
                               rope_base=pin.rope_base, q_out_fp8=q8,
                               q_fp8_scale=q_fp8_scale or 1.0, k_scale=w.k_scale,
                               v_scale=w.v_scale, device_error=err)
    torch.cuda.synchronize()
    return q_out.cpu(), (q8.cpu() if q8 is not None else None), kc.cpu(), vc.cpu()


def _oracle(w, pin):
    return PR.prologue(_f64(pin.q_in), _f64(pin.k_in), _f64(pin.v_in), w.seq_lens.tolist(),
                       w.block_table.numpy(), _f64(pin.w_q), _f64(pin.w_k), pin.eps,
                       pin.rope_base)


def _close(got, ref):
    assert np.all(np.abs(got - ref) <= OUT_ATOL + OUT_RTOL * np.abs(ref)), np.abs(got - ref).max()


def _oracle_codes(ref_vals, scale):
    return np.array([PR.e4m3_encode(x / scale) for x in ref_vals.ravel()], dtype=np.int64)


def _check_codes_exact(got_bytes, ref_vals, scale):
    """A pure quantisation of exact bf16 inputs (the V row): reading p5 fixes
    every byte, e4m3(x / scale) rounded to nearest even from the exact
    quotient, so the kernel's bytes must equal the oracle's."""
    ref_codes = _oracle_codes(ref_vals, scale)
    got = got_bytes.ravel().astype(np.int64)
    bad = np.flatnonzero(got != ref_codes)
    assert bad.size == 0, (f"{bad.size} of {got.size} e4m3 bytes differ, first at {bad[0]}: "
                           f"got {got[bad[0]]:#04x}, oracle {ref_codes[bad[0]]:#04x}")


def _check_codes_near(got_bytes, ref_vals, scale, label):
    """e4m3 bytes of a value the kernel computes in fp32 (normed and rotated
    q and k) vs the oracle's encoding of its fp64 value: the two values differ
    by fp32 rounding, which moves a value across a code boundary only when it
    lies within that rounding of the boundary. Every code is within one step,
    and the mismatches are few (reported, asserted below 1 %)."""
    ref_codes = _oracle_codes(ref_vals, scale)
    got = got_bytes.ravel().astype(np.int64)
    mag = lambda c: np.where(c & 0x80, -(c & 0x7F), c & 0x7F)
    assert np.all(np.abs(mag(got) - mag(ref_codes)) <= 1)
    n_bad = int(np.sum(got != ref_codes))
    print(f"{label}: {n_bad} of {got.size} e4m3 codes one step from the oracle's")
    assert n_bad <= got.size // 100
    return n_bad


@pytest.mark.parametrize("hq,hkv,base", [(64, 8, 1e4), (8, 1, 1e6), (32, 4, 5e5)])
def test_prologue_bf16_cache(hq, hkv, base):
    lens = [1, 64, 65, 1000, 131072, 0, 4097]
    w = W.make_workload(_cfg(hq, hkv), lengths=lens, seed=51, slack_blocks=3)
    pin = W.make_prologue_inputs(w, seed=52, rope_base=base)
    q_out, _, kc, vc = _run(w, pin)
    q_ref, k_ref, v_ref, slots = _oracle(w, pin)
    k0, v0 = w.k_cache, w.v_cache
    touched = np.zeros(k0.shape[:1] + k0.shape[2:3], dtype=bool)  # [block][slot]
    for b, sl in enumerate(slots):
        if sl is None:
            continue
        _close(_f64(q_out[b]), q_ref[b])
        blk, slot = sl
        touched[blk, slot] = True
        _close(_f64(kc[blk, :, slot]), k_ref[b])
        assert torch.equal(vc[blk, :, slot], pin.v_in[b])  # V is copied exactly
    # nothing else in either cache changed
    m = torch.from_numpy(~touched)
    assert torch.equal(kc.permute(0, 2, 1, 3)[m], k0.permute(0, 2, 1, 3)[m])
    assert torch.equal(vc.permute(0, 2, 1, 3)[m], v0.permute(0, 2, 1, 3)[m])


def test_prologue_fp8_cache_and_fp8_query():
    lens = [3, 700, 64, 129, 9000]
    w = W.make_workload(_cfg(64, 8, fp8=True), lengths=lens, seed=53)
    pin = W.make_prologue_inputs(w, seed=54)
    q_out, q8, kc, vc = _run(w, pin, q_fp8_scale=0.02)
    q_ref, k_ref, v_ref, slots = _oracle(w, pin)
    for b, (blk, slot) in enumerate(slots):
        _close(_f64(q_out[b]), q_ref[b])
        _check_codes_near(q8[b].numpy(), q_ref[b], 0.02, f"q seq {b}")
        _check_codes_near(kc[blk, :, slot].numpy(), k_ref[b], w.k_scale, f"k seq {b}")
        _check_codes_exact(vc[blk, :, slot].numpy(), v_ref[b], w.v_scale)


def test_prologue_fp8_v_bytes_exact_on_many_rows():
    """V quantisation alone over 256 sequences x 8 heads x 128 values with a
    scale that is not a power of two, so the quotient is almost never exact
    and every rounding decision is exercised (sub-normal and saturating codes
    included: the inputs span 2^-12 .. 2^10 times the scale)."""
    lens = [1 + (37 * i) % 200 for i in range(256)]
    w = W.make_workload(_cfg(64, 8, fp8=True), lengths=lens, seed=59)
    pin = W.make_prologue_inputs(w, seed=60)
    g = torch.Generator().manual_seed(61)
    mag = torch.exp2(torch.empty(pin.v_in.shape).uniform_(-12.0, 10.0, generator=g))
    sgn = torch.where(torch.rand(pin.v_in.shape, generator=g) < 0.5, -1.0, 1.0)
    v_in = (mag * sgn * w.v_scale).to(torch.bfloat16)
    v_in[0, 0, :4] = torch.tensor([0.0, -0.0, 448.0 * w.v_scale, -1e4 * w.v_scale])
    pin.v_in = v_in
    _, _, _, vc = _run(w, pin)
    _, _, v_ref, slots = _oracle(w, pin)
    for b, (blk, slot) in enumerate(slots):
        _check_codes_exact(vc[blk, :, slot].numpy(), v_ref[b], w.v_scale)


def test_prologue_in_place_query_and_bad_block():
    w = W.make_workload(_cfg(), lengths=[200, 300], seed=55)
    pin = W.make_prologue_inputs(w, seed=56)
    q_ref, k_ref, _, slots = _oracle(w, pin)
    q_out, _, kc, _ = _run(w, pin, inplace=True)
    for b in range(2):
        _close(_f64(q_out[b]), q_ref[b])
    bt = w.block_table.clone()
    bt[1, 300 // 64] = w.k_cache.shape[0] + 3  # the new token's block is out of range
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, _, kc2, _ = _run(w, pin, bt=bt, err=err)
    assert int(err.item()) & hpc.HPC_DEVCHK_BAD_BLOCK
    blk0, slot0 = slots[0]
    _close(_f64(kc2[blk0, :, slot0]), k_ref[0])  # the other sequence is still written


@pytest.mark.parametrize("fp8", [False, True])
def test_prologue_then_decode_step_matches_chained_oracle(fp8):
    lens = [37, 64, 1000, 4096, 1]
    w = W.make_workload(_cfg(64, 8, fp8), lengths=lens, seed=57)
    pin = W.make_prologue_inputs(w, seed=58)
    # oracle chain: prologue in fp64, rows stored in the cache format, then decode
    q_ref, k_ref, v_ref, slots = _oracle(w, pin)
    wo = W.Workload(w.config_name, w.seq_lens, w.block_table, torch.from_numpy(q_ref).to(torch.bfloat16),
                    w.k_cache.clone(), w.v_cache.clone(), w.k_scale, w.v_scale, w.kv_dtype,
                    w.softmax_scale, w.num_q_heads, w.num_kv_heads)
    for b, (blk, slot) in enumerate(slots):
        if fp8:
            wo.k_cache[blk, :, slot] = torch.tensor([PR.e4m3_encode(x / w.k_scale) for x in k_ref[b].ravel()],
                                                    dtype=torch.uint8).view(-1, 128)
            wo.v_cache[blk, :, slot] = torch.tensor([PR.e4m3_encode(x / w.v_scale) for x in v_ref[b].ravel()],
                                                    dtype=torch.uint8).view(-1, 128)
        else:
            wo.k_cache[blk, :, slot] = torch.from_numpy(k_ref[b]).to(torch.bfloat16)
            wo.v_cache[blk, :, slot] = torch.from_numpy(v_ref[b]).to(torch.bfloat16)
    ref_out, ref_lse = oracle.decode_workload(wo)
    # GPU chain: prologue kernel then the decode step, on one stream
    dev = "cuda"
    kc, vc = w.k_cache.clone().to(dev), w.v_cache.clone().to(dev)
    q = torch.empty(pin.q_in.shape, dtype=torch.bfloat16, device=dev)
    sl, bt = w.seq_lens.to(dev), w.block_table.to(dev)
    hpc.hpc_rope_norm_kv_write(pin.q_in.to(dev), pin.k_in.to(dev), pin.v_in.to(dev), sl, bt,
                               pin.w_q.to(dev), pin.w_k.to(dev), q, kc, vc, eps=pin.eps,
                               rope_base=pin.rope_base, k_scale=w.k_scale, v_scale=w.v_scale)
    sms = hpc.hpc_device_sm_count()
    plan = hpc.hpc_decode_plan_create(len(lens), sms, 64)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    hpc.hpc_decode_step(q, kc, vc, bt, sl, plan, sms, out, lse, k_scale=w.k_scale, v_scale=w.v_scale)
    torch.cuda.synchronize()
    assert hpc.hpc_decode_plan_status(plan) == 0
    plan.destroy()
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse,
                  label=f"prologue+decode fp8={fp8}")
