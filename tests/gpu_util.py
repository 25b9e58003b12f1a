"""Helpers for the GPU parity tests: move a seeded workload to the device,
run the CUDA path through the C ABI, and compare with the fp64 oracle."""
import numpy as np
import torch

import oracle
import paged_gqa_decode_hpc_gb300 as hpc

OUT_ATOL = OUT_RTOL = 1e-2   # |out - ref| <= 1e-2 + 1e-2 |ref|  (bf16 output)
LSE_ATOL = 1e-3              # |lse - ref| <= 1e-3
REL_FRO = 1e-2               # ||out - ref||_F / ||ref||_F per case (stricter check)


def device_workload(w, dev="cuda"):
    return dict(q=w.q.to(dev), k=w.k_cache.to(dev), v=w.v_cache.to(dev),
                bt=w.block_table.to(dev), sl=w.seq_lens.to(dev))


def run_cuda(w, d=None, plan="host", num_sms=None, splits=0, stream=None):
    """Run plan + attention + merge on the GPU; returns (out f64, lse f64) numpy."""
    d = d or device_workload(w)
    if num_sms is None:
        num_sms = hpc.hpc_device_sm_count()
    B, hq = w.q.shape[0], w.q.shape[1]
    out = torch.full((B, hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
    if plan == "host":
        p = hpc.hpc_decode_plan(w.seq_lens.tolist(), num_sms)
    elif plan == "device":
        p = hpc.hpc_decode_plan_create(max(B, 1), num_sms, hq)
        hpc.hpc_decode_plan_device(d["sl"], num_sms, p, stream)
    elif plan == "static":
        p = hpc.hpc_decode_plan_static(w.seq_lens.tolist(), num_sms, w.num_kv_heads, splits)
    else:
        raise ValueError(plan)
    hpc.hpc_decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], p, out, lse, stream=stream,
                        k_scale=w.k_scale, v_scale=w.v_scale)
    torch.cuda.synchronize()
    err = hpc.hpc_decode_plan_status(p)
    p.destroy()
    assert err == 0, f"device check bits {err}"
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def assert_parity(out, lse, ref_out, ref_lse, label=""):
    assert np.isfinite(out).all(), f"{label}: non-finite output"
    diff = np.abs(out - ref_out)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    bad = diff > bound
    assert not bad.any(), (f"{label}: {bad.sum()} outputs out of tolerance, "
                           f"worst {diff.max():.3e} at {np.unravel_index(diff.argmax(), diff.shape)}")
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{label}: lse finiteness differs"
    if fin.any():
        le = np.abs(lse[fin] - ref_lse[fin]).max()
        assert le <= LSE_ATOL, f"{label}: lse error {le:.3e}"
    assert np.array_equal(lse[~fin], ref_lse[~fin]), f"{label}: lse of empty sequences"
    nref = np.linalg.norm(ref_out)
    if nref > 0:
        rel = np.linalg.norm(out - ref_out) / nref
        assert rel <= REL_FRO, f"{label}: relative Frobenius error {rel:.3e}"


def check_against_oracle(w, **kw):
    ref_out, ref_lse = oracle.decode_workload(w)
    out, lse = run_cuda(w, **kw)
    assert_parity(out, lse, ref_out, ref_lse, label=f"{w.config_name} {kw}")
    return out, lse
