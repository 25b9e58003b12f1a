#!/usr/bin/env python
"""Decode-step benchmark of mixed-length paged GQA decode attention on GB300.

One step = the whole hot path on one batch already resident in HBM, through
hpc_decode_step on one stream. With one query token per sequence that is one
launch of the step kernel: its CTAs plan the step (balanced parts of 64-token
(tile, KV head) units plus a pool of chunks), compute the split-KV attention
and merge split (sequence, KV head) pairs by log-sum-exp rescaling in the same
kernel (batches above 3072 sequences run the planner, attention and merge
kernels instead). Reported `value` is
achieved HBM GB/s = algorithmic bytes (KV of the actual tokens + Q + O) per
step / device time per step, summed over ranks (weak scaling: every rank
runs its own replica of the batch). The default workload is the skewed
batch (1 x 131072 + 31 x 4096 KV tokens, 64 q / 8 kv heads, head_dim 128,
bf16 KV in 64-token blocks).

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   (the fp64 CPU oracle, timed on host cores)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-step µs and achieved HBM GB/s (% of GB300 peak), mixed-length paged GQA"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024
WORKLOAD_TEXT = {
    "tiny": "tiny: 4 seqs KV {37,64,200,1000}, 8 q / 1 kv heads, d128, bf16 KV",
    "uniform": "uniform: 64 seqs x 512 KV tokens, 64 q / 8 kv heads, d128, bf16 KV",
    "skewed": "skewed: 1 x 131072 + 31 x 4096 KV tokens, 64 q / 8 kv heads, d128, bf16 KV",
    "skewed_fp8": "skewed FP8: 1 x 131072 + 31 x 4096 KV tokens, 64 q / 8 kv heads, d128, "
                  "fp8_e4m3 KV (per-tensor scales), bf16 q/out",
    "random_mixed": "random mixed: 256 seqs, KV lengths log-uniform in [16, 65536], "
                    "64 q / 8 kv heads, d128, bf16 KV",
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["hpc", "reference"], default="hpc")
    ap.add_argument("--config", default="skewed", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--no-static", action="store_true", help="skip the static split-KV ablation")
    ap.add_argument("--static-sweep", default="1,2,4,8,16,32",
                    help="split counts timed for the static ablation ('' = rule only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip timing the step replayed from a CUDA graph")
    ap.add_argument("--no-flush", action="store_true", help="do not flush L2 between steps")
    ap.add_argument("--json-out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--q-lens", default="2,4",
                    help="query-token counts timed for multi-token decode ('' = none)")
    ap.add_argument("--tc-min-q-len", type=int, default=0,
                    help="smallest q_len run on the tensor-core decode kernel (0: the "
                         "library's per-dtype default; 9: never)")
    ap.add_argument("--no-prologue", action="store_true",
                    help="skip timing the fused prologue kernel")
    ap.add_argument("--no-copy-probe", action="store_true",
                    help="skip the device-to-device copy bandwidth probe")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill / extend (tcgen05) timings")
    ap.add_argument("--prefill-cases",
                    default="q512_prefill,prefill_4x4096,extend_8x(8192+512),prefill_4x4096_fp8",
                    help="prefill / extend cases to time (comma list)")
    ap.add_argument("--scale-lengths", type=float, default=1.0,
                    help="scale every KV length of the config (smaller profiling cases)")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers
def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if k in d and d[k]:
                return float(d[k]), "measured (MEASURED_PEAKS.json)"
    except Exception:
        pass
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def measured_peak_bf16_tflops():
    """Dense bf16 tensor peak for a kernel timed alone (the burst figure)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("bf16_tflops"):
            return float(d["bf16_tflops"]), "measured burst (MEASURED_PEAKS.json)"
    except Exception:
        pass
    return FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s (no MEASURED_PEAKS.json)"


def extend_flops(lens, qn, num_q_heads):
    """Useful FLOPs of causal prefill / extend attention: per query row and
    visible key, 2*128 for q.k and 2*128 for p*v."""
    vis = 0
    for L, n in zip(lens, qn):
        # new token i sees L - n + 1 + i keys
        vis += n * (L - n + 1) + n * (n - 1) // 2
    return 4 * 128 * num_q_heads * vis


def _code_only(text):
    """C / C++ source without its comments and with whitespace runs
    collapsed: what the compiler sees of it (string literals in this
    source hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_digest():
    """Digest of the timed kernel's code: step_kernel.cu and every file it
    includes from the package's csrc/ or include/ directories, transitively,
    each without its comments (a comment edit does not make a profile
    stale; any code change does)."""
    dirs = [os.path.join(ROOT, "paged_gqa_decode_hpc_gb300", "csrc"), os.path.join(ROOT, "include")]
    h = hashlib.sha256()
    seen, todo = set(), ["step_kernel.cu"]
    while todo:
        name = todo.pop(0)
        if name in seen:
            continue
        path = next((os.path.join(d, name) for d in dirs
                     if os.path.exists(os.path.join(d, name))), None)
        if path is None:
            continue  # a system header
        seen.add(name)
        with open(path, "rb") as f:
            data = f.read()
        h.update(name.encode() + b"\0" + _code_only(data.decode("utf-8", "replace")).encode())
        todo += re.findall(r'^\s*#\s*include\s+"([^"]+)"', data.decode("utf-8", "replace"), re.M)
    return h.hexdigest()[:16]


def profiled_traffic(config_name):
    """DRAM bytes per step-kernel launch from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"step_kernel_{config_name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_digest():
        return None
    return int(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        busy = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, value):
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_workload(args):
    from paged_gqa_decode_hpc_gb300 import workloads as W
    if args.scale_lengths == 1.0:
        return W.make_workload(args.config)
    cfg = W.CONFIG_BY_NAME[args.config]
    import torch
    lens = W.draw_lengths(cfg, torch.Generator().manual_seed(cfg.seed))
    lens = [max(1, int(round(L * args.scale_lengths))) for L in lens]
    return W.make_workload(cfg, lengths=lens)


# ------------------------------------------------------------ CPU oracle leg
def oracle_sample(w, budget_s=4.0):
    """A bounded sample of the workload for the oracle: whole sequences, taken
    in order until the estimated fp64 CPU time reaches `budget_s`."""
    import oracle
    from paged_gqa_decode_hpc_gb300 import workloads as W
    lens = w.seq_lens.tolist()
    # calibrate on the shortest non-empty sequences (about 0.2 s of work)
    order = sorted(range(len(lens)), key=lambda b: lens[b])
    calib, tok = [], 0
    for b in order:
        if lens[b] > 0:
            calib.append(b)
            tok += lens[b]
        if tok > 20000:
            break
    t0 = time.perf_counter()
    oracle.decode_workload(_subset(w, calib))
    rate = tok / max(time.perf_counter() - t0, 1e-6)  # tokens / s
    chosen, est = [], 0.0
    for b in range(len(lens)):
        cost = lens[b] / rate
        if chosen and est + cost > budget_s:
            continue
        chosen.append(b)
        est += cost
    return _subset(w, chosen), chosen


def _subset(w, seqs):
    from paged_gqa_decode_hpc_gb300 import workloads as W
    import torch
    idx = torch.tensor(seqs, dtype=torch.long)
    return W.Workload(w.config_name, w.seq_lens[idx].clone(), w.block_table[idx].clone(),
                      w.q[idx].clone(), w.k_cache, w.v_cache, w.k_scale, w.v_scale, w.kv_dtype,
                      w.softmax_scale, w.num_q_heads, w.num_kv_heads)


def time_oracle(sample, reps, keep=False):
    """Wall times of `reps` oracle runs on the sample; with keep, also the
    last run's (out, lse)."""
    import oracle
    times, res = [], None
    for _ in range(reps):
        t0 = time.perf_counter()
        res = oracle.decode_workload(sample)
        times.append(time.perf_counter() - t0)
    return (times, res) if keep else times


def parity_summary(out, lse, ref_out, ref_lse, atol=1e-2, rtol=1e-2, lse_atol=1e-3):
    """Worst errors of a GPU result against the oracle's for the same rows:
    max |out - ref|, the largest ratio of that error to the bound
    atol + rtol |ref| (<= 1 passes), max |lse - ref| over finite entries, and
    whether the infinite lse entries (empty sequences) agree."""
    import numpy as np
    out, lse = np.asarray(out, dtype=np.float64), np.asarray(lse, dtype=np.float64)
    ref_out, ref_lse = np.asarray(ref_out, dtype=np.float64), np.asarray(ref_lse, dtype=np.float64)
    err = np.abs(out - ref_out)
    ratio = err / (atol + rtol * np.abs(ref_out))
    fin = np.isfinite(ref_lse)
    lse_err = np.abs(lse[fin] - ref_lse[fin])
    inf_match = bool(np.array_equal(np.isfinite(lse), fin))
    worst_ratio = float(ratio.max()) if ratio.size else 0.0
    worst_lse = float(lse_err.max()) if lse_err.size else 0.0
    return {"max_abs_out_err": float(err.max()) if err.size else 0.0,
            "max_err_over_bound": round(worst_ratio, 6),
            "max_abs_lse_err": worst_lse, "lse_inf_match": inf_match,
            "bounds": f"|out - ref| <= {atol} + {rtol}|ref|, |lse - ref| <= {lse_atol}",
            "pass": bool(worst_ratio <= 1.0 and worst_lse <= lse_atol and inf_match)}


# ------------------------------------------------------------- reference arm
def run_reference(args, ws, rank):
    if rank != 0:
        return
    import oracle
    from paged_gqa_decode_hpc_gb300 import workloads as W
    w = load_workload(args)
    budget = max(0.5, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    sample, seqs = oracle_sample(w, budget_s=budget)
    time_oracle(sample, args.warmup)
    times = time_oracle(sample, args.steps)
    step_s = statistics.mean(times)
    gbs = sample.algorithmic_bytes() / step_s / 1e9
    desc = (f"{len(seqs)} of {w.num_seqs} sequences ({int(sample.seq_lens.sum())} of "
            f"{int(w.seq_lens.sum())} KV tokens) per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, the pages' shapes)",
        "config": {"workload": WORKLOAD_TEXT[args.config], "sample": desc},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": oracle.num_cpus(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    emit(line, args)


def emit(line, args):
    s = json.dumps(line)
    print(s, flush=True)
    if args.json_out:
        with open(args.json_out, "a") as f:
            f.write(s + "\n")


# ---------------------------------------------------------------- hpc arm
def run_hpc(args, ws, rank, local):
    import torch
    import paged_gqa_decode_hpc_gb300 as hpc
    from paged_gqa_decode_hpc_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    hpc.load_library()
    dev = torch.device("cuda", local)
    w = load_workload(args)
    B, hq, hkv = w.num_seqs, w.num_q_heads, w.num_kv_heads
    fp8 = w.kv_dtype == "fp8_e4m3"
    q, kc, vc = w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev)
    bt, sl = w.block_table.to(dev), w.seq_lens.to(dev)
    out = torch.empty((B, hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev)
    num_sms = hpc.hpc_device_sm_count()
    plan = hpc.hpc_decode_plan_create(B, num_sms, hq)
    # the step kernel alone; above 3072 sequences the planner, attention and merge kernels
    one_kernel = 0 < B <= 3072
    launches_per_step = 1 if one_kernel else 3
    stream = torch.cuda.current_stream()
    nbytes = w.algorithmic_bytes()
    flush = None if args.no_flush else torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = None if args.no_flush else torch.ones(2 * L2_BYTES // 4, dtype=torch.int32,
                                                     device=dev)

    def flush_l2():
        # Write 2x L2, then read another 2x L2 so that L2 ends up holding clean
        # lines: no write-back of the flush lands inside the next timed step.
        if flush is not None:
            flush.fill_(1)
            flush_rd.sum()

    def mk():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)  # materialise the handle
        return e

    def step(evs=None):
        if evs:
            evs[0].record(stream)
            hpc.hpc_decode_plan_set_timing_events(plan, evs[1], evs[2], evs[3])
        hpc.hpc_decode_step(q, kc, vc, bt, sl, plan, num_sms, out, lse, stream=stream,
                            k_scale=w.k_scale, v_scale=w.v_scale)
        if evs:
            hpc.hpc_decode_plan_set_timing_events(plan)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    assert hpc.hpc_decode_plan_status(plan) == 0, "device checks fired during warm-up"
    # Timed region: events at step boundaries only (events between the three
    # kernels would serialise them and hide the programmatic-launch overlap).
    ev = [[mk(), mk()] for _ in range(args.steps)]
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    barrier(ws)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    if hpc.hpc_decode_plan_status(plan) != 0:
        raise SystemExit("device checks fired during the timed steps")
    if not torch.isfinite(out.float()).all():
        raise SystemExit("non-finite output")
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # Breakdown pass (not in the timed region): events around each kernel.
    nb = max(3, min(args.steps, 10))
    evb = [[mk() for _ in range(4)] for _ in range(nb)]
    torch.cuda.synchronize()
    for i in range(nb):
        flush_l2()
        step(evb[i])
    torch.cuda.synchronize()
    plan_ms = [e[0].elapsed_time(e[1]) for e in evb]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evb]
    merge_ms = [e[2].elapsed_time(e[3]) for e in evb]
    ms = statistics.mean(step_ms)
    ms_all = max_over_ranks(ws, ms)
    value = ws * nbytes / (ms_all * 1e-3) / 1e9

    peak, peak_src = measured_peak_gbs()
    attn_mean = statistics.mean(attn_ms)
    achieved = nbytes / (attn_mean * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_all, 5),
        "us_per_step": round(ms_all * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, shuffled block table; the pages' shapes)",
        "config": {
            "workload": WORKLOAD_TEXT[args.config] + (
                f" (lengths scaled x{args.scale_lengths})" if args.scale_lengths != 1.0 else ""),
            "num_seqs": B,
            "kv_tokens": int(w.seq_lens.sum()), "num_sms": num_sms,
            "algorithmic_bytes_per_step": nbytes,
            "l2": ("flushed between steps (write 2x L2, then read 2x L2)" if flush is not None
                   else "not flushed"),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
        },
        "step_us": {"mean": round(ms * 1e3, 2), "median": round(statistics.median(step_ms) * 1e3, 2),
                    "min": round(min(step_ms) * 1e3, 2), "max": round(max(step_ms) * 1e3, 2)},
        "breakdown_us": ({"note": "separate pass, events around the step kernel, which plans, "
                                  "computes and merges the step",
                          "step_kernel": round(attn_mean * 1e3, 2)} if one_kernel else
                         {"note": "separate pass, events between kernels (no launch overlap)",
                          "launch_to_attention": round(statistics.mean(plan_ms) * 1e3, 2),
                          "attention": round(attn_mean * 1e3, 2),
                          "merge": round(statistics.mean(merge_ms) * 1e3, 2)}),
        "frac_of_peak_step": round(value / ws / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(args.config) if one_kernel else None,
                     "kernel": "step_kernel" if one_kernel else "attn_kernel",
                     "peak_source": peak_src,
                     "bytes_per_launch": nbytes},
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if clocks:
        line["clocks"] = clocks

    # ---- static split-KV ablation (attention + merge, host-built plans), set
    # against the dynamic step timed above and the pages' tile plan run through
    # the plan-based attention + merge kernels
    if not args.no_static:
        def time_plan(p, steps):
            es = [[mk(), mk()] for _ in range(steps)]
            for _ in range(2):
                flush_l2()
                hpc.hpc_decode_attn(q, kc, vc, bt, sl, p, out, lse, stream=stream,
                                    k_scale=w.k_scale, v_scale=w.v_scale)
            torch.cuda.synchronize()
            for e in es:
                flush_l2()
                e[0].record(stream)
                hpc.hpc_decode_attn(q, kc, vc, bt, sl, p, out, lse, stream=stream,
                                    k_scale=w.k_scale, v_scale=w.v_scale)
                e[1].record(stream)
            torch.cuda.synchronize()
            assert hpc.hpc_decode_plan_status(p) == 0
            return statistics.mean(e[0].elapsed_time(e[1]) for e in es) * 1e3

        n_st = max(3, min(args.steps, 10))
        lens = w.seq_lens.tolist()
        with hpc.hpc_decode_plan(lens, num_sms) as pd:
            dyn_us = time_plan(pd, n_st)
        with hpc.hpc_decode_plan_static(lens, num_sms, hkv, 0) as ps:
            rule_S = int(hpc.hpc_decode_plan_export(ps)[7])
            st_us = time_plan(ps, n_st)
        sweep = {}
        for s in [int(x) for x in args.static_sweep.split(",") if x.strip()]:
            with hpc.hpc_decode_plan_static(lens, num_sms, hkv, s) as ps:
                sweep[s] = round(time_plan(ps, n_st), 2)
        best = min(sweep.values()) if sweep else st_us
        step_us = ms * 1e3
        line["static_ablation"] = {
            "dynamic_step_us": round(step_us, 2),
            "dynamic_tile_plan_attn_merge_us": round(dyn_us, 2),
            "static_rule_splits": rule_S,
            "static_rule_us": round(st_us, 2), "static_sweep_us": sweep,
            "speedup_vs_static_rule": round(st_us / step_us, 3),
            "speedup_vs_best_static": round(best / step_us, 3),
            "note": "speedups of the dynamic step over static split-KV (attention + merge, L2 "
                    "flushed before each launch); the hpc_decode_plan tile plan through the same "
                    "attention + merge kernels is reported beside it"}

    # ---- the same step captured once in a CUDA graph and replayed
    if not args.no_graph:
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):  # one call on the capture stream before capturing
            hpc.hpc_decode_step(q, kc, vc, bt, sl, plan, num_sms, out, lse, stream=gs,
                                k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            hpc.hpc_decode_step(q, kc, vc, bt, sl, plan, num_sms, out, lse, stream=gs,
                                k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        for _ in range(3):
            flush_l2()
            graph.replay()
        eg = [[mk(), mk()] for _ in range(args.steps)]
        torch.cuda.synchronize()
        for a, b_ in eg:
            flush_l2()
            a.record(stream)
            graph.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        if hpc.hpc_decode_plan_status(plan) != 0:
            raise SystemExit("device checks fired during the graph replays")
        g_us = statistics.mean(x.elapsed_time(y) for x, y in eg) * 1e3
        line["graph"] = {"us_per_step": round(g_us, 2),
                         "gbs": round(nbytes / (g_us * 1e-6) / 1e9, 1),
                         "note": "hpc_decode_step captured once in a CUDA graph and replayed"}
        line["gpu_launches"] += launches_per_step * args.steps
        del graph

    # ---- end to end through the public API, host buffers
    if not args.no_e2e:
        # The batch and the results in pinned host memory; the library's
        # hpc_decode_step_host enqueues the copies in, the step and the copies
        # out (one cudaMemcpyAsync per buffer) on the stream.
        def pinned_like(t):
            return torch.empty(t.shape, dtype=t.dtype, device="cpu", pin_memory=True)
        q_h, sl_h, bt_h = pinned_like(w.q), pinned_like(w.seq_lens), pinned_like(w.block_table)
        q_h.copy_(w.q)
        sl_h.copy_(w.seq_lens)
        bt_h.copy_(w.block_table)
        out_h, lse_h = pinned_like(out), pinned_like(lse)
        nb = lambda t: t.numel() * t.element_size()
        h2d = nb(q_h) + nb(sl_h) + nb(bt_h)
        d2h = nb(out_h) + nb(lse_h)

        def e2e_step():
            hpc.hpc_decode_step_host(q_h, kc, vc, bt_h, sl_h, plan, num_sms, out_h, lse_h,
                                     stream=stream, k_scale=w.k_scale, v_scale=w.v_scale)

        for _ in range(max(3, args.warmup)):
            flush_l2()
            e2e_step()
        es = [[mk(), mk()] for _ in range(args.steps)]
        torch.cuda.synchronize()
        barrier(ws)
        for e in es:
            flush_l2()
            e[0].record(stream)
            e2e_step()
            e[1].record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(ws, statistics.mean(a.elapsed_time(b) for a, b in es))
        # the host copy of the result must equal a device-resident step's
        hpc.hpc_decode_step(q, kc, vc, bt, sl, plan, num_sms, out, lse, stream=stream,
                            k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        same = bool(torch.equal(out_h, out.cpu()) and torch.equal(lse_h, lse.cpu()))
        line["e2e"] = {"value": round(ws * nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                       "us_per_step": round(e2e_ms * 1e3, 2),
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "api": "hpc_decode_step_host (host q, lengths, block table, out, lse)",
                       "result_matches_device_step": same}
        line["gpu_launches"] += launches_per_step * args.steps

    # ---- fp64 CPU oracle on host cores (rank 0, N = 1 only)
    if not args.no_cpu_baseline and ws == 1 and rank == 0:
        import oracle
        sample, seqs = oracle_sample(w, budget_s=6.0)
        times, ref = time_oracle(sample, 3, keep=True)
        t = statistics.median(times)
        line["cpu_baseline"] = {
            "value": round(sample.algorithmic_bytes() / t / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_cpus(), "kind": "oracle",
            "sample": f"{len(seqs)} of {B} sequences ({int(sample.seq_lens.sum())} of "
                      f"{int(w.seq_lens.sum())} KV tokens), median of 3 runs, {t:.2f} s"}
        # the step's own output on the same sequences against the oracle's: one
        # dynamic step right here, so the report covers hpc_decode_step whatever
        # legs ran before it
        try:
            hpc.hpc_decode_step(q, kc, vc, bt, sl, plan, num_sms, out, lse, stream=stream,
                                k_scale=w.k_scale, v_scale=w.v_scale)
            torch.cuda.synchronize()
            idx = torch.tensor(seqs, dtype=torch.long, device=out.device)
            line["parity_sample"] = dict(
                parity_summary(out[idx].double().cpu().numpy(), lse[idx].double().cpu().numpy(),
                               ref[0], ref[1]),
                sequences=len(seqs))
        except Exception as e:  # a report, never a reason to lose the line
            line["parity_sample"] = {"error": f"{type(e).__name__}: {e}"[:200]}

    # ---- multi-token decode (q_len new tokens per sequence share one KV read)
    if args.q_lens:
        hpc.hpc_decode_tc_min_q_len(args.tc_min_q_len)
        mt = {"tc_min_q_len": hpc.hpc_decode_tc_min_q_len(-1)}
        for T in [int(x) for x in args.q_lens.split(",") if x.strip()]:
            qm = W.make_multi_query(w, T, seed=8000 + T).to(dev)
            om = torch.empty_like(qm)
            lm = torch.empty(qm.shape[:3], dtype=torch.float32, device=dev)
            pm = hpc.hpc_decode_plan_create(B, num_sms, T * hq)

            def mstep():
                hpc.hpc_decode_step(qm, kc, vc, bt, sl, pm, num_sms, om, lm, stream=stream,
                                    k_scale=w.k_scale, v_scale=w.v_scale)

            for _ in range(3):
                flush_l2()
                mstep()
            es = [[mk(), mk()] for _ in range(max(5, min(args.steps, 20)))]
            for a, b_ in es:
                flush_l2()
                a.record(stream)
                mstep()
                b_.record(stream)
            torch.cuda.synchronize()
            assert hpc.hpc_decode_plan_status(pm) == 0
            pm.destroy()
            us = statistics.mean(a.elapsed_time(b_) for a, b_ in es) * 1e3
            mbytes = w.kv_bytes() + T * w.qo_bytes()
            mt[f"q_len_{T}"] = {"us_per_step": round(us, 2), "algorithmic_bytes": mbytes,
                                "gbs": round(mbytes / (us * 1e-6) / 1e9, 1),
                                "us_per_query_token": round(us / T, 2)}
        line["multi_token"] = mt

    # ---- the fused prologue (QK-Norm + RoPE + KV write) for this batch's new tokens
    if not args.no_prologue:
        pin = W.make_prologue_inputs(w, seed=7000)
        qi, ki, vi = pin.q_in.to(dev), pin.k_in.to(dev), pin.v_in.to(dev)
        wq, wk = pin.w_q.to(dev), pin.w_k.to(dev)
        q_new = torch.empty_like(qi)
        kc2, vc2 = kc.clone(), vc.clone()

        def prologue():
            hpc.hpc_rope_norm_kv_write(qi, ki, vi, sl, bt, wq, wk, q_new, kc2, vc2, eps=pin.eps,
                                       rope_base=pin.rope_base, k_scale=w.k_scale,
                                       v_scale=w.v_scale, stream=stream)

        def prologue_and_step():
            prologue()
            hpc.hpc_decode_step(q_new, kc2, vc2, bt, sl, plan, num_sms, out, lse, stream=stream,
                                k_scale=w.k_scale, v_scale=w.v_scale)

        res = {}
        for name, fn in (("prologue_us", prologue), ("prologue_plus_step_us", prologue_and_step)):
            for _ in range(3):
                flush_l2()
                fn()
            es = [[mk(), mk()] for _ in range(max(5, min(args.steps, 20)))]
            for a, b_ in es:
                flush_l2()
                a.record(stream)
                fn()
                b_.record(stream)
            torch.cuda.synchronize()
            res[name] = round(statistics.mean(a.elapsed_time(b_) for a, b_ in es) * 1e3, 2)
        rows_in = B * (hq + 2 * hkv) * 128 * 2
        rows_out = B * hq * 128 * 2 + B * 2 * hkv * 128 * (1 if fp8 else 2)
        pbytes = rows_in + rows_out
        res["algorithmic_bytes"] = pbytes
        res["achieved_gbs"] = round(pbytes / (res["prologue_us"] * 1e-6) / 1e9, 1)
        res["note"] = "latency-bound: the bytes are small; one launch of B*(H_q+2*H_kv) warps"
        line["prologue"] = res
        del kc2, vc2

    # ---- prefill / extend attention (tcgen05), the pages' prefill shapes
    if not args.no_prefill and rank == 0:
        peak_tf, peak_src = measured_peak_bf16_tflops()
        cases = [("q512_prefill", [512], [512], "bf16"),
                 ("prefill_4x4096", [4096] * 4, [4096] * 4, "bf16"),
                 ("extend_8x(8192+512)", [8704] * 8, [512] * 8, "bf16"),
                 ("prefill_4x4096_fp8", [4096] * 4, [4096] * 4, "fp8_e4m3")]
        pf = {}
        wanted = [c.strip() for c in args.prefill_cases.split(",") if c.strip()]
        for name, lens, qn, kvd in cases:
            if name not in wanted:
                continue
            cfgp = W.Config(90, "prefill", 64, 8, kvd)
            wp = W.make_workload(cfgp, lengths=lens, seed=9000)
            qp, cup = W.make_extend_query(wp, qn, seed=9001)
            qd, kd, vd = qp.to(dev), wp.k_cache.to(dev), wp.v_cache.to(dev)
            btd, sld, cud = wp.block_table.to(dev), wp.seq_lens.to(dev), cup.to(dev)
            od = torch.empty_like(qd)
            ld = torch.empty(qd.shape[:2], dtype=torch.float32, device=dev)
            errd = torch.zeros(1, dtype=torch.int32, device=dev)

            def ext():
                hpc.hpc_extend_attn(qd, kd, vd, btd, sld, cud, od, ld, device_error=errd,
                                    stream=stream, k_scale=wp.k_scale, v_scale=wp.v_scale)

            for _ in range(3):
                flush_l2()
                ext()
            es = [[mk(), mk()] for _ in range(max(5, min(args.steps, 20)))]
            for a, b_ in es:
                flush_l2()
                a.record(stream)
                ext()
                b_.record(stream)
            torch.cuda.synchronize()
            if int(errd.item()) != 0:
                raise RuntimeError(f"prefill case {name}: device check bits {int(errd.item())}")
            us = statistics.mean(a.elapsed_time(b_) for a, b_ in es) * 1e3
            fl = extend_flops(lens, qn, 64)
            tf = fl / (us * 1e-6) / 1e12
            pf[name] = {"us": round(us, 2), "flops": fl, "tflops": round(tf, 1), "kv": kvd,
                        "frac_of_bf16_peak": round(tf / peak_tf, 4),
                        "new_tokens": sum(qn), "kv_tokens": sum(lens)}
            line["gpu_launches"] += len(es)
            del qd, kd, vd, od, ld
        pf["peak_tflops"] = peak_tf
        pf["peak_source"] = peak_src
        pf["note"] = ("hpc_extend_attn, 64 q / 8 kv heads, d128, bf16 or e4m3 cache; useful causal "
                      "FLOPs (4*128*H_q per visible key and query row) / CUDA-event time, "
                      "L2 flushed between launches")
        line["prefill"] = pf

    # ---- context: a plain device-to-device copy on this GPU (read + write bytes)
    if not args.no_copy_probe:
        n = 1 << 30
        src = torch.empty(n, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        for _ in range(3):
            dst.copy_(src)
        es = [[mk(), mk()] for _ in range(10)]
        for a, b in es:
            a.record(stream)
            dst.copy_(src)
            b.record(stream)
        torch.cuda.synchronize()
        t = statistics.median(a.elapsed_time(b) for a, b in es)
        line["copy_probe_gbs"] = round(2 * n / (t * 1e-3) / 1e9, 1)
        del src, dst

    plan.destroy()
    if rank == 0:
        emit(line, args)


def main():
    args = parse_args()
    ws, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        else:
            run_hpc(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    main()
