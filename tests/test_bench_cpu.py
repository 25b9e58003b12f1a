"""Host-side pieces of bench.py (no GPU): the parity report it adds to its
JSON line, comparing the step's output on the oracle's sample sequences with
the oracle's."""
import numpy as np

import bench


def _case(seed=0):
    rng = np.random.default_rng(seed)
    ref_out = rng.standard_normal((3, 8, 128))
    ref_lse = rng.standard_normal((3, 8))
    ref_lse[1] = -np.inf  # an empty sequence
    return ref_out, ref_lse


def test_identical_results_pass_with_zero_error():
    ref_out, ref_lse = _case()
    r = bench.parity_summary(ref_out.copy(), ref_lse.copy(), ref_out, ref_lse)
    assert r["pass"] and r["max_abs_out_err"] == 0 and r["max_abs_lse_err"] == 0
    assert r["lse_inf_match"]


def test_error_at_and_beyond_the_bound():
    ref_out, ref_lse = _case(1)
    out = ref_out.copy()
    j = np.unravel_index(np.argmax(np.abs(ref_out)), ref_out.shape)
    bound = 1e-2 + 1e-2 * abs(ref_out[j])
    out[j] += 0.999 * bound
    assert bench.parity_summary(out, ref_lse, ref_out, ref_lse)["pass"]
    out[j] = ref_out[j] + 1.01 * bound
    r = bench.parity_summary(out, ref_lse, ref_out, ref_lse)
    assert not r["pass"] and 1.0 < r["max_err_over_bound"] < 1.02


def test_lse_error_and_infinities():
    ref_out, ref_lse = _case(2)
    lse = ref_lse.copy()
    lse[0, 0] += 2e-3
    r = bench.parity_summary(ref_out, lse, ref_out, ref_lse)
    assert not r["pass"] and abs(r["max_abs_lse_err"] - 2e-3) < 1e-12
    lse = ref_lse.copy()
    lse[1, 3] = 0.0  # an empty sequence reported with a finite lse
    r = bench.parity_summary(ref_out, lse, ref_out, ref_lse)
    assert not r["pass"] and not r["lse_inf_match"]


def test_time_oracle_keeps_the_last_result():
    # the bench's CPU leg times the oracle and keeps its result for the report
    from paged_gqa_decode_hpc_gb300 import workloads as W
    import oracle
    w = W.make_workload("tiny")
    times, (out, lse) = bench.time_oracle(w, 2, keep=True)
    assert len(times) == 2 and all(t > 0 for t in times)
    ref_out, ref_lse = oracle.decode_workload(w)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)
    assert len(bench.time_oracle(w, 1)) == 1
    r = bench.parity_summary(out, lse, ref_out, ref_lse)
    assert r["pass"]


def test_kernel_source_digest_follows_includes(tmp_path, monkeypatch):
    """The digest that keys the committed ncu traffic figure covers the kernel
    file and every local header it includes, transitively, not the kernel
    file alone: editing an included helper invalidates the figure."""
    csrc = tmp_path / "paged_gqa_decode_hpc_gb300" / "csrc"
    inc = tmp_path / "include"
    csrc.mkdir(parents=True)
    inc.mkdir()
    (csrc / "step_kernel.cu").write_text('#include <cuda.h>\n#include "a.h"\nkernel\n')
    (csrc / "a.h").write_text('#include "b.cuh"\n#include "api.h"\n')
    (csrc / "b.cuh").write_text("helper v1\n")
    (inc / "api.h").write_text("abi v1\n")
    (csrc / "unrelated.cu").write_text("other v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.kernel_source_digest()
    (csrc / "unrelated.cu").write_text("other v2\n")
    assert bench.kernel_source_digest() == d0
    (csrc / "b.cuh").write_text("helper v2\n")
    d1 = bench.kernel_source_digest()
    assert d1 != d0
    (inc / "api.h").write_text("abi v2\n")
    assert bench.kernel_source_digest() != d1


def test_kernel_source_digest_ignores_comments_only(tmp_path, monkeypatch):
    """A comment or whitespace edit keeps the digest (the compiled kernel is
    the same); any code edit changes it."""
    csrc = tmp_path / "paged_gqa_decode_hpc_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    k = csrc / "step_kernel.cu"
    k.write_text('// v1 of a comment\nint f(int x) { /* block */ return x + 1; }\n')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.kernel_source_digest()
    k.write_text('// a different comment\n\nint f(int x) {  /* other\n block */ return x + 1; }\n')
    assert bench.kernel_source_digest() == d0
    k.write_text('// v1 of a comment\nint f(int x) { /* block */ return x + 2; }\n')
    assert bench.kernel_source_digest() != d0
