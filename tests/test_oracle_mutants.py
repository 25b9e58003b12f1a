"""Mistakes planted in the oracle (on the CPU) must fail its pins.

Each mutant is a copy of oracle/decode_ref.c with one plausible slip (a
dropped term, a wrong sign or index, a swapped operand), compiled into a
temporary library. The pin battery below -- the independent brute force
on BF16 and FP8 inputs with several KV heads and ragged tails, the format
tables checked against torch, and the empty-sequence rule -- must reject
every one of them, and must accept the unmodified source.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_pins import _brute, _mk

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "decode_ref.c")).read()

MUTANTS = {
    "kv_head_map_interleaved": ("int j = h * G + g;", "int j = g * J->num_kv_heads + h;"),
    "softmax_scale_dropped": ("s[t] = J->softmax_scale * acc;", "s[t] = acc;"),
    "k_slot_off_by_one": ("int slot = t % ORACLE_BLOCK;\n      double acc",
                          "int slot = (t + 1) % ORACLE_BLOCK;\n      double acc"),
    "v_block_first_only": ("long blk = J->block_table[(long)b * J->max_blocks + t / ORACLE_BLOCK];\n      int slot = t % ORACLE_BLOCK;\n      double p",
                           "long blk = J->block_table[(long)b * J->max_blocks];\n      int slot = t % ORACLE_BLOCK;\n      double p"),
    "e4m3_bias_8": ("e - 7);", "e - 8);"),
    "e4m3_subnormal_exp": ("(double)m / 8.0, -6)", "(double)m / 8.0, -7)"),
    "e4m3_sign_dropped": ("return sign ? -mag : mag;", "return mag;"),
    "lse_without_max": ("m + log(l);", "log(l);"),
    "v_scale_dropped": ("kv_value(J, J->v_cache, J->v_scale,", "kv_value(J, J->v_cache, 1.0,"),
    "k_scale_dropped": ("kv_value(J, J->k_cache, J->k_scale,", "kv_value(J, J->k_cache, 1.0,"),
    "k_and_v_swapped": ("kv_value(J, J->v_cache, J->v_scale,", "kv_value(J, J->k_cache, J->v_scale,"),
    "no_normalisation": ("for (int d = 0; d < D; ++d) o[d] /= l;", ""),
    "max_shift_mismatch": ("double p = exp(s[t] - m);", "double p = exp(s[t]);"),
    "last_token_dropped": ("for (int t = 0; t < N; ++t) {\n      long blk = J->block_table[(long)b * J->max_blocks + t / ORACLE_BLOCK];\n      int slot = t % ORACLE_BLOCK;\n      double p",
                           "for (int t = 0; t < N - 1; ++t) {\n      long blk = J->block_table[(long)b * J->max_blocks + t / ORACLE_BLOCK];\n      int slot = t % ORACLE_BLOCK;\n      double p"),
    "empty_lse_zero": ("J->lse[(long)b * J->num_q_heads + j] = -INFINITY;",
                       "J->lse[(long)b * J->num_q_heads + j] = 0.0;"),
    "bf16_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
}


def _compile(tmp_path, name, src):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           str(c), "-o", str(so), "-lm"])
    return oracle.load_library(str(so))


def _battery(lib) -> bool:
    """True when every pin passes."""
    for lens, hq, hkv, fp8 in [([1, 63, 65, 200], 16, 2, False), ([5, 129, 70], 8, 4, True)]:
        w = _mk(lens, hq, hkv, seed=21, fp8=fp8, slack=2)
        try:
            out, lse = oracle.decode_workload(w, lib=lib)
        except RuntimeError:
            return False
        bo, bl = _brute(w)
        if not (np.allclose(out, bo, rtol=1e-10, atol=1e-12) and
                np.allclose(lse, bl, rtol=1e-12, atol=1e-12)):
            return False
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([lib.oracle_e4m3_to_f64(c) for c in range(256)])
    if not np.array_equal(np.nan_to_num(got, nan=7.0), np.nan_to_num(ref, nan=7.0)):
        return False
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    refb = bits.view(torch.bfloat16).to(torch.float64).numpy()
    gotb = np.array([lib.oracle_bf16_to_f64(c) for c in range(0, 1 << 16, 97)])
    if not np.array_equal(np.nan_to_num(gotb, nan=7.0), np.nan_to_num(refb[::97], nan=7.0)):
        return False
    w = _mk([0, 5], 8, 1, seed=3)
    out, lse = oracle.decode_workload(w, lib=lib)
    if not (np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))):
        return False
    return True


def test_unmodified_source_passes(tmp_path):
    assert _battery(_compile(tmp_path, "orig", SRC))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation anchor for {name} not unique"
    assert not _battery(_compile(tmp_path, name, SRC.replace(old, new)))
