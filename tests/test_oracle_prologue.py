"""Pins for the prologue oracle (QK-Norm + RoPE + paged KV write): closed
forms and invariants of RMSNorm and rotate-half RoPE, the e4m3 encoder
against torch's float8 conversion, and the cache slot of the new token."""
import math

import numpy as np
import pytest
import torch

from oracle import prologue_ref as P

D = 128


def test_rms_norm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(5, D)) * 3
    y = P.rms_norm(x, np.ones(D), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(P.rms_norm(7.5 * x, np.ones(D), 0.0), y, rtol=1e-13)
    w = rng.normal(size=D)
    np.testing.assert_allclose(P.rms_norm(x, w, 0.0), y * w, rtol=1e-13)
    # eps enters under the root: a constant row c gives c / sqrt(c^2 + eps)
    c, eps = 0.5, 1e-2
    np.testing.assert_allclose(P.rms_norm(np.full(D, c), np.ones(D), eps), c / math.sqrt(c * c + eps))


def test_rope_hand_values_and_identity_at_zero():
    x = np.zeros(D)
    x[3], x[3 + 64] = 1.0, 2.0
    pos, base = 5, 10000.0
    th = pos * base ** (-2 * 3 / D)
    y = P.rope(x, pos, base)
    assert y[3] == pytest.approx(math.cos(th) - 2 * math.sin(th), rel=1e-14)
    assert y[67] == pytest.approx(2 * math.cos(th) + math.sin(th), rel=1e-14)
    assert np.count_nonzero(y) == 2
    rng = np.random.default_rng(1)
    z = rng.normal(size=(3, D))
    np.testing.assert_array_equal(P.rope(z, 0, base), z)
    # pair 0 turns by pos radians, pair 63 by pos * base^(-126/128)
    e0 = np.zeros(D); e0[0] = 1.0; e0[63] = 1.0
    y = P.rope(e0, 12345, base)
    a63 = 12345 * base ** (-126 / 128)
    np.testing.assert_allclose([y[0], y[64], y[63], y[127]],
                               [math.cos(12345), math.sin(12345), math.cos(a63), math.sin(a63)],
                               rtol=1e-12, atol=1e-15)


def test_rope_is_a_rotation_with_relative_positions():
    rng = np.random.default_rng(2)
    q, k = rng.normal(size=D), rng.normal(size=D)
    for base in (10000.0, 1e6):
        # norm preserved, composition adds positions
        np.testing.assert_allclose(np.linalg.norm(P.rope(q, 777, base)), np.linalg.norm(q), rtol=1e-13)
        np.testing.assert_allclose(P.rope(P.rope(q, 300, base), 450, base), P.rope(q, 750, base),
                                   rtol=1e-9, atol=1e-12)
        # the score depends on the position difference only
        s1 = P.rope(q, 1000, base) @ P.rope(k, 990, base)
        s2 = P.rope(q, 20, base) @ P.rope(k, 10, base)
        assert s1 == pytest.approx(s2, rel=1e-9, abs=1e-12)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.normal(size=4000) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    xs = np.clip(xs, -448, 448)
    ref = torch.tensor(xs, dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([P.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_ties_saturation_and_signed_zero():
    assert P.e4m3_encode(1.0625) == 0x38  # halfway 1.0 / 1.125 -> even mantissa (1.0)
    assert P.e4m3_encode(1.1875) == 0x3A  # halfway 1.125 / 1.25 -> 1.25 (even)
    assert P.e4m3_encode(1000.0) == 0x7E and P.e4m3_encode(-1e9) == 0xFE  # saturate
    assert P.e4m3_encode(0.0) == 0x00 and P.e4m3_encode(-0.0) == 0x80
    assert P.e4m3_encode(-1e-6) == 0x80
    for c in range(256):
        v = P.e4m3_decode(c)
        if not math.isnan(v) and c not in (0x80,):
            assert P.e4m3_encode(v) == c


def test_prologue_slot_and_empty_sequence():
    rng = np.random.default_rng(4)
    B, hq, hkv = 3, 16, 2
    q, k, v = rng.normal(size=(B, hq, D)), rng.normal(size=(B, hkv, D)), rng.normal(size=(B, hkv, D))
    bt = np.array([[7, 2, 9], [4, -1, -1], [5, 6, -1]])
    lens = [130, 0, 64]
    qo, ko, vo, slots = P.prologue(q, k, v, lens, bt, np.ones(D), np.ones(D), 1e-6, 1e4)
    assert slots == [(9, 1), None, (5, 63)]
    np.testing.assert_array_equal(qo[1], 0) and np.testing.assert_array_equal(vo, v)
    np.testing.assert_allclose(qo[0], P.rope(P.rms_norm(q[0], np.ones(D), 1e-6), 129, 1e4))
    np.testing.assert_allclose(ko[2], P.rope(P.rms_norm(k[2], np.ones(D), 1e-6), 63, 1e4))
