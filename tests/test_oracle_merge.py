"""Pins for the oracle's split-softmax merge: split-then-merge equals the
unsplit softmax for every split point, and the oracle's decode equals the
merge of its own slices."""
import numpy as np
import pytest

from oracle import merge_ref


def _direct(scores, v):
    e = np.exp(scores - scores.max())
    return (e @ v) / e.sum(), scores.max() + np.log(e.sum())


@pytest.mark.parametrize("n", [1, 2, 5, 64, 130])
def test_every_two_way_split_equals_unsplit(n):
    rng = np.random.default_rng(n)
    s = rng.normal(size=n) * 3
    v = rng.normal(size=(n, 16))
    ref_o, ref_l = _direct(s, v)
    for cut in range(1, n):
        o, l = merge_ref.merge_states([merge_ref.partial_state(s[:cut], v[:cut]),
                                       merge_ref.partial_state(s[cut:], v[cut:])])
        np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-13)
        assert l == pytest.approx(ref_l, rel=1e-13, abs=1e-13)


def test_many_way_random_splits_and_order_independence():
    rng = np.random.default_rng(1)
    for _ in range(50):
        n = int(rng.integers(2, 400))
        s = rng.normal(size=n) * 5
        v = rng.normal(size=(n, 8))
        k = int(rng.integers(2, min(n, 20) + 1))
        cuts = sorted(rng.choice(np.arange(1, n), size=k - 1, replace=False).tolist())
        bounds = [0] + cuts + [n]
        st = [merge_ref.partial_state(s[a:b], v[a:b]) for a, b in zip(bounds, bounds[1:])]
        o1, l1 = merge_ref.merge_states(st)
        o2, l2 = merge_ref.merge_states(st[::-1])
        ref_o, ref_l = _direct(s, v)
        np.testing.assert_allclose(o1, ref_o, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(o2, ref_o, rtol=1e-11, atol=1e-13)
        assert l1 == pytest.approx(ref_l, rel=1e-13) and l2 == pytest.approx(ref_l, rel=1e-13)


def test_single_state_and_extreme_offsets():
    s = np.array([1000.0, 999.0, -1000.0])
    v = np.eye(3)
    m, l, o = merge_ref.partial_state(s, v)
    assert m == 1000.0
    out, lse = merge_ref.merge_states([(m, l, o)])
    e1 = np.exp(-1.0)
    np.testing.assert_allclose(out, [1 / (1 + e1), e1 / (1 + e1), 0.0], rtol=1e-14, atol=1e-300)
    assert lse == pytest.approx(1000.0 + np.log1p(e1), rel=1e-15)
    with pytest.raises(ValueError):
        merge_ref.merge_states([])
