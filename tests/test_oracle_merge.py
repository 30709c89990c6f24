"""Pins for oracle/merge.py."""
import numpy as np

from oracle import merge


def _softmax_attn(s, v):
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e @ v / e.sum(axis=1, keepdims=True), (m + np.log(e.sum(axis=1, keepdims=True)))[:, 0]


def test_two_way_merge_equals_softmax_over_concatenation():
    rng = np.random.default_rng(1)
    s = rng.standard_normal((6, 11)) * 3
    v = rng.standard_normal((11, 5))
    oa, la = _softmax_attn(s[:, :4], v[:4])
    ob, lb = _softmax_attn(s[:, 4:], v[4:])
    o, lse = merge.lse_merge2(oa, la, ob, lb)
    oref, lref = _softmax_attn(s, v)
    np.testing.assert_allclose(o, oref, atol=1e-14)
    np.testing.assert_allclose(lse, lref, atol=1e-14)


def test_n_way_merge_any_partition_and_order():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((5, 30)) * 4
    v = rng.standard_normal((30, 3))
    cuts = [0, 3, 4, 17, 29, 30]
    parts = [_softmax_attn(s[:, a:b], v[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    oref, lref = _softmax_attn(s, v)
    for perm in ([0, 1, 2, 3, 4], [4, 2, 0, 3, 1]):
        o, lse = merge.lse_merge(np.stack([parts[i][0] for i in perm]),
                                 np.stack([parts[i][1] for i in perm]))
        np.testing.assert_allclose(o, oref, atol=1e-14)
        np.testing.assert_allclose(lse, lref, atol=1e-14)


def test_empty_partial_is_identity_and_all_empty_is_zero():
    rng = np.random.default_rng(3)
    o = rng.standard_normal((4, 3))
    lse = rng.standard_normal(4)
    z, zl = np.zeros((4, 3)), np.full(4, -np.inf)
    mo, ml = merge.lse_merge2(o, lse, z, zl)
    np.testing.assert_array_equal(mo, o)
    np.testing.assert_array_equal(ml, lse)
    mo, ml = merge.lse_merge2(z, zl, z, zl)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))
    assert not np.any(np.isnan(mo))


def test_merge_of_equal_lse_is_mean():
    o1 = np.array([[1.0, 2.0]])
    o2 = np.array([[3.0, -2.0]])
    l = np.array([0.7])
    o, lse = merge.lse_merge2(o1, l, o2, l)
    np.testing.assert_allclose(o, [[2.0, 0.0]], atol=1e-15)
    np.testing.assert_allclose(lse, [0.7 + np.log(2.0)], atol=1e-15)


def test_merge_is_stable_for_large_lse():
    o1 = np.array([[1.0]])
    o2 = np.array([[5.0]])
    o, lse = merge.lse_merge2(o1, np.array([1000.0]), o2, np.array([1000.0 + np.log(3.0)]))
    np.testing.assert_allclose(o, [[4.0]], atol=1e-12)
    np.testing.assert_allclose(lse, [1000.0 + np.log(4.0)], atol=1e-12)
