"""Pins for oracle/repack.py."""
import numpy as np
import pytest

from oracle import repack, schedule


def _pack_by_reshape(x, P):
    n, p, sl, H, d = x.shape
    y = x.reshape(n, P, sl, P, H // P, d).transpose(0, 3, 1, 2, 4, 5)
    return y.reshape(n, P, P * sl, H // P, d)


@pytest.mark.parametrize("n,P,sl,H,d", [(1, 2, 3, 4, 2), (3, 4, 5, 8, 3), (2, 8, 2, 8, 1)])
def test_ulysses_pack_matches_reshape_and_round_trips(n, P, sl, H, d):
    x = np.arange(n * P * sl * H * d, dtype=np.int64).reshape(n, P, sl, H, d)
    y = repack.ulysses_pack(x, P)
    np.testing.assert_array_equal(y, _pack_by_reshape(x, P))
    np.testing.assert_array_equal(repack.ulysses_unpack(y, P), x)


def test_pack_moves_head_slices_between_ranks():
    # rank q's tokens land at [q*s_local, (q+1)*s_local) on every destination rank p,
    # carrying heads [p*H/P, (p+1)*H/P)
    x = np.zeros((1, 2, 3, 4, 1), dtype=np.int64)
    for q in range(2):
        for t in range(3):
            for h in range(4):
                x[0, q, t, h, 0] = 100 * q + 10 * t + h
    y = repack.ulysses_pack(x, 2)
    assert y[0, 1, 4, 0, 0] == 100 * 1 + 10 * 1 + 2   # p=1, q=1, t=1, h'=0 -> head 2
    assert y[0, 0, 2, 1, 0] == 10 * 2 + 1             # p=0, q=0, t=2, h'=1 -> head 1


def test_headctx_pack_with_zigzag_round_trip():
    S, H, d, cp, P = 32, 4, 2, 4, 2
    x = np.arange(S * H * d).reshape(S, H, d)
    y = repack.headctx_pack(x, cp, P)
    assert y.shape == (cp, P, S // cp, H // P, d)
    np.testing.assert_array_equal(repack.headctx_unpack(y, cp, P), x)
    # rank c, head rank p sees its zigzag tokens for its head slice
    for c in range(cp):
        toks = schedule.rank_tokens(S, cp, c)
        for p in range(P):
            np.testing.assert_array_equal(y[c, p], x[toks][:, p * 2:(p + 1) * 2])
