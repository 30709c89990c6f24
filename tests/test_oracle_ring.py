"""The chunked ring oracle against the plain oracle: any (hp, cp) split,
placement, ring shape and step order gives plain attention (to rounding)."""
import numpy as np
import pytest

from oracle import attention, ring, schedule


def _inputs(seed, S, hq, hkv, d):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(s) for s in ((S, hq, d), (S, hkv, d), (S, hkv, d), (S, hq, d))]


@pytest.mark.parametrize("S,hq,hkv,d,hp,cp,inner,outer,placement", [
    (32, 4, 2, 4, 2, 4, 4, 1, schedule.ZIGZAG),
    (48, 4, 2, 4, 2, 4, 2, 2, schedule.ZIGZAG),
    (48, 8, 4, 3, 4, 6, 3, 2, schedule.ZIGZAG),
    (40, 2, 1, 5, 1, 4, 1, 4, schedule.CONTIGUOUS),
    (36, 4, 4, 2, 1, 3, 3, 1, schedule.CONTIGUOUS),
])
def test_ring_forward_backward_equal_plain(S, hq, hkv, d, hp, cp, inner, outer, placement):
    q, k, v, do = _inputs(S + cp, S, hq, hkv, d)
    o, lse = attention.attention_forward(q, k, v)
    dq, dk, dv, *_ = attention.attention_backward(q, k, v, do)
    ro, rl = ring.ring_forward(q, k, v, hp, cp, inner, outer, placement)
    np.testing.assert_allclose(ro, o, atol=1e-12)
    np.testing.assert_allclose(rl, lse, atol=1e-12)
    g = ring.ring_backward(q, k, v, do, ro, rl, hp, cp, inner, outer, placement)
    for a, b in zip(g, (dq, dk, dv)):
        np.testing.assert_allclose(a, b, atol=1e-11)


def test_ring_result_independent_of_step_order():
    q, k, v, _ = _inputs(5, 32, 4, 2, 4)
    base, bl = ring.ring_forward(q, k, v, 2, 4, 2, 2)
    for order in ([3, 1, 0, 2], [2, 3, 1, 0]):
        o, l = ring.ring_forward(q, k, v, 2, 4, 2, 2, step_order=order)
        np.testing.assert_allclose(o, base, atol=1e-12)
        np.testing.assert_allclose(l, bl, atol=1e-12)


def test_full_attention_after_step_zero_is_wrong_for_paired_blocks():
    """The guide's step masks only step 0; at later steps some paired blocks are
    wholly in the future, so unmasked attention there would leak future keys."""
    S, cp = 16, 2
    q, k, v, _ = _inputs(6, S, 1, 1, 2)
    # rank 0 (blocks 0 and 3) at step 1 holds rank 1's blocks 1 and 2
    qpos = schedule.rank_tokens(S, cp, 0)
    kpos = schedule.rank_tokens(S, cp, 1)
    future = kpos[None, :] > qpos[:, None]
    assert future.any() and not future.all()
    # block A of rank 0 must skip both of rank 1's blocks; block B sees both in full
    assert future[:4].all() and not future[4:].any()
