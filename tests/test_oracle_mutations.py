"""The oracle's pins catch plausible mistakes.  Each case plants one mistake in
a copy of an oracle function (monkeypatched, CPU only) and checks that at
least one pin test then fails."""
import numpy as np
import pytest

from oracle import attention, merge, repack, schedule
from tests import test_oracle_attention as TA
from tests import test_oracle_merge as TM
from tests import test_oracle_repack as TR
from tests import test_oracle_ring as TRG
from tests import test_oracle_schedule as TS

_orig_fwd = attention.attention_forward
_orig_bwd = attention.attention_backward


def fwd_no_scale(q, k, v, scale=None, causal=True):
    return _orig_fwd(q, k, v, 1.0, causal)


def fwd_strict_mask(q, k, v, scale=None, causal=True):
    """Mask j >= i instead of j > i (drops the diagonal)."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    S, hq, d = q.shape
    g = hq // k.shape[1]
    scale = 1 / np.sqrt(d) if scale is None else scale
    o = np.zeros_like(q)
    lse = np.zeros((hq, S))
    fut = np.arange(S)[None, :] >= np.arange(S)[:, None]
    fut[0, 0] = False
    for h in range(hq):
        s = np.where(fut, -np.inf, scale * q[:, h] @ k[:, h // g].T)
        m = s.max(1, keepdims=True)
        e = np.exp(s - m)
        lse[h] = (m + np.log(e.sum(1, keepdims=True)))[:, 0]
        o[:, h] = e / e.sum(1, keepdims=True) @ v[:, h // g]
    return o, lse


def fwd_k_for_v(q, k, v, scale=None, causal=True):
    return _orig_fwd(q, k, k, scale, causal)


def fwd_gqa_modulo(q, k, v, scale=None, causal=True):
    """Query head h uses kv head h % Hkv instead of h // G."""
    q = np.asarray(q, dtype=np.float64)
    hq, hkv = q.shape[1], k.shape[1]
    idx = [h % hkv for h in range(hq)]
    kk = np.asarray(k)[:, idx]
    vv = np.asarray(v)[:, idx]
    return _orig_fwd(q, kk, vv, scale, causal)


def bwd_ds_sign(q, k, v, do, scale=None, causal=True):
    dq, dk, dv, o, lse, dvec = _orig_bwd(q, k, v, do, scale, causal)
    return -dq, -dk, dv, o, lse, dvec


def bwd_dk_unscaled(q, k, v, do, scale=None, causal=True):
    dq, dk, dv, o, lse, dvec = _orig_bwd(q, k, v, do, scale, causal)
    d = np.asarray(q).shape[2]
    return dq, dk * np.sqrt(d), dv, o, lse, dvec


def merge_linear(o_parts, lse_parts):
    """Weights proportional to L_p instead of exp(L_p)."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    w = np.asarray(lse_parts, dtype=np.float64)
    w = np.where(np.isneginf(w), 0.0, np.abs(w))
    tot = np.where(w.sum(0) == 0, 1.0, w.sum(0))
    return np.einsum("nr,nrd->rd", w / tot, o_parts), np.log(np.exp(lse_parts).sum(0))


def ring_source_wrong_dir(c, t, inner, outer):
    o, i = divmod(t, inner)
    g, l = divmod(c, inner)
    return ((g + o) % outer) * inner + ((l - i) % inner)


def paired_blocks_off_by_one(p_seq, r):
    return r, 2 * p_seq - r


CASES = [
    ("attention_forward", attention, fwd_no_scale,
     [TA.test_forward_matches_brute_force_loops, TA.test_row_zero_sees_only_its_own_key]),
    ("attention_forward", attention, fwd_strict_mask,
     [TA.test_forward_matches_brute_force_loops, TA.test_forward_matches_torch_sdpa_float64]),
    ("attention_forward", attention, fwd_k_for_v,
     [TA.test_forward_matches_torch_sdpa_float64, TA.test_row_zero_sees_only_its_own_key]),
    ("attention_forward", attention, fwd_gqa_modulo,
     [TA.test_forward_matches_brute_force_loops, TA.test_forward_matches_torch_sdpa_float64]),
    ("attention_backward", attention, bwd_ds_sign,
     [TA.test_backward_matches_torch_autograd_float64]),
    ("attention_backward", attention, bwd_dk_unscaled,
     [TA.test_backward_matches_torch_autograd_float64]),
    ("lse_merge", merge, merge_linear,
     [TM.test_two_way_merge_equals_softmax_over_concatenation, TM.test_merge_of_equal_lse_is_mean]),
    ("ring_source", schedule, ring_source_wrong_dir,
     [lambda: TS.test_double_ring_table_properties(8, 4),
      lambda: TS.test_double_ring_table_properties(3, 3)]),
    ("paired_blocks", schedule, paired_blocks_off_by_one,
     [TS.test_paired_blocks_golden, TS.test_zigzag_tokens_golden]),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_planted_mistake_is_caught(monkeypatch, i):
    name, mod, mutant, pins = CASES[i]
    monkeypatch.setattr(mod, name, mutant)
    caught = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught >= 1, f"no pin caught the planted mistake in {name} ({mutant.__name__})"


def test_planted_repack_mistake_is_caught(monkeypatch):
    orig = repack.ulysses_pack

    def swapped(x, P):
        y = orig(x, P)
        return y[:, ::-1].copy()        # destination ranks reversed
    monkeypatch.setattr(repack, "ulysses_pack", swapped)
    with pytest.raises(AssertionError):
        TR.test_ulysses_pack_matches_reshape_and_round_trips(3, 4, 5, 8, 3)


def test_planted_ring_merge_order_mistake_is_caught(monkeypatch):
    """A ring pass that forgets the merge (keeps only the last step) fails."""
    def last_only(o_a, lse_a, o_b, lse_b):
        return np.where(np.isneginf(lse_b)[:, None], o_a, o_b), np.where(np.isneginf(lse_b), lse_a, lse_b)
    monkeypatch.setattr(merge, "lse_merge2", last_only)
    with pytest.raises(AssertionError):
        TRG.test_ring_forward_backward_equal_plain(32, 4, 2, 4, 2, 4, 4, 1, schedule.ZIGZAG)
