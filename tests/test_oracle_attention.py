"""Pins for oracle/attention.py: brute force, closed forms, a library special
case, finite differences and the gradient-sum invariants."""
import math

import numpy as np
import pytest
import torch

from oracle import attention


def _rand(rng, S, hq, hkv, d):
    return (rng.standard_normal((S, hq, d)), rng.standard_normal((S, hkv, d)),
            rng.standard_normal((S, hkv, d)), rng.standard_normal((S, hq, d)))


def _brute_forward(q, k, v, scale):
    """Textbook causal softmax attention with scalar Python loops."""
    S, hq, d = len(q), len(q[0]), len(q[0][0])
    g = hq // len(k[0])
    o = [[[0.0] * d for _ in range(hq)] for _ in range(S)]
    lse = [[0.0] * S for _ in range(hq)]
    for h in range(hq):
        kv = h // g
        for i in range(S):
            logits = []
            for j in range(i + 1):
                dot = 0.0
                for c in range(d):
                    dot += q[i][h][c] * k[j][kv][c]
                logits.append(scale * dot)
            den = sum(math.exp(x) for x in logits)
            lse[h][i] = math.log(den)
            for c in range(d):
                o[i][h][c] = sum(math.exp(logits[j]) / den * v[j][kv][c] for j in range(i + 1))
    return np.array(o), np.array(lse)


def test_forward_matches_brute_force_loops():
    rng = np.random.default_rng(11)
    q, k, v, _ = _rand(rng, 7, 4, 2, 3)
    scale = 1 / math.sqrt(3)
    o, lse = attention.attention_forward(q, k, v)
    ob, lb = _brute_forward(q.tolist(), k.tolist(), v.tolist(), scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-13)


def test_forward_matches_torch_sdpa_float64():
    rng = np.random.default_rng(12)
    q, k, v, _ = _rand(rng, 33, 8, 2, 16)
    o, _ = attention.attention_forward(q, k, v)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None].repeat_interleave(4, dim=1)
    tv = torch.from_numpy(v).permute(1, 0, 2)[None].repeat_interleave(4, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_row_zero_sees_only_its_own_key():
    rng = np.random.default_rng(13)
    q, k, v, _ = _rand(rng, 9, 4, 2, 5)
    o, lse = attention.attention_forward(q, k, v)
    for h in range(4):
        np.testing.assert_array_equal(o[0, h], v[0, h // 2])
        assert lse[h, 0] == pytest.approx(q[0, h] @ k[0, h // 2] / math.sqrt(5), abs=1e-14)


def test_identical_keys_give_running_mean_of_values():
    rng = np.random.default_rng(14)
    S, d = 12, 4
    q = rng.standard_normal((S, 2, d))
    k = np.tile(rng.standard_normal((1, 1, d)), (S, 1, 1))
    v = rng.standard_normal((S, 1, d))
    o, lse = attention.attention_forward(q, k, v)
    for i in range(S):
        for h in range(2):
            np.testing.assert_allclose(o[i, h], v[:i + 1, 0].mean(axis=0), atol=1e-13)
            s = q[i, h] @ k[0, 0] / math.sqrt(d)
            assert lse[h, i] == pytest.approx(s + math.log(i + 1), abs=1e-12)


def test_causal_mask_ignores_future_keys():
    rng = np.random.default_rng(15)
    q, k, v, _ = _rand(rng, 16, 2, 1, 4)
    o, lse = attention.attention_forward(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[9:] = rng.standard_normal(k2[9:].shape) * 50
    v2[9:] = rng.standard_normal(v2[9:].shape) * 50
    o2, lse2 = attention.attention_forward(q, k2, v2)
    np.testing.assert_array_equal(o[:9], o2[:9])
    np.testing.assert_array_equal(lse[:, :9], lse2[:, :9])
    assert np.abs(o[9:] - o2[9:]).max() > 1e-3


def test_gqa_equals_repeated_kv_heads():
    rng = np.random.default_rng(16)
    q, k, v, do = _rand(rng, 10, 6, 2, 4)
    o, lse = attention.attention_forward(q, k, v)
    o2, lse2 = attention.attention_forward(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1))
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)


def _loss(q, k, v, do):
    o, _ = attention.attention_forward(q, k, v)
    return float(np.sum(o * do))


@pytest.mark.parametrize("which", ["q", "k", "v"])
def test_backward_matches_central_differences(which):
    rng = np.random.default_rng(17)
    q, k, v, do = _rand(rng, 6, 4, 2, 3)
    dq, dk, dv, *_ = attention.attention_backward(q, k, v, do)
    x = {"q": q, "k": k, "v": v}[which]
    grad = {"q": dq, "k": dk, "v": dv}[which]
    eps = 1e-6
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        old = x[idx]
        x[idx] = old + eps
        fp = _loss(q, k, v, do)
        x[idx] = old - eps
        fm = _loss(q, k, v, do)
        x[idx] = old
        num[idx] = (fp - fm) / (2 * eps)
    np.testing.assert_allclose(grad, num, atol=1e-8, rtol=0)


def test_backward_matches_torch_autograd_float64():
    rng = np.random.default_rng(18)
    q, k, v, do = _rand(rng, 20, 4, 2, 8)
    dq, dk, dv, *_ = attention.attention_backward(q, k, v, do)
    tq = torch.from_numpy(q).requires_grad_()
    tk = torch.from_numpy(k).requires_grad_()
    tv = torch.from_numpy(v).requires_grad_()
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.permute(1, 0, 2)[None].repeat_interleave(2, dim=1),
        tv.permute(1, 0, 2)[None].repeat_interleave(2, dim=1), is_causal=True)
    ref[0].permute(1, 0, 2).backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_gradient_sum_invariants():
    rng = np.random.default_rng(19)
    q, k, v, do = _rand(rng, 24, 4, 2, 8)
    dq, dk, dv, *_ = attention.attention_backward(q, k, v, do)
    # rows of dS sum to zero, so sum_j dK_j = 0 per kv head
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    # rows of P sum to one, so sum_j dV_j = sum over the group of sum_i dO_i
    grp = do.reshape(24, 2, 2, 8).sum(axis=(0, 2))
    np.testing.assert_allclose(dv.sum(axis=0), grp, atol=1e-12)


def test_sampled_rows_match_full():
    rng = np.random.default_rng(20)
    q, k, v, do = _rand(rng, 40, 4, 2, 8)
    o, lse = attention.attention_forward(q, k, v)
    dq, dk, dv, *_ = attention.attention_backward(q, k, v, do)
    rows = [0, 3, 17, 39]
    heads = [1, 2]
    ro, rl = attention.attention_rows(q, k, v, rows, heads)
    rdq = attention.attention_backward_rows(q, k, v, do, rows, heads)
    for a, h in enumerate(heads):
        np.testing.assert_allclose(ro[a], o[rows, h], atol=1e-13)
        np.testing.assert_allclose(rl[a], lse[h, rows], atol=1e-13)
        np.testing.assert_allclose(rdq[a], dq[rows, h], atol=1e-12)
    keys = [5, 30, 39]
    sk, sv = attention.attention_backward_keys(q, k, v, do, keys, kv_head=1)
    np.testing.assert_allclose(sk, dk[keys, 1], atol=1e-12)
    np.testing.assert_allclose(sv, dv[keys, 1], atol=1e-12)


def test_round_bf16_matches_torch_conversion():
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-6, 6, 100000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, -3.5e-30]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(attention.round_bf16(x), want)


def test_d_from_bf16_o_only_moves_the_d_term():
    rng = np.random.default_rng(22)
    q, k, v, do = _rand(rng, 16, 4, 2, 8)
    exact = attention.attention_backward(q, k, v, do)
    rounded = attention.attention_backward(q, k, v, do, d_from_bf16_o=True)
    np.testing.assert_array_equal(exact[2], rounded[2])              # dV has no D term
    o = exact[3]
    np.testing.assert_allclose(rounded[5], np.einsum("shd,shd->hs", do, attention.round_bf16(o)),
                               atol=1e-15)
    assert 0 < np.abs(rounded[0] - exact[0]).max() < 1e-2


# ---- non-causal attention ([G] "Step 3" carries an is_causal flag)
def test_noncausal_forward_matches_torch_sdpa_float64():
    rng = np.random.default_rng(21)
    q, k, v, _ = _rand(rng, 29, 8, 2, 16)
    o, lse = attention.attention_forward(q, k, v, causal=False)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None].repeat_interleave(4, dim=1)
    tv = torch.from_numpy(v).permute(1, 0, 2)[None].repeat_interleave(4, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=False)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    s = torch.einsum("hqd,hkd->hqk", tq[0], tk[0]) / math.sqrt(16)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_noncausal_output_ignores_key_order():
    """Without the mask a query attends to a set of keys: permuting the K/V
    rows together leaves every output unchanged (a mask bug would not)."""
    rng = np.random.default_rng(22)
    q, k, v, _ = _rand(rng, 17, 4, 2, 8)
    perm = rng.permutation(17)
    o1, l1 = attention.attention_forward(q, k, v, causal=False)
    o2, l2 = attention.attention_forward(q, k[perm], v[perm], causal=False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
    oc, _ = attention.attention_forward(q, k, v, causal=True)
    assert np.abs(oc[0] - o1[0]).max() > 1e-3   # row 0 sees all keys here, only key 0 when causal


def test_noncausal_backward_matches_torch_autograd_float64():
    rng = np.random.default_rng(23)
    q, k, v, do = _rand(rng, 19, 4, 2, 8)
    dq, dk, dv, *_ = attention.attention_backward(q, k, v, do, causal=False)
    tq = torch.from_numpy(q).requires_grad_()
    tk = torch.from_numpy(k).requires_grad_()
    tv = torch.from_numpy(v).requires_grad_()
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.permute(1, 0, 2)[None].repeat_interleave(2, dim=1),
        tv.permute(1, 0, 2)[None].repeat_interleave(2, dim=1), is_causal=False)
    ref[0].permute(1, 0, 2).backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)
