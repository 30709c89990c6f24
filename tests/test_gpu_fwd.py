"""Forward parity: the CUDA ring-attention forward against the float64 oracle,
element by element, on seeded bf16 inputs (O within atol 2e-2 / rtol 2e-2,
LSE within 1e-3 absolute).  O + o_res, the forward's fp32 result before its
bf16 rounding, is checked ten times tighter: the P V product takes fp16
probabilities (unit roundoff 2^-11) with fp32 accumulation."""
import numpy as np
import pytest
import torch

from head_context_attention_gb300 import inputs, ops
from oracle import attention, ring
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3

CASES = {
    # name: (S, hq, hkv, d, hp, cp, inner, outer, placement, batch)
    "tiny-gqa-s1k": (1024, 4, 2, 64, 2, 4, 4, 1, 1, 1),
    "d128-double-ring": (1024, 4, 2, 128, 2, 4, 2, 2, 1, 1),
    "ragged-blocks": (1200, 2, 1, 128, 1, 3, 3, 1, 1, 1),        # blk = 200: partial tiles
    "odd-group": (512, 3, 1, 128, 1, 2, 2, 1, 1, 1),             # G = 3
    "contiguous": (1000, 4, 2, 64, 2, 4, 2, 2, 0, 1),            # blk = 250
    "batch2": (512, 4, 1, 128, 1, 2, 1, 2, 1, 2),
    "tiny-blocks": (96, 2, 2, 64, 2, 3, 3, 1, 1, 1),             # blk = 16 < one tile
    "single-rank": (384, 2, 1, 128, 1, 1, 1, 1, 1, 1),
    "g8-cp8": (2048, 16, 2, 128, 2, 8, 4, 2, 1, 1),
}


def _workload(name):
    S, hq, hkv, d, hp, cp, inner, outer, pl, B = CASES[name]
    return inputs.Workload(name, S, hq, hkv, d, hp, cp, inner, outer, False, placement=pl, batch=B)


def _oracle(w, x):
    outs = []
    for b in range(w.batch):
        o, lse = attention.attention_forward(to64(x["q"][b]), to64(x["k"][b]), to64(x["v"][b]))
        outs.append((o, lse))
    return np.stack([o for o, _ in outs]), np.stack([l for _, l in outs])


@pytest.mark.parametrize("mode", [ops.MODE_FUSED, ops.MODE_STEPWISE])
@pytest.mark.parametrize("name", list(CASES))
def test_forward_matches_oracle(cuda_device, name, mode):
    w = _workload(name)
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o, lse, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    want_o, want_lse = _oracle(w, x)
    assert_close("O", to64(o), want_o, O_ATOL, O_RTOL)
    assert_close("LSE", to64(lse), want_lse, LSE_ATOL, 0.0)


@pytest.mark.parametrize("mode", [ops.MODE_FUSED, ops.MODE_STEPWISE])
@pytest.mark.parametrize("d", [64, 128])
def test_forward_with_peaky_keys_matches_oracle(cuda_device, d, mode):
    """Keys scaled x8 at 5 % of the positions make a row's running maximum jump
    by more than the lazy-rescale threshold at many tiles of a long walk (16
    paired blocks, 32 key tiles for the last query tile), so O is rescaled
    often.  At d = 64 the scores of a head's next tile are computed while its
    previous P V may still be queued; each rescale first waits for that P V."""
    w = inputs.Workload("peaky-fwd", 4096, 4, 2, d, 2, 8, 4, 2, False, placement=1, peaky_keys=0.05)
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o, lse, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    want_o, want_lse = _oracle(w, x)
    assert_close("O", to64(o), want_o, O_ATOL, O_RTOL)
    assert_close("LSE", to64(lse), want_lse, LSE_ATOL, 0.0)


@pytest.mark.parametrize("d", [64, 128])
def test_forward_with_stepped_key_levels_matches_oracle(cuda_device, d):
    """Every 128-key tile gets its own score level, 0 to 40 in log2 units (key
    feature 0 times query feature 0, the rest small noise), in a seeded order.
    Along a walk the running maximum then meets tiles a few units above it
    (P sums past 2^15 with no rescale: the softmax falls back to the full
    path and keeps its maximum), tiles more than 8 units above it (a rescale)
    and tiles far below it.  Query rows weight the level by 1, 1/2 or 0, so
    one warp mixes rows of each kind."""
    w = inputs.Workload("stepped-levels", 4096, 4, 2, d, 2, 4, 2, 2, False, placement=1)
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    g = torch.Generator().manual_seed(20260)
    ntile = w.seqlen // 128
    level = torch.randint(0, 21, (ntile,), generator=g).double() * 2.0          # log2 units
    a = (level * (d ** 0.5) / np.log2(np.e)).repeat_interleave(128)              # s = a / sqrt(d) in nats
    k = torch.randn(w.batch, w.seqlen, w.hkv, d, generator=g) * 0.05
    k[..., 0] = a.float()[None, :, None]
    q = torch.randn(w.batch, w.seqlen, w.hq, d, generator=g) * 0.05
    wq = torch.tensor([1.0, 0.5, 1.0, 0.0]).repeat(w.seqlen // 4)
    q[..., 0] = wq[None, :, None]
    x["q"] = q.to(torch.bfloat16).cuda()
    x["k"] = k.to(torch.bfloat16).cuda()
    o, lse, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"])
    assert ops.loong_get_device_status() == ops.LOONG_OK
    want_o, want_lse = _oracle(w, x)
    assert_close("O", to64(o), want_o, O_ATOL, O_RTOL)
    assert_close("LSE", to64(lse), want_lse, LSE_ATOL, 0.0)


def test_chunked_oracle_agrees_on_gpu_inputs(cuda_device):
    """The GPU result also matches the second (ring-walking) oracle."""
    w = _workload("d128-double-ring")
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o, lse, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"])
    ro, rl = ring.ring_forward(to64(x["q"][0]), to64(x["k"][0]), to64(x["v"][0]), w.hp, w.cp,
                               w.ring_inner, w.ring_outer)
    assert_close("O", to64(o[0]), ro, O_ATOL, O_RTOL)
    assert_close("LSE", to64(lse[0]), rl, LSE_ATOL, 0.0)


def test_fused_and_stepwise_agree(cuda_device):
    w = _workload("g8-cp8")
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o1, l1, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=ops.MODE_FUSED)
    o2, l2, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=ops.MODE_STEPWISE)
    assert_close("O", to64(o1), to64(o2), 1e-2, 1e-2)
    assert_close("LSE", to64(l1), to64(l2), 1e-4, 0.0)


def test_causal_mask_future_keys_do_not_change_past_rows(cuda_device):
    w = _workload("d128-double-ring")
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o, lse, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"])
    k2, v2 = x["k"].clone(), x["v"].clone()
    k2[:, 700:] = torch.randn_like(k2[:, 700:], dtype=torch.float32).to(torch.bfloat16) * 4
    v2[:, 700:] = 7.0
    o2, lse2, _ = ops.attn_fwd(w, x["q"], k2, v2)
    # rows before 700 see identical keys in an identical order: bit-identical
    assert torch.equal(o[:, :700], o2[:, :700])
    assert torch.equal(lse[:, :, :700], lse2[:, :, :700])
    assert not torch.equal(o[:, 700:], o2[:, 700:])


def test_row_zero_returns_its_value_row(cuda_device):
    w = _workload("tiny-gqa-s1k")
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o, lse, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"])
    G = w.hq // w.hkv
    for h in range(w.hq):
        assert torch.equal(o[0, 0, h], x["v"][0, 0, h // G])
        s = (to64(x["q"][0, 0, h]) @ to64(x["k"][0, 0, h // G])) / np.sqrt(w.head_dim)
        assert abs(float(lse[0, h, 0]) - s) < LSE_ATOL


@pytest.mark.parametrize("name", ["tiny-gqa-s1k", "d128-double-ring", "ragged-blocks", "g8-cp8"])
@pytest.mark.parametrize("mode", [ops.MODE_FUSED, ops.MODE_STEPWISE])
def test_output_residual_carries_the_unrounded_output(cuda_device, name, mode):
    """o_res = bf16(O32 - bf16(O32)): at most half a bf16 spacing of O, and
    O + o_res is O32, within 2e-3 of exact attention."""
    w = _workload(name)
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o, lse, r = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    o64, r64 = to64(o), to64(r)
    assert np.all(np.abs(r64) <= 2.0 ** -8 * np.abs(o64) + 1e-30)
    want_o, _ = _oracle(w, x)
    assert_close("O + o_res", o64 + r64, want_o, 2e-3, 2e-3)
    # the forward without the residual writes the same O and LSE
    o2, lse2, none = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode, res=False)
    assert none is None and torch.equal(o2, o) and torch.equal(lse2, lse)


@pytest.mark.parametrize("exp2", [20, -20])
def test_values_beyond_fp16_range_are_scaled(cuda_device, exp2):
    """V * 2^20 lies far beyond fp16's range and V * 2^-20 far below its normal
    range: the forward stores V * 2^-e in fp16 with its largest value in
    [2^14, 2^15) and multiplies O by 2^e (exact), so O follows V's scale at full
    precision and LSE does not change at all."""
    w = _workload("d128-double-ring")
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o, lse, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"])
    v2 = x["v"] * (2.0 ** exp2)          # exact in bf16
    o2, lse2, r2 = ops.attn_fwd(w, x["q"], x["k"], v2)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    assert torch.equal(lse2, lse)
    assert torch.isfinite(o2.float()).all()
    want_o, _ = _oracle(w, x)
    scaled = (to64(o2) + to64(r2)) * 2.0 ** -exp2
    assert_close("O(V * 2^k) * 2^-k", scaled, want_o, 2e-3, 2e-3)
