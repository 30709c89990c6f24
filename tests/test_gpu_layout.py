"""The rank-major layout and the rank-restricted forward.

* RANK_MAJOR: the kernels read and write [B*cp, hp, S/cp, H/hp, d], the layout
  each emulated rank holds after the Ulysses exchange (loong_headctx_pack).
  The end-to-end 2D-attention path natural -> pack -> ring forward / backward
  on the packed tensors -> inverse pack gives what the natural layout gives:
  the same tiles in the same order, so O, LSE, dK and dV are equal bit for
  bit.  dQ is summed by fp32 reductions whose order between CTAs is not fixed,
  so it is equal to within one bf16 spacing (plus the reordering error of
  sums that cancel), as two runs of the natural layout are.  The natural path itself is
  checked against the oracle elsewhere; one case here checks the packed path
  against the oracle directly.
* loong_attn_fwd_ranks: one ring rank's query rows at a time; their union is
  the full forward, bit for bit, and rows of other ranks are not touched.
"""
import pytest
import torch

from head_context_attention_gb300 import inputs, ops
from oracle import attention, schedule
from tests.helpers import assert_close, to64
from tests.test_gpu_fwd import CASES, _workload

pytestmark = pytest.mark.gpu

GATHER = {1: 1, 0: 2}   # placement -> headctx_pack gather (paired / contiguous blocks)


def _pack(w, t):
    return ops.headctx_pack(t, w.cp, w.hp, GATHER[w.placement])


def _unpack(w, t):
    return ops.headctx_unpack(t, w.batch, w.cp, w.hp, GATHER[w.placement])


def _within_one_bf16_spacing(a, b):
    """One bf16 spacing, plus 2^-16 max|b| for the fp32 sums that cancel: S/128
    tile partials added in another order move an fp32 sum by about
    (S/128) 2^-24 times the largest partial, which is more than a bf16 spacing
    of a near-zero result.  Two runs of the natural layout differ the same way
    (measured: at most 2.6e-9 max|dQ| beyond one spacing)."""
    a, b = a.double(), b.double()
    bound = 2.0 ** -7 * torch.maximum(a.abs(), b.abs()) + 2.0 ** -16 * b.abs().max()
    return bool(((a - b).abs() <= bound).all())


@pytest.mark.parametrize("mode", [ops.MODE_FUSED, ops.MODE_STEPWISE])
@pytest.mark.parametrize("name", list(CASES))
def test_rank_major_path_equals_natural(cuda_device, name, mode):
    w = _workload(name)
    x = inputs.make_inputs(w, device="cuda", with_do=True)
    o_n, lse_n, r_n = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode)
    dq_n, dk_n, dv_n = ops.attn_bwd(w, x["q"], x["k"], x["v"], o_n, lse_n, x["do"], o_res=r_n, mode=mode)
    p = {n: _pack(w, x[n]) for n in ("q", "k", "v", "do")}
    o_p, lse_p, r_p = ops.attn_fwd(w, p["q"], p["k"], p["v"], mode=mode, layout=ops.LAYOUT_RANK_MAJOR)
    dq_p, dk_p, dv_p = ops.attn_bwd(w, p["q"], p["k"], p["v"], o_p, lse_p, p["do"], o_res=r_p, mode=mode,
                                    layout=ops.LAYOUT_RANK_MAJOR)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    assert torch.equal(_unpack(w, o_p), o_n)
    assert torch.equal(_unpack(w, r_p), r_n)
    assert torch.equal(lse_p, lse_n)
    assert torch.equal(_unpack(w, dk_p), dk_n)
    assert torch.equal(_unpack(w, dv_p), dv_n)
    assert _within_one_bf16_spacing(_unpack(w, dq_p), dq_n)


def test_rank_major_path_matches_oracle(cuda_device):
    w = _workload("d128-double-ring")
    x = inputs.make_inputs(w, device="cuda", with_do=True)
    p = {n: _pack(w, x[n]) for n in ("q", "k", "v", "do")}
    o_p, lse_p, r_p = ops.attn_fwd(w, p["q"], p["k"], p["v"], layout=ops.LAYOUT_RANK_MAJOR)
    dq_p, dk_p, dv_p = ops.attn_bwd(w, p["q"], p["k"], p["v"], o_p, lse_p, p["do"], o_res=r_p,
                                    layout=ops.LAYOUT_RANK_MAJOR)
    q, k, v, do = (to64(x[n][0]) for n in ("q", "k", "v", "do"))
    want_o, want_lse = attention.attention_forward(q, k, v)
    assert_close("O", to64(_unpack(w, o_p)[0]), want_o, 2e-2, 2e-2)
    assert_close("LSE", to64(lse_p[0]), want_lse, 1e-3, 0.0)
    dq, dk, dv = attention.attention_backward(q, k, v, do)[:3]
    assert_close("dQ", to64(_unpack(w, dq_p)[0]), dq, 5e-2, 5e-2)
    assert_close("dK", to64(_unpack(w, dk_p)[0]), dk, 5e-2, 5e-2)
    assert_close("dV", to64(_unpack(w, dv_p)[0]), dv, 5e-2, 5e-2)


def _rank_rows(w, layout, o, c):
    """View of ring rank c's query rows of O, [B, rows, H, d] in either layout."""
    if layout == ops.LAYOUT_RANK_MAJOR:
        return o.view(w.batch, w.cp, *o.shape[1:])[:, c]
    tok = torch.as_tensor(schedule.rank_tokens(w.seqlen, w.cp, c, w.placement), device=o.device)
    return o[:, tok]


@pytest.mark.parametrize("layout", [ops.LAYOUT_NATURAL, ops.LAYOUT_RANK_MAJOR])
@pytest.mark.parametrize("name", ["d128-double-ring", "contiguous", "ragged-blocks", "batch2", "odd-group",
                                  "g8-cp8"])
def test_fwd_ranks_union_is_the_full_forward(cuda_device, name, layout):
    w = _workload(name)
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    if layout == ops.LAYOUT_RANK_MAJOR:
        x = {n: _pack(w, x[n]) for n in ("q", "k", "v")}
    o_full, lse_full, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"], layout=layout, res=False)
    desc = ops.make_desc(w, layout=layout)
    ws = ops.workspace(desc, 0)
    o = torch.full_like(o_full, float("nan"))
    lse = torch.full_like(lse_full, float("nan"))
    ops.loong_attn_fwd_ranks(desc, 0, 1, x["q"], x["k"], x["v"], o, lse, ws)
    torch.cuda.synchronize()
    # rank 0's rows are written, every other row untouched
    assert torch.equal(_rank_rows(w, layout, o, 0), _rank_rows(w, layout, o_full, 0))
    tok0 = torch.as_tensor(schedule.rank_tokens(w.seqlen, w.cp, 0, w.placement), device=lse.device)
    assert torch.equal(lse[:, :, tok0], lse_full[:, :, tok0])
    written = torch.zeros(w.seqlen, dtype=torch.bool, device=lse.device)
    written[tok0] = True
    assert bool(lse[:, :, ~written].isnan().all())
    for c in range(1, w.cp):
        assert bool(_rank_rows(w, layout, o, c).isnan().all())
    if w.cp > 1:
        ops.loong_attn_fwd_ranks(desc, 1, w.cp, x["q"], x["k"], x["v"], o, lse, ws)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    assert torch.equal(o, o_full)
    assert torch.equal(lse, lse_full)


@pytest.mark.parametrize("name", ["d128-double-ring", "contiguous", "ragged-blocks", "batch2", "g8-cp8",
                                  "tiny-blocks", "single-rank"])
def test_stepwise_copy_equals_stepwise(cuda_device, name):
    """STEPWISE_COPY (one ring) and STEPWISE_COPY_AB (blocks A and B on two
    rings) read every step's K/V from the receive buffers the exchange copies
    filled; the arithmetic is STEPWISE's, so the results are equal (dQ up to
    its reduction order)."""
    w = _workload(name)
    x = inputs.make_inputs(w, device="cuda", with_do=True)
    p = {n: _pack(w, x[n]) for n in ("q", "k", "v", "do")}
    rm = ops.LAYOUT_RANK_MAJOR
    res = {}
    # the two-ring variant needs two blocks per rank (paired placement)
    modes = [ops.MODE_STEPWISE, ops.MODE_STEPWISE_COPY] + ([ops.MODE_STEPWISE_COPY_AB] if w.placement == 1 else [])
    for mode in modes:
        o, lse, r = ops.attn_fwd(w, p["q"], p["k"], p["v"], mode=mode, layout=rm)
        res[mode] = (o, lse) + ops.attn_bwd(w, p["q"], p["k"], p["v"], o, lse, p["do"], o_res=r, mode=mode,
                                            layout=rm) + (r,)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    a = res[ops.MODE_STEPWISE]
    for mode in modes[1:]:
        b = res[mode]
        for i in (0, 1, 3, 4, 5):   # O, LSE, dK, dV, O's residual
            assert torch.equal(a[i], b[i]), (mode, i)
        assert _within_one_bf16_spacing(b[2], a[2])
