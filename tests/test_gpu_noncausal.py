"""Non-causal ring attention (causal = 0: every query sees every key; [G]
"Step 3" carries the is_causal flag): forward and backward against the
float64 oracle with causal=False, over both placements, both step modes, the
rank-major layout and a ragged block length.  Tolerances as for the causal
path (O 2e-2, LSE 1e-3, dQ/dK/dV 5e-2)."""
import pytest
import torch

from head_context_attention_gb300 import inputs, ops
from oracle import attention
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu

CASES = {
    # name: (S, hq, hkv, d, hp, cp, inner, outer, placement, batch)
    "nc-d64": (1024, 4, 2, 64, 2, 4, 4, 1, 1, 1),
    "nc-d128-double-ring": (1024, 4, 2, 128, 2, 4, 2, 2, 1, 1),
    "nc-ragged": (1200, 2, 1, 128, 1, 3, 3, 1, 1, 1),
    "nc-contiguous": (1000, 4, 2, 64, 2, 4, 2, 2, 0, 1),
    "nc-batch2-g3": (512, 3, 1, 128, 1, 2, 1, 2, 1, 2),
}


def _workload(name):
    S, hq, hkv, d, hp, cp, inner, outer, pl, B = CASES[name]
    return inputs.Workload(name, S, hq, hkv, d, hp, cp, inner, outer, True, placement=pl, batch=B, causal=False)


@pytest.mark.parametrize("mode", [ops.MODE_FUSED, ops.MODE_STEPWISE])
@pytest.mark.parametrize("name", list(CASES))
def test_noncausal_matches_oracle(cuda_device, name, mode):
    w = _workload(name)
    x = inputs.make_inputs(w, device="cuda")
    o, lse, r = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode)
    dq, dk, dv = ops.attn_bwd(w, x["q"], x["k"], x["v"], o, lse, x["do"], o_res=r, mode=mode)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    for b in range(w.batch):
        q, k, v, do = (to64(x[n][b]) for n in ("q", "k", "v", "do"))
        want_o, want_lse = attention.attention_forward(q, k, v, causal=False)
        assert_close("O", to64(o[b]), want_o, 2e-2, 2e-2)
        assert_close("LSE", to64(lse[b]), want_lse, 1e-3, 0.0)
        g = attention.attention_backward(q, k, v, do, causal=False)[:3]
        for nm, got, exp in zip(("dQ", "dK", "dV"), (dq, dk, dv), g):
            assert_close(nm, to64(got[b]), exp, 5e-2, 5e-2)


def test_noncausal_rank_major_and_copy_mode_equal_natural(cuda_device):
    w = _workload("nc-d128-double-ring")
    x = inputs.make_inputs(w, device="cuda")
    o, lse, r = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=ops.MODE_STEPWISE)
    dq, dk, dv = ops.attn_bwd(w, x["q"], x["k"], x["v"], o, lse, x["do"], o_res=r, mode=ops.MODE_STEPWISE)
    p = {n: ops.headctx_pack(x[n], w.cp, w.hp, 1) for n in ("q", "k", "v", "do")}
    rm = ops.LAYOUT_RANK_MAJOR
    un = lambda t: ops.headctx_unpack(t, w.batch, w.cp, w.hp, 1)
    for mode in (ops.MODE_STEPWISE, ops.MODE_STEPWISE_COPY):
        o2, lse2, r2 = ops.attn_fwd(w, p["q"], p["k"], p["v"], mode=mode, layout=rm)
        _, dk2, dv2 = ops.attn_bwd(w, p["q"], p["k"], p["v"], o2, lse2, p["do"], o_res=r2, mode=mode, layout=rm)
        assert torch.equal(un(o2), o) and torch.equal(lse2, lse) and torch.equal(un(r2), r)
        assert torch.equal(un(dk2), dk) and torch.equal(un(dv2), dv)
