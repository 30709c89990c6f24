"""Backward parity: dQ, dK, dV of the CUDA ring-attention backward against the
float64 oracle's exact gradient on the same seeded bf16 inputs (atol 5e-2 /
rtol 5e-2), plus the gradient-sum invariants.  The CUDA backward forms
D = rowsum(dO * O) from O and the forward's rounding residual of O; the oracle
from its own float64 O.  Without the residual the library forms D from the
bf16 O alone: that path is checked against the oracle's D from O rounded to
bf16, the tensor the forward returns."""
import numpy as np
import pytest

from head_context_attention_gb300 import inputs, ops
from oracle import attention
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu

ATOL, RTOL = 5e-2, 5e-2

CASES = {
    # name: (S, hq, hkv, d, hp, cp, inner, outer, placement, batch)
    "tiny-gqa-s1k": (1024, 4, 2, 64, 2, 4, 4, 1, 1, 1),
    "d128-double-ring": (1024, 4, 2, 128, 2, 4, 2, 2, 1, 1),
    "ragged-blocks": (1200, 2, 1, 128, 1, 3, 3, 1, 1, 1),
    "odd-group": (512, 3, 1, 128, 1, 2, 2, 1, 1, 1),
    "contiguous": (1000, 4, 2, 64, 2, 4, 2, 2, 0, 1),
    "batch2": (512, 4, 1, 128, 1, 2, 1, 2, 1, 2),
    "tiny-blocks": (96, 2, 2, 64, 2, 3, 3, 1, 1, 1),
    "g8-cp8": (2048, 16, 2, 128, 2, 8, 4, 2, 1, 1),
}


def _workload(name):
    S, hq, hkv, d, hp, cp, inner, outer, pl, B = CASES[name]
    return inputs.Workload(name, S, hq, hkv, d, hp, cp, inner, outer, True, placement=pl, batch=B)


def _run(w, mode, res=True):
    x = inputs.make_inputs(w, device="cuda")
    o, lse, o_res = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode, res=res)
    dq, dk, dv = ops.attn_bwd(w, x["q"], x["k"], x["v"], o, lse, x["do"], o_res=o_res, mode=mode)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    return x, (dq, dk, dv)


def _check_against_oracle(w, x, grads, d_from_bf16_o):
    errors = []
    for b in range(w.batch):
        want = attention.attention_backward(to64(x["q"][b]), to64(x["k"][b]), to64(x["v"][b]),
                                            to64(x["do"][b]), d_from_bf16_o=d_from_bf16_o)[:3]
        for nm, got, exp in zip(("dQ", "dK", "dV"), grads, want):
            try:
                assert_close(nm, to64(got[b]), exp, ATOL, RTOL)
            except AssertionError as e:
                errors.append(str(e))
    assert not errors, "\n".join(errors)


@pytest.mark.parametrize("mode", [ops.MODE_FUSED, ops.MODE_STEPWISE])
@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(cuda_device, name, mode):
    w = _workload(name)
    x, grads = _run(w, mode)
    _check_against_oracle(w, x, grads, d_from_bf16_o=False)


@pytest.mark.parametrize("name", ["tiny-gqa-s1k", "d128-double-ring", "g8-cp8"])
def test_backward_without_residual_matches_bf16_o_oracle(cuda_device, name):
    """No residual: D from the bf16 O, as the oracle's d_from_bf16_o reading."""
    w = _workload(name)
    x, grads = _run(w, ops.MODE_FUSED, res=False)
    _check_against_oracle(w, x, grads, d_from_bf16_o=True)


def test_backward_gradient_sums(cuda_device):
    w = _workload("g8-cp8")
    x, (dq, dk, dv) = _run(w, ops.MODE_FUSED)
    G = w.hq // w.hkv
    # sum over keys: scale * sum_i (D_exact,i - D_i) q_i, 0 when D is exact;
    # what remains is the bf16 rounding of S dK values of magnitude ~1
    dk_sum = to64(dk[0]).sum(axis=0)
    assert np.abs(dk_sum).max() < 0.25, np.abs(dk_sum).max()
    do_grp = to64(x["do"][0]).reshape(w.seqlen, w.hkv, G, w.head_dim).sum(axis=(0, 2))
    assert_close("sum dV", to64(dv[0]).sum(axis=0), do_grp, 1.0, 1e-2)
