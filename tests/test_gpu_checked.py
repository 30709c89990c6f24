"""The checked library (libloong_attn_checked.so, built with LOONG_CHECKED):
every TMA coordinate, bulk-copy range and plain global store is checked
against its tensor on the device.  On the parity cases of the other tests it
trips no check (loong_get_device_status stays LOONG_OK) and gives the regular
library's results (dQ up to the order of its fp32 reductions)."""
import contextlib

import pytest
import torch

from head_context_attention_gb300 import inputs, ops
from tests.test_gpu_fwd import CASES, _workload
from tests.test_gpu_layout import _pack, _unpack, _within_one_bf16_spacing

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def _library(path):
    saved = ops.LIB_PATH, ops._lib
    ops.LIB_PATH, ops._lib = path, None
    try:
        yield ops.lib()
    finally:
        ops.LIB_PATH, ops._lib = saved


def _pass(w, x, mode, layout):
    t = {n: _pack(w, x[n]) for n in ("q", "k", "v", "do")} if layout == ops.LAYOUT_RANK_MAJOR else x
    o, lse, r = ops.attn_fwd(w, t["q"], t["k"], t["v"], mode=mode, layout=layout)
    dq, dk, dv = ops.attn_bwd(w, t["q"], t["k"], t["v"], o, lse, t["do"], o_res=r, mode=mode, layout=layout)
    st = ops.loong_get_device_status()
    if layout == ops.LAYOUT_RANK_MAJOR:
        o, dq, dk, dv, r = (_unpack(w, a) for a in (o, dq, dk, dv, r))
    return st, (o, lse, dq, dk, dv, r)


@pytest.mark.parametrize("mode,layout", [(ops.MODE_FUSED, ops.LAYOUT_NATURAL),
                                         (ops.MODE_STEPWISE, ops.LAYOUT_NATURAL),
                                         (ops.MODE_FUSED, ops.LAYOUT_RANK_MAJOR),
                                         (ops.MODE_STEPWISE_COPY, ops.LAYOUT_RANK_MAJOR)])
@pytest.mark.parametrize("name", list(CASES))
def test_checked_library_trips_no_check_and_agrees(cuda_device, name, mode, layout):
    w = _workload(name)
    x = inputs.make_inputs(w, device="cuda", with_do=True)
    st, want = _pass(w, x, mode, layout)
    assert st == ops.LOONG_OK
    with _library(ops.CHECKED_LIB_PATH):
        st, got = _pass(w, x, mode, layout)
    assert st == ops.LOONG_OK, "an address check failed"
    for i in (0, 1, 3, 4, 5):   # O, LSE, dK, dV, O's residual
        assert torch.equal(got[i], want[i]), i
    assert _within_one_bf16_spacing(got[2], want[2])


@pytest.mark.parametrize("name", ["d128-double-ring", "ragged-blocks", "contiguous"])
def test_checked_library_non_causal_and_rank_forward(cuda_device, name):
    w = _workload(name).with_(causal=False)
    x = inputs.make_inputs(w, device="cuda", with_do=True)
    st, want = _pass(w, x, ops.MODE_FUSED, ops.LAYOUT_NATURAL)
    assert st == ops.LOONG_OK
    with _library(ops.CHECKED_LIB_PATH):
        st, got = _pass(w, x, ops.MODE_FUSED, ops.LAYOUT_NATURAL)
        assert st == ops.LOONG_OK
        desc = ops.make_desc(w)
        ws = ops.workspace(desc, 0)
        o = torch.full_like(x["q"], float("nan"))
        lse = torch.full((w.batch, w.hq, w.seqlen), float("nan"), device="cuda")
        for c in range(w.cp):
            ops.loong_attn_fwd_ranks(desc, c, c + 1, x["q"], x["k"], x["v"], o, lse, ws)
        assert ops.loong_get_device_status() == ops.LOONG_OK
    assert torch.equal(got[0], want[0]) and torch.equal(o, want[0]) and torch.equal(lse, want[1])
