"""The allocation-free backward entry point, for callers that cannot allocate
device memory (a plugin whose host framework owns the whole device pool, a loop
that cannot take cudaMalloc's implicit synchronisation).  It is called through
the C ABI and must match loong_attn_bwd, within the backward parity tolerance,
on two calls in a row (the second finds the first call's contents in the
shared scratch array).  Collected last so a failure here cannot hide others."""
import ctypes

import pytest
import torch

from head_context_attention_gb300 import inputs, ops
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu

ATOL, RTOL = 5e-2, 5e-2


def _call(desc, x, o, lse):
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = ops.lib().loong_attn_bwd_noalloc(ctypes.byref(desc), p(x["q"]), p(x["k"]), p(x["v"]), p(o), p(lse),
                                          p(x["do"]), p(dq), p(dk), p(dv),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ops.LOONG_OK, ops.lib().loong_status_string(st)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    return dq, dk, dv


@pytest.mark.parametrize("mode", [ops.MODE_FUSED, ops.MODE_STEPWISE])
def test_noalloc_backward_matches_workspace_backward_twice(cuda_device, mode):
    w = inputs.Workload("noalloc", 1024, 4, 2, 128, 2, 4, 2, 2, True)
    desc = ops.make_desc(w, mode)
    assert ops.loong_attn_workspace_size(desc, 1) <= ops.NOALLOC_SCRATCH_BYTES
    x = inputs.make_inputs(w, device="cuda")
    o, lse = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode)
    want = ops.attn_bwd(w, x["q"], x["k"], x["v"], o, lse, x["do"], mode=mode)
    for _ in range(2):
        got = _call(desc, x, o, lse)
        for nm, g, e in zip(("dQ", "dK", "dV"), got, want):
            assert_close(nm, to64(g), to64(e), ATOL, RTOL)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    w = inputs.WORKLOADS["llama3-8b-s128k"]
    desc = ops.make_desc(w)
    assert ops.loong_attn_workspace_size(desc, 1) > ops.NOALLOC_SCRATCH_BYTES
    st = ops.lib().loong_attn_bwd_noalloc(ctypes.byref(desc), *([ctypes.c_void_p(16)] * 3), ctypes.c_void_p(16),
                                          ctypes.c_void_p(16), *([ctypes.c_void_p(16)] * 4), None)
    assert st == ops.LOONG_ERR_WORKSPACE
