"""The allocation-free backward entry point, for callers that cannot allocate
device memory: a plugin whose host framework owns the whole device pool and
hands it only inputs and outputs, or a loop that cannot take cudaMalloc's
implicit device synchronisation.  Called through the C ABI, it runs the same
kernels on the same inputs as loong_attn_bwd, so dK and dV must be equal bit
for bit and dQ within one bf16 spacing (its fp32 reductions have no fixed
order).  The checks cover two calls in a row (the second finds the first
call's contents in the shared scratch array), a larger problem followed by a
smaller one (nothing of the larger one may leak into the smaller one's
results), the exchange mode whose receive buffers also live in the array, and
that a call allocates no device memory.  Collected last so that a failure here
cannot hide others."""
import ctypes

import pytest
import torch

from head_context_attention_gb300 import inputs, ops
from tests.test_gpu_layout import _within_one_bf16_spacing

pytestmark = pytest.mark.gpu


def _call(desc, t, o, r, lse, out=None):
    dq, dk, dv = out if out is not None else (torch.empty_like(t["q"]), torch.empty_like(t["k"]),
                                              torch.empty_like(t["v"]))
    p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())
    st = ops.lib().loong_attn_bwd_noalloc(ctypes.byref(desc), p(t["q"]), p(t["k"]), p(t["v"]), p(o), p(r), p(lse),
                                          p(t["do"]), p(dq), p(dk), p(dv),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ops.LOONG_OK, ops.lib().loong_status_string(st)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    return dq, dk, dv


def _problem(w, mode, layout):
    x = inputs.make_inputs(w, device="cuda")
    if layout == ops.LAYOUT_RANK_MAJOR:
        x = {n: ops.headctx_pack(x[n], w.cp, w.hp, 1) for n in ("q", "k", "v", "do")}
    o, lse, r = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode, layout=layout)
    want = ops.attn_bwd(w, x["q"], x["k"], x["v"], o, lse, x["do"], o_res=r, mode=mode, layout=layout)
    return x, o, r, lse, want


def _assert_same(got, want):
    assert torch.equal(got[1], want[1]), "dK"
    assert torch.equal(got[2], want[2]), "dV"
    assert _within_one_bf16_spacing(got[0], want[0]), "dQ"


SMALL = inputs.Workload("noalloc", 1024, 4, 2, 128, 2, 4, 2, 2, True)
LARGE = inputs.Workload("noalloc-large", 4096, 8, 1, 128, 1, 4, 2, 2, True)


@pytest.mark.parametrize("mode,layout", [(ops.MODE_FUSED, ops.LAYOUT_NATURAL),
                                         (ops.MODE_STEPWISE, ops.LAYOUT_NATURAL),
                                         (ops.MODE_STEPWISE_COPY, ops.LAYOUT_RANK_MAJOR)])
def test_noalloc_backward_equals_workspace_backward_twice(cuda_device, mode, layout):
    desc = ops.make_desc(SMALL, mode, layout=layout)
    assert ops.loong_attn_workspace_size(desc, 1) <= ops.NOALLOC_SCRATCH_BYTES
    x, o, r, lse, want = _problem(SMALL, mode, layout)
    for _ in range(2):
        _assert_same(_call(desc, x, o, r, lse), want)


def test_noalloc_larger_then_smaller_problem_leaks_nothing(cuda_device):
    """The header's example size (S = 4096, Hq = 8, Hkv = 1, d = 128) fills
    most of the array; the smaller problem after it still equals its own
    workspace backward."""
    big = ops.make_desc(LARGE)
    assert 20 << 20 < ops.loong_attn_workspace_size(big, 1) <= ops.NOALLOC_SCRATCH_BYTES
    xb, ob, rb, lb, wb = _problem(LARGE, ops.MODE_FUSED, ops.LAYOUT_NATURAL)
    xs, os_, rs, ls, ws = _problem(SMALL, ops.MODE_FUSED, ops.LAYOUT_NATURAL)
    _assert_same(_call(big, xb, ob, rb, lb), wb)
    _assert_same(_call(ops.make_desc(SMALL), xs, os_, rs, ls), ws)


def test_noalloc_call_allocates_no_device_memory(cuda_device):
    desc = ops.make_desc(SMALL)
    x, o, r, lse, want = _problem(SMALL, ops.MODE_FUSED, ops.LAYOUT_NATURAL)
    out = (torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]))
    _call(desc, x, o, r, lse, out)       # the first call looks up the array's address
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    got = _call(desc, x, o, r, lse, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    _assert_same(got, want)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    w = inputs.WORKLOADS["llama3-8b-s128k"]
    desc = ops.make_desc(w)
    assert ops.loong_attn_workspace_size(desc, 1) > ops.NOALLOC_SCRATCH_BYTES
    st = ops.lib().loong_attn_bwd_noalloc(ctypes.byref(desc), *([ctypes.c_void_p(16)] * 5), ctypes.c_void_p(16),
                                          ctypes.c_void_p(16), *([ctypes.c_void_p(16)] * 3), None)
    assert st == ops.LOONG_ERR_WORKSPACE
