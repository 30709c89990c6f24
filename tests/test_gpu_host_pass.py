"""loong_attn_2d_host: one whole 2D-attention pass from host memory to host
memory, its copies on the library's copy streams.

Its results must be those of the device entry points on the same inputs:
O, LSE, dK, dV bit for bit (deterministic kernels) and dQ within one bf16
spacing (fp32 reductions in an order that is not fixed).  The device path is
itself checked against the oracle elsewhere; one case here checks the host
pass against the oracle directly.  Consecutive calls with different inputs
and alternating slots check that no copy races the kernels of another call.
"""
import pytest
import torch

from head_context_attention_gb300 import inputs, ops
from oracle import attention
from tests.helpers import assert_close, to64
from tests.test_gpu_layout import _within_one_bf16_spacing

pytestmark = pytest.mark.gpu

GATHER = {1: 1, 0: 2}


def _device_pass(w, x, layout, mode=ops.MODE_FUSED):
    """The same pass through the device entry points: (o, lse, dq, dk, dv)."""
    if layout == ops.LAYOUT_NATURAL:
        o, lse, r = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=mode)
        if not w.backward:
            return o, lse
        return (o, lse) + ops.attn_bwd(w, x["q"], x["k"], x["v"], o, lse, x["do"], o_res=r, mode=mode)
    g = GATHER[w.placement]
    p = {n: ops.headctx_pack(t, w.cp, w.hp, g) for n, t in x.items()}
    o, lse, r = ops.attn_fwd(w, p["q"], p["k"], p["v"], mode=mode, layout=layout)
    un = lambda t: ops.headctx_unpack(t, w.batch, w.cp, w.hp, g)
    if not w.backward:
        return un(o), lse
    dq, dk, dv = ops.attn_bwd(w, p["q"], p["k"], p["v"], o, lse, p["do"], o_res=r, mode=mode, layout=layout)
    return un(o), lse, un(dq), un(dk), un(dv)


def _host_buffers(w, x, pinned=True):
    host_in = {n: (t.cpu().pin_memory() if pinned else t.cpu()) for n, t in x.items()}
    mk = lambda shape, dt: torch.full(shape, 7.0, dtype=dt, pin_memory=pinned)
    B, S, d = w.batch, w.seqlen, w.head_dim
    out = {"o": mk((B, S, w.hq, d), torch.bfloat16), "lse": mk((B, w.hq, S), torch.float32)}
    if w.backward:
        out |= {"dq": mk((B, S, w.hq, d), torch.bfloat16), "dk": mk((B, S, w.hkv, d), torch.bfloat16),
                "dv": mk((B, S, w.hkv, d), torch.bfloat16)}
    return host_in, out


def _host_pass(desc, w, slot, hin, hout, ws, done=None):
    g = (hout["dq"], hout["dk"], hout["dv"]) if w.backward else (None, None, None)
    ops.loong_attn_2d_host(desc, slot, hin["q"], hin["k"], hin["v"], hin.get("do"), hout["o"], hout["lse"], *g,
                           ws, done_event=done)


def _check_equal(w, hout, want):
    names = ("o", "lse", "dq", "dk", "dv")[:len(want)]
    for n, t in zip(names, want):
        got = hout[n]
        if n == "dq":
            assert _within_one_bf16_spacing(got.cuda(), t), n
        else:
            assert torch.equal(got, t.cpu()), n


CASES = [
    ("rank-major zigzag", inputs.small(2048, 8, 2, 128, hp=2, cp=4, inner=2, outer=2), ops.LAYOUT_RANK_MAJOR),
    ("rank-major contiguous d64", inputs.small(1536, 4, 2, 64, hp=2, cp=3, inner=3, placement=0),
     ops.LAYOUT_RANK_MAJOR),
    ("natural", inputs.small(2048, 8, 2, 128, hp=2, cp=4, inner=4), ops.LAYOUT_NATURAL),
    ("rank-major forward only", inputs.small(2048, 8, 2, 128, hp=2, cp=4, inner=2, outer=2, backward=False),
     ops.LAYOUT_RANK_MAJOR),
    ("natural forward only", inputs.small(1024, 4, 2, 64, hp=1, cp=2, backward=False), ops.LAYOUT_NATURAL),
]


@pytest.mark.parametrize("name,w,layout", CASES, ids=[c[0] for c in CASES])
def test_host_pass_equals_device_pass(cuda_device, name, w, layout):
    x = inputs.make_inputs(w, device="cuda")
    desc = ops.make_desc(w, layout=layout)
    ws = torch.empty(ops.loong_attn_2d_host_workspace_size(desc, 1 if w.backward else 0), dtype=torch.uint8,
                     device="cuda")
    hin, hout = _host_buffers(w, x)
    done = torch.cuda.Event()
    done.record()
    _host_pass(desc, w, 0, hin, hout, ws, done)
    done.synchronize()
    assert ops.loong_get_device_status() == ops.LOONG_OK
    _check_equal(w, hout, _device_pass(w, x, layout))


def test_host_pass_matches_oracle(cuda_device):
    w = inputs.small(1024, 4, 2, 64, hp=2, cp=2, inner=2)
    x = inputs.make_inputs(w, device="cuda")
    desc = ops.make_desc(w, layout=ops.LAYOUT_RANK_MAJOR)
    ws = torch.empty(ops.loong_attn_2d_host_workspace_size(desc, 1), dtype=torch.uint8, device="cuda")
    hin, hout = _host_buffers(w, x)
    _host_pass(desc, w, 1, hin, hout, ws)          # done_event NULL: the stream waits for the copies
    torch.cuda.synchronize()
    q, k, v, do = (to64(x[n][0]) for n in ("q", "k", "v", "do"))
    want_o, want_lse = attention.attention_forward(q, k, v)
    assert_close("O", to64(hout["o"][0]), want_o, 2e-2, 2e-2)
    assert_close("LSE", to64(hout["lse"][0]), want_lse, 1e-3, 0.0)
    g = attention.attention_backward(q, k, v, do)[:3]
    for n, exp in zip(("dq", "dk", "dv"), g):
        assert_close(n, to64(hout[n][0]), exp, 5e-2, 5e-2)


@pytest.mark.parametrize("layout", [ops.LAYOUT_RANK_MAJOR, ops.LAYOUT_NATURAL])
def test_consecutive_calls_with_other_inputs_do_not_race(cuda_device, layout):
    """Four calls enqueued back to back, each with its own inputs and host
    outputs, slots alternating, no synchronisation between them: every call's
    results equal the device pass of its own inputs."""
    w = inputs.small(4096, 8, 2, 128, hp=2, cp=4, inner=2, outer=2)
    desc = ops.make_desc(w, layout=layout)
    ws = torch.empty(ops.loong_attn_2d_host_workspace_size(desc, 1), dtype=torch.uint8, device="cuda")
    xs = [inputs.make_inputs(w, device="cuda", seed_offset=100 * i) for i in range(4)]
    bufs = [_host_buffers(w, x) for x in xs]
    dones = [torch.cuda.Event() for _ in xs]
    for e in dones:
        e.record()
    torch.cuda.synchronize()
    for i, ((hin, hout), e) in enumerate(zip(bufs, dones)):
        _host_pass(desc, w, i % 2, hin, hout, ws, e)
    for e in dones:
        e.synchronize()
    assert ops.loong_get_device_status() == ops.LOONG_OK
    for x, (_, hout) in zip(xs, bufs):
        _check_equal(w, hout, _device_pass(w, x, layout))


def test_pageable_host_memory_works(cuda_device):
    w = inputs.small(1024, 4, 2, 64, hp=2, cp=2, inner=2)
    x = inputs.make_inputs(w, device="cuda")
    desc = ops.make_desc(w, layout=ops.LAYOUT_RANK_MAJOR)
    ws = torch.empty(ops.loong_attn_2d_host_workspace_size(desc, 1), dtype=torch.uint8, device="cuda")
    hin, hout = _host_buffers(w, x, pinned=False)
    _host_pass(desc, w, 0, hin, hout, ws)
    torch.cuda.synchronize()
    _check_equal(w, hout, _device_pass(w, x, ops.LAYOUT_RANK_MAJOR))


def test_library_host_buffers_work_and_are_pinned(cuda_device):
    """Inputs and outputs in loong_host_alloc memory (registered, on huge pages
    where the kernel offers them): torch sees it as pinned, the pass equals the
    device path, and every buffer is released again."""
    w = inputs.small(2048, 8, 2, 128, hp=2, cp=4, inner=2, outer=2)
    x = inputs.make_inputs(w, device="cuda")
    desc = ops.make_desc(w, layout=ops.LAYOUT_RANK_MAJOR)
    ws = torch.empty(ops.loong_attn_2d_host_workspace_size(desc, 1), dtype=torch.uint8, device="cuda")
    hin = {n: ops.host_empty(t.shape, t.dtype) for n, t in x.items()}
    for n, t in x.items():
        hin[n].copy_(t)
    _, ref_out = _host_buffers(w, x)
    hout = {n: ops.host_empty(t.shape, t.dtype) for n, t in ref_out.items()}
    assert all(t.is_pinned() for t in list(hin.values()) + list(hout.values()))
    _host_pass(desc, w, 0, hin, hout, ws)
    torch.cuda.synchronize()
    _check_equal(w, hout, _device_pass(w, x, ops.LAYOUT_RANK_MAJOR))
    for t in list(hin.values()) + list(hout.values()):
        ops.host_release(t)


def test_host_allocator_edge_cases(cuda_device):
    """Zero bytes gives no buffer; freeing NULL is a no-op; a pointer the
    allocator did not return is refused."""
    assert ops.loong_host_alloc(0) is None
    assert ops.lib().loong_host_free(None) == ops.LOONG_OK
    foreign = torch.empty(16, dtype=torch.uint8, pin_memory=True)
    assert ops.lib().loong_host_free(foreign.data_ptr()) == ops.LOONG_ERR_INVALID_ARG
    p = ops.loong_host_alloc(1)
    assert p is not None
    assert ops.lib().loong_host_free(p) == ops.LOONG_OK
    assert ops.lib().loong_host_free(p) == ops.LOONG_ERR_INVALID_ARG


def test_device_memory_in_host_arguments_is_refused(cuda_device):
    w = inputs.small(1024, 4, 2, 64, hp=2, cp=2, inner=2)
    x = inputs.make_inputs(w, device="cuda")
    desc = ops.make_desc(w, layout=ops.LAYOUT_RANK_MAJOR)
    ws = torch.empty(ops.loong_attn_2d_host_workspace_size(desc, 1), dtype=torch.uint8, device="cuda")
    hin, hout = _host_buffers(w, x)
    with pytest.raises(ops.LoongError) as e:
        ops.loong_attn_2d_host(desc, 0, x["q"], hin["k"], hin["v"], hin["do"], hout["o"], hout["lse"], hout["dq"],
                               hout["dk"], hout["dv"], ws)
    assert e.value.status == ops.LOONG_ERR_INVALID_ARG
    with pytest.raises(ops.LoongError) as e:   # the workspace must be device memory
        ops.loong_attn_2d_host(desc, 0, hin["q"], hin["k"], hin["v"], hin["do"], hout["o"], hout["lse"],
                               hout["dq"], hout["dk"], hout["dv"], ws.cpu().pin_memory())
    assert e.value.status in (ops.LOONG_ERR_INVALID_ARG, ops.LOONG_ERR_WORKSPACE)
    torch.cuda.synchronize()
    assert bool((hout["o"].float() == 7.0).all())   # nothing was enqueued
    assert ops.loong_get_device_status() == ops.LOONG_OK


MODE_CASES = [
    ("stepwise", inputs.small(2048, 8, 2, 128, hp=2, cp=4, inner=2, outer=2), ops.MODE_STEPWISE),
    ("stepwise-copy", inputs.small(2048, 8, 2, 128, hp=2, cp=4, inner=2, outer=2), ops.MODE_STEPWISE_COPY),
    ("non-causal batch 2", inputs.small(1024, 4, 2, 64, hp=2, cp=2, inner=2).with_(causal=False, batch=2),
     ops.MODE_FUSED),
]


@pytest.mark.parametrize("name,w,mode", MODE_CASES, ids=[c[0] for c in MODE_CASES])
def test_host_pass_other_modes_equal_device_pass(cuda_device, name, w, mode):
    """The host pass passes the descriptor's mode, causality and batch through to
    the ring kernels: its results equal the device entry points' in that mode."""
    x = inputs.make_inputs(w, device="cuda")
    desc = ops.make_desc(w, mode, layout=ops.LAYOUT_RANK_MAJOR)
    assert ops.loong_attn_check(desc) == ops.LOONG_OK
    ws = torch.empty(ops.loong_attn_2d_host_workspace_size(desc, 1), dtype=torch.uint8, device="cuda")
    hin, hout = _host_buffers(w, x)
    _host_pass(desc, w, 0, hin, hout, ws)
    torch.cuda.synchronize()
    assert ops.loong_get_device_status() == ops.LOONG_OK
    _check_equal(w, hout, _device_pass(w, x, ops.LAYOUT_RANK_MAJOR, mode))
