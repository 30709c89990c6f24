"""Failure detection on the GPU without a fault: a bounded mbarrier wait that
nothing completes gives up after its limit, the device error word reports it
through loong_get_device_status, the word is cleared by reading it, and the
context keeps working (a forward pass afterwards still matches the oracle)."""
import time

import pytest

from head_context_attention_gb300 import inputs, ops
from oracle import attention
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives(cuda_device):
    assert ops.loong_get_device_status() == ops.LOONG_OK        # nothing pending
    t0 = time.perf_counter()
    assert ops.loong_selftest_wait_timeout(50_000) == ops.LOONG_OK   # 50 ms limit
    assert ops.loong_get_device_status() == ops.LOONG_ERR_DEVICE_TIMEOUT
    waited = time.perf_counter() - t0
    assert 0.04 < waited < 5.0, waited                          # the wait ran to its limit, then returned
    assert ops.loong_get_device_status() == ops.LOONG_OK        # reading cleared the word
    w = inputs.WORKLOADS["tiny-gqa-s1k"]
    x = inputs.make_inputs(w, device="cuda", with_do=False)
    o, lse, _ = ops.attn_fwd(w, x["q"], x["k"], x["v"])
    assert ops.loong_get_device_status() == ops.LOONG_OK
    want_o, want_lse = attention.attention_forward(to64(x["q"][0]), to64(x["k"][0]), to64(x["v"][0]))
    assert_close("O", to64(o[0]), want_o, 2e-2, 2e-2)


def test_host_memory_is_refused_before_any_work(cuda_device):
    """Every tensor pointer must be memory of the current device: pinned host
    memory (which the GPU could read over the chip-to-chip link) and pageable
    host memory are refused with LOONG_ERR_INVALID_ARG, and nothing is written."""
    import torch

    w = inputs.WORKLOADS["tiny-gqa-s1k"]
    x = inputs.make_inputs(w, device="cuda", with_do=True)
    desc = ops.make_desc(w)
    ws0, ws1 = ops.workspace(desc, 0), ops.workspace(desc, 1)
    o = torch.full_like(x["q"], 7.0)
    lse = torch.full((w.batch, w.hq, w.seqlen), 7.0, device="cuda")
    for host in (x["q"].cpu().pin_memory(), x["q"].cpu()):
        with pytest.raises(ops.LoongError) as e:
            ops.loong_attn_fwd(desc, host, x["k"], x["v"], o, lse, None, ws0)
        assert e.value.status == ops.LOONG_ERR_INVALID_ARG
        with pytest.raises(ops.LoongError) as e:
            ops.loong_attn_fwd(desc, x["q"], x["k"], x["v"], o, lse.cpu().pin_memory(), None, ws0)
        assert e.value.status == ops.LOONG_ERR_INVALID_ARG
        with pytest.raises(ops.LoongError) as e:   # the residual output too
            ops.loong_attn_fwd(desc, x["q"], x["k"], x["v"], o, lse, host, ws0)
        assert e.value.status == ops.LOONG_ERR_INVALID_ARG
        with pytest.raises(ops.LoongError) as e:
            ops.loong_attn_bwd(desc, x["q"], x["k"], x["v"], o, None, lse, x["do"], host, x["k"].clone(),
                               x["v"].clone(), ws1)
        assert e.value.status == ops.LOONG_ERR_INVALID_ARG
        with pytest.raises(ops.LoongError) as e:
            ops.loong_headctx_pack(host, torch.empty_like(x["q"]), w.batch, w.cp, w.hp, w.seqlen // (w.cp * w.hp),
                                   w.hq, w.head_dim, 0, 1)
        assert e.value.status == ops.LOONG_ERR_INVALID_ARG
    parts = torch.zeros((2, 64, 128), device="cuda")
    with pytest.raises(ops.LoongError) as e:
        ops.loong_lse_merge(parts, torch.zeros((2, 64), device="cuda"), torch.empty((64, 128)).pin_memory(),
                            torch.empty(64, device="cuda"))
    assert e.value.status == ops.LOONG_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())   # nothing was enqueued
    assert ops.loong_get_device_status() == ops.LOONG_OK
