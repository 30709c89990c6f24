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
    o, lse = ops.attn_fwd(w, x["q"], x["k"], x["v"])
    assert ops.loong_get_device_status() == ops.LOONG_OK
    want_o, want_lse = attention.attention_forward(to64(x["q"][0]), to64(x["k"][0]), to64(x["v"][0]))
    assert_close("O", to64(o[0]), want_o, 2e-2, 2e-2)
