"""Host-side checks of the C-ABI library: it loads without a GPU, exports every
declared symbol, validates descriptors, sizes workspaces and produces the ring
table the oracle defines.  No compute call is made."""
import ctypes
import os
import re

import numpy as np
import pytest

from head_context_attention_gb300 import inputs, ops
from oracle import schedule

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            with open(os.path.join(inc, f)) as fh:
                names |= set(re.findall(r"LOONG_API\s+[\w\s\*]+?\b(loong_\w+)\s*\(", fh.read()))
    return names


def test_library_exports_every_declared_symbol(loong_lib):
    names = _declared()
    assert len(names) >= 11
    assert names == set(ops.EXPORTS)
    for n in names:
        assert hasattr(loong_lib, n), n


def test_status_strings(loong_lib):
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert ops.lib().loong_status_string(st)
    assert ops.lib().loong_version() >= 1


@pytest.mark.parametrize("inner,outer", [(4, 1), (4, 2), (8, 2), (8, 4), (8, 8), (3, 5)])
def test_ring_schedule_matches_oracle(loong_lib, inner, outer):
    got = np.array(ops.loong_ring_schedule(inner, outer))
    np.testing.assert_array_equal(got, schedule.schedule_table(inner, outer))


def _desc(**kw):
    w = inputs.WORKLOADS["llama3-8b-s128k"]
    d = ops.make_desc(w)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("field,value,status", [
    ("hq", 30, ops.LOONG_ERR_INVALID_ARG),          # Hq % Hkv
    ("hp", 16, ops.LOONG_ERR_INVALID_ARG),          # Hkv % hp: a kv head would be split
    ("ring_inner", 4, ops.LOONG_ERR_INVALID_ARG),   # inner * outer != cp
    ("seqlen", 131072 + 32, ops.LOONG_ERR_INVALID_ARG),  # S % (2 cp)
    ("head_dim", 96, ops.LOONG_ERR_UNSUPPORTED),
    ("causal", 0, ops.LOONG_OK),
    ("causal", 2, ops.LOONG_ERR_INVALID_ARG),
    ("placement", 7, ops.LOONG_ERR_INVALID_ARG),
    ("mode", 5, ops.LOONG_ERR_INVALID_ARG),
    ("mode", ops.MODE_STEPWISE_COPY_AB, ops.LOONG_ERR_UNSUPPORTED),   # needs the rank-major layout
    ("batch", 0, ops.LOONG_ERR_INVALID_ARG),
    ("layout", 2, ops.LOONG_ERR_INVALID_ARG),
    ("mode", ops.MODE_STEPWISE_COPY, ops.LOONG_ERR_UNSUPPORTED),   # needs the rank-major layout
    ("layout", ops.LAYOUT_RANK_MAJOR, ops.LOONG_OK),
])
def test_descriptor_validation(loong_lib, field, value, status):
    assert ops.loong_attn_check(_desc()) == ops.LOONG_OK
    assert ops.loong_attn_check(_desc(**{field: value})) == status


def test_block_length_must_split_over_hp(loong_lib):
    # S = 2*cp*blk with blk = 12 and hp = 8: the Ulysses split of a block fails
    d = _desc(seqlen=2 * 16 * 12)
    assert ops.loong_attn_check(d) == ops.LOONG_ERR_INVALID_ARG
    d = _desc(seqlen=2 * 16 * 16)
    assert ops.loong_attn_check(d) == ops.LOONG_OK


def test_workspace_sizes(loong_lib):
    w = inputs.WORKLOADS["llama3-8b-s128k"]
    fused, step = ops.make_desc(w, ops.MODE_FUSED), ops.make_desc(w, ops.MODE_STEPWISE)
    q_el = w.seqlen * w.hq * w.head_dim
    kv_el = w.seqlen * w.hkv * w.head_dim
    up = lambda x: (x + 255) // 256 * 256
    # the forward's fp16 copy of V and the word for max |V|; STEPWISE adds the fp32 O accumulator
    assert ops.loong_attn_workspace_size(fused, 0) == up(kv_el * 2) + 256
    assert ops.loong_attn_workspace_size(step, 0) == up(kv_el * 2) + 256 + q_el * 4
    copy = ops.make_desc(w, ops.MODE_STEPWISE_COPY, layout=ops.LAYOUT_RANK_MAJOR)
    assert ops.loong_attn_workspace_size(copy, 0) == up(kv_el * 2) + 256 + q_el * 4 + 4 * up(kv_el * 2)
    blk = w.seqlen // (2 * w.cp)
    stats = 2 * w.hq * (2 * w.cp * ((blk + 3) // 4 * 4) + 128) * 4
    # the backward: fp32 dQ accumulator, row statistics, fp32 dK, dV accumulators
    assert ops.loong_attn_workspace_size(fused, 1) == up(q_el * 4) + up(stats) + 2 * up(kv_el * 4)
    assert ops.loong_attn_workspace_size(step, 1) == up(q_el * 4) + up(stats) + 2 * up(kv_el * 4)
    bad = _desc(hq=30)
    assert ops.loong_attn_workspace_size(bad, 0) == 0


def test_null_pointers_rejected_before_any_cuda_call(loong_lib):
    d = _desc()
    L = ops.lib()
    assert L.loong_attn_fwd(ctypes.byref(d), None, None, None, None, None, None, None, 0, None) == \
        ops.LOONG_ERR_INVALID_ARG
    assert L.loong_attn_bwd(ctypes.byref(d), *([None] * 11), 0, None) == ops.LOONG_ERR_INVALID_ARG
    assert L.loong_lse_merge(10, 3, 2, None, None, None, None, 0, None) == ops.LOONG_ERR_INVALID_ARG
    assert L.loong_lse_merge(0, 128, 2, None, None, None, None, 0, None) == ops.LOONG_OK
    assert L.loong_headctx_pack(1, 2, 3, 4, 8, 128, 0, 0, None, None, None) == \
        ops.LOONG_ERR_INVALID_ARG   # heads % P
    assert L.loong_headctx_pack(0, 2, 2, 4, 8, 128, 0, 0, None, None, None) == ops.LOONG_OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(ops, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(ops, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        ops.lib()


def test_rank_major_view_rows_must_fit_int32(loong_lib):
    # the rank-major view has B*S*hp rows; its TMA row coordinate is 32-bit
    d = _desc(batch=2048, layout=ops.LAYOUT_RANK_MAJOR)      # 2048 * 131072 * 8 rows
    assert ops.loong_attn_check(d) == ops.LOONG_ERR_UNSUPPORTED
    d = _desc(batch=2, layout=ops.LAYOUT_RANK_MAJOR)
    assert ops.loong_attn_check(d) == ops.LOONG_OK


def test_fwd_ranks_validation_before_any_cuda_call(loong_lib):
    L = ops.lib()
    d = _desc()
    args = (None,) * 5 + (None, 0, None)   # q, k, v, o, lse, ws, ws_bytes, stream
    for lo, hi in ((-1, 2), (3, 3), (4, 2), (0, d.cp + 1)):
        assert L.loong_attn_fwd_ranks(ctypes.byref(d), lo, hi, *args) == ops.LOONG_ERR_INVALID_ARG
    assert L.loong_attn_fwd_ranks(ctypes.byref(d), 0, 1, *args) == ops.LOONG_ERR_INVALID_ARG  # null tensors
    step = _desc(mode=ops.MODE_STEPWISE)
    assert L.loong_attn_fwd_ranks(ctypes.byref(step), 0, 1, *args) == ops.LOONG_ERR_UNSUPPORTED


def test_stepwise_copy_mode_needs_rank_major_and_receive_buffers(loong_lib):
    w = inputs.WORKLOADS["llama3-8b-s128k"]
    d = ops.make_desc(w, ops.MODE_STEPWISE_COPY, layout=ops.LAYOUT_RANK_MAJOR)
    assert ops.loong_attn_check(d) == ops.LOONG_OK
    step = ops.make_desc(w, ops.MODE_STEPWISE, layout=ops.LAYOUT_RANK_MAJOR)
    recv = 4 * ((w.seqlen * w.hkv * w.head_dim * 2 + 255) // 256 * 256)
    for p in (0, 1):
        assert ops.loong_attn_workspace_size(d, p) == ops.loong_attn_workspace_size(step, p) + recv


def test_selftest_wait_limit_validated_before_any_cuda_call(loong_lib):
    L = ops.lib()
    for bad in (0, 1000001):
        assert L.loong_selftest_wait_timeout(bad, None) == ops.LOONG_ERR_INVALID_ARG


def test_two_ring_copy_mode_needs_paired_blocks(loong_lib):
    w = inputs.WORKLOADS["llama3-8b-s128k"]
    d = ops.make_desc(w, ops.MODE_STEPWISE_COPY_AB, layout=ops.LAYOUT_RANK_MAJOR)
    assert ops.loong_attn_check(d) == ops.LOONG_OK
    one = ops.make_desc(w, ops.MODE_STEPWISE_COPY, layout=ops.LAYOUT_RANK_MAJOR)
    assert ops.loong_attn_workspace_size(d, 1) == ops.loong_attn_workspace_size(one, 1)
    d.placement = ops.PLACEMENT_CONTIGUOUS
    assert ops.loong_attn_check(d) == ops.LOONG_ERR_UNSUPPORTED
    d = ops.make_desc(w, 4, layout=ops.LAYOUT_RANK_MAJOR)
    assert ops.loong_attn_check(d) == ops.LOONG_ERR_INVALID_ARG


@pytest.mark.parametrize("layout", [ops.LAYOUT_NATURAL, ops.LAYOUT_RANK_MAJOR])
def test_2d_host_workspace_sizes(loong_lib, layout):
    """Two slots of natural inputs, the natural outputs and LSE, the forward's
    residual of O (fwd+bwd), the rank-major tensors (RANK_MAJOR only) and the
    ring workspaces, each 256-byte aligned."""
    w = inputs.WORKLOADS["llama3-8b-s128k"]
    d = ops.make_desc(w, ops.MODE_FUSED, layout=layout)
    up = lambda x: (x + 255) // 256 * 256
    qb = w.seqlen * w.hq * w.head_dim * 2
    kvb = w.seqlen * w.hkv * w.head_dim * 2
    lse = w.hq * w.seqlen * 4
    rm = layout == ops.LAYOUT_RANK_MAJOR
    fwd = 2 * (up(qb) + 2 * up(kvb)) + up(qb) + up(lse) + (up(qb) + 2 * up(kvb) + up(qb) if rm else 0)
    both = 2 * (2 * up(qb) + 2 * up(kvb)) + 2 * up(qb) + 2 * up(kvb) + up(lse) + \
        ((3 * up(qb) + 2 * up(kvb)) + (up(qb) + 2 * up(kvb)) if rm else 0) + up(qb) + \
        ops.loong_attn_workspace_size(d, 0) + ops.loong_attn_workspace_size(d, 1)
    assert ops.loong_attn_2d_host_workspace_size(d, 0) == fwd + ops.loong_attn_workspace_size(d, 0)
    assert ops.loong_attn_2d_host_workspace_size(d, 1) == both
    assert ops.loong_attn_2d_host_workspace_size(d, 2) == 0
    assert ops.loong_attn_2d_host_workspace_size(_desc(hq=30), 1) == 0


def test_2d_host_validation_before_any_cuda_call(loong_lib):
    d = ops.make_desc(inputs.WORKLOADS["tiny-gqa-s1k"], layout=ops.LAYOUT_RANK_MAJOR)
    L = ops.lib()
    need = ops.loong_attn_2d_host_workspace_size(d, 1)
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, ctypes.c_void_p)
    ws = ctypes.c_void_p(1 << 20)   # never dereferenced: every case below fails before any CUDA call
    call = lambda slot, dout, grads, ws_, n: L.loong_attn_2d_host(
        ctypes.byref(d), slot, p, p, p, dout, p, p, *(grads or (None, None, None)), ws_, n, None, None)
    assert call(2, p, (p, p, p), ws, need) == ops.LOONG_ERR_INVALID_ARG        # slot
    assert call(-1, p, (p, p, p), ws, need) == ops.LOONG_ERR_INVALID_ARG
    assert call(0, p, (p, None, p), ws, need) == ops.LOONG_ERR_INVALID_ARG     # a gradient missing
    assert call(0, None, (p, p, p), ws, need) == ops.LOONG_ERR_INVALID_ARG     # gradients without dO
    assert call(0, p, (p, p, p), ws, need - 256) == ops.LOONG_ERR_WORKSPACE
    assert call(0, p, (p, p, p), None, need) == ops.LOONG_ERR_WORKSPACE
    assert call(0, p, (p, p, p), ctypes.c_void_p((1 << 20) + 16), need) == ops.LOONG_ERR_WORKSPACE  # alignment
    assert L.loong_attn_2d_host(ctypes.byref(d), 0, None, p, p, p, p, p, p, p, p, ws, need, None, None) == \
        ops.LOONG_ERR_INVALID_ARG


def test_headctx_pack_n_validation_before_any_cuda_call(loong_lib):
    L = ops.lib()
    P_ = ctypes.c_void_p
    heads = (ctypes.c_int32 * 4)(8, 2, 2, 8)
    bad_heads = (ctypes.c_int32 * 2)(8, 3)
    ptrs = (P_ * 4)(16, 32, 48, 64)   # never dereferenced
    nul = (P_ * 4)(16, None, 48, 64)
    call = lambda n, h, i, o, d=128, direction=0, gather=1: L.loong_headctx_pack_n(
        n, 1, 4, 2, 128, h, d, direction, gather, i, o, None)
    for n in (0, 5, -1):
        assert call(n, heads, ptrs, ptrs) == ops.LOONG_ERR_INVALID_ARG
    assert call(2, bad_heads, ptrs, ptrs) == ops.LOONG_ERR_INVALID_ARG        # heads % P
    assert call(4, heads, nul, ptrs) == ops.LOONG_ERR_INVALID_ARG             # a null tensor
    assert call(4, None, ptrs, ptrs) == ops.LOONG_ERR_INVALID_ARG             # no head array
    assert call(4, heads, ptrs, ptrs, d=4) == ops.LOONG_ERR_INVALID_ARG       # d*2 not a multiple of 16
    assert call(4, heads, ptrs, ptrs, direction=2) == ops.LOONG_ERR_INVALID_ARG
    assert call(4, heads, ptrs, ptrs, gather=3) == ops.LOONG_ERR_INVALID_ARG
    mis = (P_ * 4)(16, 40, 48, 64)                                            # 8-byte aligned only
    assert call(4, heads, mis, ptrs) == ops.LOONG_ERR_INVALID_ARG
    assert L.loong_headctx_pack_n(4, 0, 4, 2, 128, heads, 128, 0, 1, ptrs, ptrs, None) == ops.LOONG_OK  # empty


def test_noalloc_scratch_example_fits(loong_lib):
    """The header's example for the allocation-free backward (S = 4096,
    Hq = 8, Hkv = 1, d = 128) fits its 32 MiB array in FUSED and STEPWISE
    mode, within the header's bound."""
    w = inputs.Workload("example", 4096, 8, 1, 128, 1, 4, 2, 2, True)
    for mode in (ops.MODE_FUSED, ops.MODE_STEPWISE):
        need = ops.loong_attn_workspace_size(ops.make_desc(w, mode), 1)
        assert need <= ops.NOALLOC_SCRATCH_BYTES
        nblocks = 2 * w.cp
        estimate = 4 * w.seqlen * w.hq * 128 + 8 * w.seqlen * w.hkv * 128 + 8 * w.hq * (w.seqlen + 3 * nblocks + 128)
        assert estimate - 8 * w.hq * 3 * nblocks <= need <= estimate + 4 * 256   # block padding, 256-byte rounding
        assert abs(need / 2 ** 20 - 20.3) < 0.05, need / 2 ** 20
