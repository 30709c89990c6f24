"""ctypes binding of libloong_attn.so: argument marshalling only.

Every function named ``loong_*`` calls the C entry point of the same name in
``include/loong_attn.h``; tensors are passed as raw device pointers and every
step of the computation runs in the library's kernels.  The library is loaded
on first use; a missing library raises ``RuntimeError`` (there is no other
implementation to fall back to).
"""
import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libloong_attn.so")
# the same library with device address checks (LOONG_CHECKED)
CHECKED_LIB_PATH = os.path.join(_PKG, "libloong_attn_checked.so")

LOONG_OK = 0
LOONG_ERR_INVALID_ARG = -1
LOONG_ERR_WORKSPACE = -2
LOONG_ERR_UNSUPPORTED = -3
LOONG_ERR_CUDA = -4
LOONG_ERR_DEVICE_TIMEOUT = -5
LOONG_ERR_DEVICE_CHECK = -6
PLACEMENT_CONTIGUOUS, PLACEMENT_ZIGZAG = 0, 1
MODE_STEPWISE, MODE_FUSED, MODE_STEPWISE_COPY, MODE_STEPWISE_COPY_AB = 0, 1, 2, 3
LAYOUT_NATURAL, LAYOUT_RANK_MAJOR = 0, 1

EXPORTS = ("loong_version", "loong_status_string", "loong_last_cuda_error", "loong_attn_check",
           "loong_attn_workspace_size", "loong_ring_schedule", "loong_attn_fwd", "loong_attn_fwd_ranks",
           "loong_attn_bwd",
           "loong_attn_bwd_noalloc", "loong_lse_merge", "loong_headctx_pack", "loong_headctx_pack_n",
           "loong_attn_2d_host_workspace_size", "loong_attn_2d_host", "loong_host_alloc", "loong_host_free",
           "loong_set_timing_events", "loong_get_device_status", "loong_selftest_wait_timeout")
NOALLOC_SCRATCH_BYTES = 32 << 20   # LOONG_NOALLOC_SCRATCH_BYTES


class LoongAttnDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("hp", ctypes.c_int32), ("cp", ctypes.c_int32),
                ("ring_inner", ctypes.c_int32), ("ring_outer", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("placement", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("layout", ctypes.c_int32)]


class LoongError(RuntimeError):
    def __init__(self, fn, status, lib):
        msg = lib.loong_status_string(status).decode()
        if status == LOONG_ERR_CUDA:
            msg += " (" + lib.loong_last_cuda_error().decode() + ")"
        super().__init__(f"{fn} failed: {status} {msg}")
        self.status = status


_lib = None


def lib():
    """Load the library once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m head_context_attention_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(LoongAttnDesc)
        L.loong_version.restype = ctypes.c_int
        L.loong_status_string.restype = ctypes.c_char_p
        L.loong_status_string.argtypes = [ctypes.c_int]
        L.loong_last_cuda_error.restype = ctypes.c_char_p
        L.loong_attn_check.argtypes = [D]
        L.loong_attn_workspace_size.restype = SZ
        L.loong_attn_workspace_size.argtypes = [D, ctypes.c_int]
        L.loong_ring_schedule.argtypes = [I32, I32, ctypes.POINTER(ctypes.c_int32)]
        L.loong_attn_fwd.argtypes = [D, P, P, P, P, P, P, P, SZ, P]
        L.loong_attn_fwd_ranks.argtypes = [D, I32, I32, P, P, P, P, P, P, SZ, P]
        L.loong_attn_bwd.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
        L.loong_attn_bwd_noalloc.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P]
        L.loong_lse_merge.argtypes = [I64, I32, I32, P, P, P, P, ctypes.c_int, P]
        L.loong_headctx_pack.argtypes = [I64, I32, I32, I64, I32, I32, ctypes.c_int, ctypes.c_int,
                                         P, P, P]
        L.loong_headctx_pack_n.argtypes = [I32, I64, I32, I32, I64, ctypes.POINTER(ctypes.c_int32), I32,
                                           ctypes.c_int, ctypes.c_int, ctypes.POINTER(P), ctypes.POINTER(P), P]
        L.loong_attn_2d_host_workspace_size.restype = SZ
        L.loong_attn_2d_host_workspace_size.argtypes = [D, ctypes.c_int]
        L.loong_attn_2d_host.argtypes = [D, I32, P, P, P, P, P, P, P, P, P, P, SZ, P, P]
        L.loong_host_alloc.argtypes = [SZ, ctypes.POINTER(ctypes.c_void_p)]
        L.loong_host_free.argtypes = [P]
        L.loong_set_timing_events.argtypes = [P, P]
        L.loong_get_device_status.argtypes = [P]
        L.loong_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
        _lib = L
    return _lib


def _check(fn, status):
    if status != LOONG_OK:
        raise LoongError(fn, status, lib())
    return status


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(w, mode=MODE_FUSED, scale=0.0, layout=LAYOUT_NATURAL):
    """Descriptor for a ``inputs.Workload`` (or anything with the same fields)."""
    return LoongAttnDesc(w.batch, w.seqlen, w.hq, w.hkv, w.head_dim, w.hp, w.cp, w.ring_inner,
                         w.ring_outer, 1 if getattr(w, "causal", True) else 0, w.placement, mode, scale, layout)


# ------------------------------------------------------------------ C entry points
def loong_attn_check(desc):
    return lib().loong_attn_check(ctypes.byref(desc))


def loong_attn_workspace_size(desc, pass_):
    return lib().loong_attn_workspace_size(ctypes.byref(desc), pass_)


def loong_ring_schedule(inner, outer):
    cp = inner * outer
    buf = (ctypes.c_int32 * (cp * cp))()
    _check("loong_ring_schedule", lib().loong_ring_schedule(inner, outer, buf))
    return [[buf[t * cp + c] for c in range(cp)] for t in range(cp)]


def _nbytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def loong_attn_fwd(desc, q, k, v, o, lse, o_res, ws, stream=None):
    return _check("loong_attn_fwd", lib().loong_attn_fwd(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(o_res), _ptr(ws),
        _nbytes(ws), _stream(stream)))


def loong_attn_fwd_ranks(desc, rank_begin, rank_end, q, k, v, o, lse, ws, stream=None):
    return _check("loong_attn_fwd_ranks", lib().loong_attn_fwd_ranks(
        ctypes.byref(desc), rank_begin, rank_end, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
        _ptr(ws), _nbytes(ws), _stream(stream)))


def loong_attn_bwd(desc, q, k, v, o, o_res, lse, dout, dq, dk, dv, ws, stream=None):
    return _check("loong_attn_bwd", lib().loong_attn_bwd(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(dout),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), _nbytes(ws), _stream(stream)))


def loong_attn_bwd_noalloc(desc, q, k, v, o, o_res, lse, dout, dq, dk, dv, stream=None):
    return _check("loong_attn_bwd_noalloc", lib().loong_attn_bwd_noalloc(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(dout),
        _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))


def loong_lse_merge(o_parts, lse_parts, o_out, lse_out, stream=None):
    n, rows, d = o_parts.shape
    out_bf16 = 1 if o_out.dtype == torch.bfloat16 else 0
    return _check("loong_lse_merge", lib().loong_lse_merge(
        rows, d, n, _ptr(o_parts), _ptr(lse_parts), _ptr(o_out), _ptr(lse_out), out_bf16,
        _stream(stream)))


def loong_headctx_pack(x, out, batch, cp, P, s_local, heads, d, direction, gather, stream=None):
    return _check("loong_headctx_pack", lib().loong_headctx_pack(
        batch, cp, P, s_local, heads, d, direction, gather, _ptr(x), _ptr(out), _stream(stream)))


def loong_headctx_pack_n(xs, outs, batch, cp, P, s_local, heads, d, direction, gather, stream=None):
    """loong_headctx_pack over the tensors xs -> outs (up to 4), heads[t] heads each, one launch."""
    n = len(xs)
    hs = (ctypes.c_int32 * n)(*heads)
    ins = (ctypes.c_void_p * n)(*[t.data_ptr() for t in xs])
    ous = (ctypes.c_void_p * n)(*[t.data_ptr() for t in outs])
    return _check("loong_headctx_pack_n", lib().loong_headctx_pack_n(
        n, batch, cp, P, s_local, hs, d, direction, gather, ins, ous, _stream(stream)))


def loong_attn_2d_host_workspace_size(desc, pass_):
    return lib().loong_attn_2d_host_workspace_size(ctypes.byref(desc), pass_)


def loong_attn_2d_host(desc, slot, q, k, v, dout, o, lse, dq, dk, dv, ws, stream=None, done_event=None):
    """One 2D-attention pass from host tensors to host tensors (pinned for
    overlap); dout=None runs the forward alone.  done_event: a recorded
    torch.cuda.Event marking the host outputs ready, or None."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    ev = None if done_event is None else ctypes.c_void_p(done_event.cuda_event)
    return _check("loong_attn_2d_host", lib().loong_attn_2d_host(
        ctypes.byref(desc), slot, _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(lse), _ptr(dq),
        _ptr(dk), _ptr(dv), _ptr(ws), nbytes, _stream(stream), ev))


def loong_host_alloc(nbytes):
    """Pinned, huge-page-backed host memory of ``nbytes`` bytes (an address,
    or None for 0 bytes); release it with loong_host_free."""
    p = ctypes.c_void_p()
    _check("loong_host_alloc", lib().loong_host_alloc(nbytes, ctypes.byref(p)))
    return p.value


def loong_host_free(ptr):
    return _check("loong_host_free", lib().loong_host_free(ptr))


_HOST_BUFFERS = {}


def host_empty(shape, dtype):
    """A CPU tensor over loong_host_alloc memory (pinned, huge pages where the
    kernel offers them), for the host arguments of loong_attn_2d_host.  It
    stays allocated until host_release(t) or the end of the process."""
    n = 1
    for e in shape:
        n *= int(e)
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    if nbytes == 0:
        return torch.empty(shape, dtype=dtype)
    ptr = loong_host_alloc(nbytes)
    raw = (ctypes.c_uint8 * nbytes).from_address(ptr)
    t = torch.frombuffer(raw, dtype=torch.uint8).view(dtype).view(shape)
    _HOST_BUFFERS[t.data_ptr()] = (ptr, raw)
    return t


def host_release(t):
    """Free the memory of a host_empty tensor; the tensor must not be used afterwards."""
    ptr, _ = _HOST_BUFFERS.pop(t.data_ptr())
    loong_host_free(ptr)


def loong_set_timing_events(start=None, stop=None):
    """Record torch.cuda.Event ``start``/``stop`` around the main attention
    kernels of this thread's next fwd/bwd calls (None, None to stop).  torch
    creates an event on its first record(), so record both once before
    passing them."""
    sp = None if start is None else ctypes.c_void_p(start.cuda_event)
    ep = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    return _check("loong_set_timing_events", lib().loong_set_timing_events(sp, ep))


def loong_get_device_status(stream=None):
    return lib().loong_get_device_status(_stream(stream))


def loong_selftest_wait_timeout(limit_us, stream=None):
    return lib().loong_selftest_wait_timeout(limit_us, _stream(stream))


# ------------------------------------------------------------------ conveniences
def workspace(desc, pass_, device="cuda"):
    n = loong_attn_workspace_size(desc, pass_)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device)


def attn_fwd(w, q, k, v, mode=MODE_FUSED, stream=None, layout=LAYOUT_NATURAL, res=True):
    """Allocate O, LSE (and O's rounding residual) with torch, run
    loong_attn_fwd, return (o, lse, o_res); o_res is None when ``res`` is
    false.  With LAYOUT_RANK_MAJOR, q/k/v (and o) are headctx_pack outputs."""
    desc = make_desc(w, mode, layout=layout)
    _check("loong_attn_check", loong_attn_check(desc))
    o = torch.empty_like(q)
    o_res = torch.empty_like(q) if res else None
    lse = torch.empty((w.batch, w.hq, w.seqlen), dtype=torch.float32, device=q.device)
    loong_attn_fwd(desc, q, k, v, o, lse, o_res, workspace(desc, 0, q.device), stream)
    return o, lse, o_res


def attn_bwd(w, q, k, v, o, lse, do, o_res=None, mode=MODE_FUSED, stream=None, layout=LAYOUT_NATURAL):
    """Allocate dQ/dK/dV with torch, run loong_attn_bwd, return them (in the
    layout of q, k).  ``o_res``: the forward's residual of O (D from O + o_res),
    or None (D from O alone)."""
    desc = make_desc(w, mode, layout=layout)
    _check("loong_attn_check", loong_attn_check(desc))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    loong_attn_bwd(desc, q, k, v, o, o_res, lse, do, dq, dk, dv, workspace(desc, 1, q.device), stream)
    return dq, dk, dv


def headctx_pack(x_nat, cp, P, gather=1, stream=None):
    """Natural [B, S, H, d] -> rank-major [B*cp, P, S/cp, H/P, d]."""
    B, S, H, d = x_nat.shape
    s_local = S // (cp * P)
    out = torch.empty((B * cp, P, S // cp, H // P, d), dtype=x_nat.dtype, device=x_nat.device)
    loong_headctx_pack(x_nat, out, B, cp, P, s_local, H, d, 0, gather, stream)
    return out


def headctx_unpack(y, batch, cp, P, gather=1, stream=None):
    """Rank-major [B*cp, P, S/cp, H/P, d] -> natural [B, S, H, d]."""
    n, P_, sgrp, hp, d = y.shape
    S = cp * sgrp
    out = torch.empty((batch, S, hp * P, d), dtype=y.dtype, device=y.device)
    loong_headctx_pack(y, out, batch, cp, P, sgrp // P, hp * P, d, 1, gather, stream)
    return out


def default_scale(d):
    return 1.0 / math.sqrt(d)
