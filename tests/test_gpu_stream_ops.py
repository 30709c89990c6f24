"""Parity of the bandwidth-bound kernels: the LSE merge against the oracle's
merge (fp32 inputs, tolerance of fp32 rounding) and the head-context repack
bit-exactly against the oracle's index map."""
import numpy as np
import pytest
import torch

from head_context_attention_gb300 import ops
from oracle import merge, repack
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu


# Rows beyond a few thousand reach the two-rows-per-lane path of n <= 2 (rows
# past one grid stride); d = 256 gives lanes several vectors; n = 3, 4 are the
# other fixed-count paths, n >= 5 the general loop.
@pytest.mark.parametrize("rows,d,n,empty_frac", [(1, 4, 1, 0.0), (1000, 128, 2, 0.1),
                                                 (777, 64, 5, 0.3), (4096, 128, 16, 0.05),
                                                 (50001, 128, 2, 0.1), (40003, 64, 2, 0.5),
                                                 (30000, 256, 3, 0.2), (20011, 32, 4, 0.0),
                                                 (9001, 200, 1, 0.3)])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_lse_merge_matches_oracle(cuda_device, rows, d, n, empty_frac, out_bf16):
    g = torch.Generator(device="cuda").manual_seed(rows + n)
    o_parts = torch.randn((n, rows, d), generator=g, device="cuda")
    lse_parts = torch.randn((n, rows), generator=g, device="cuda") * 5
    drop = torch.rand((n, rows), generator=g, device="cuda") < empty_frac
    lse_parts[drop] = -torch.inf
    lse_parts[:, :3] = -torch.inf if rows > 5 else lse_parts[:, :3]   # rows with every part empty
    # an empty part is the merge's identity: whatever its O holds (NaN here)
    # must never reach the result; the oracle is given zeros there
    o_ref = to64(o_parts)
    o_ref[to64(torch.isneginf(lse_parts)).astype(bool)] = 0.0
    o_parts[torch.isneginf(lse_parts)] = float("nan")
    o_out = torch.empty((rows, d), dtype=torch.bfloat16 if out_bf16 else torch.float32, device="cuda")
    lse_out = torch.empty(rows, device="cuda")
    ops.loong_lse_merge(o_parts, lse_parts, o_out, lse_out)
    want_o, want_l = merge.lse_merge(o_ref, to64(lse_parts))
    tol = 1e-2 if out_bf16 else 1e-5
    assert_close("O", to64(o_out), want_o, tol, tol)
    gl, wl = to64(lse_out), want_l
    assert np.array_equal(np.isneginf(gl), np.isneginf(wl))
    fin = np.isfinite(wl)
    assert_close("LSE", gl[fin], wl[fin], 1e-5, 1e-6)


@pytest.mark.parametrize("B,S,H,d,cp,P,gather", [
    (1, 1024, 4, 128, 4, 2, 1), (1, 1024, 8, 64, 2, 4, 1), (2, 768, 6, 128, 3, 2, 1),
    (1, 512, 8, 128, 4, 8, 2), (1, 256, 2, 8, 2, 2, 1), (1, 4096, 64, 128, 8, 8, 1),
    (1, 512, 256, 128, 2, 4, 1), (3, 384, 12, 64, 2, 3, 2)])
def test_headctx_pack_bit_exact(cuda_device, B, S, H, d, cp, P, gather):
    g = torch.Generator(device="cuda").manual_seed(S + H)
    x = torch.randn((B, S, H, d), generator=g, device="cuda").to(torch.bfloat16)
    y = ops.headctx_pack(x, cp, P, gather)
    placement = 1 if gather == 1 else 0
    xv = x.view(torch.int16).cpu().numpy()
    want = np.concatenate([repack.headctx_pack(xv[b], cp, P, placement) for b in range(B)])
    assert np.array_equal(y.view(torch.int16).cpu().numpy(), want)
    back = ops.headctx_unpack(y, B, cp, P, gather)
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))


def test_headctx_pack_rank_major_input(cuda_device):
    n, P, sl, H, d = 3, 4, 5, 8, 64
    x = torch.arange(n * P * sl * H * d, device="cuda", dtype=torch.int32).to(torch.int16)
    x = x.view(n, P, sl, H, d)
    out = torch.empty((n, P, P * sl, H // P, d), dtype=torch.int16, device="cuda")
    ops.loong_headctx_pack(x, out, n, 1, P, sl, H, d, 0, 0)
    want = repack.ulysses_pack(x.cpu().numpy(), P)
    assert np.array_equal(out.cpu().numpy(), want)
    back = torch.empty_like(x)
    ops.loong_headctx_pack(out, back, n, 1, P, sl, H, d, 1, 0)
    assert torch.equal(back, x)


@pytest.mark.parametrize("B,S,heads,d,cp,P,gather", [
    (1, 1024, (8, 2, 2, 8), 128, 4, 2, 1), (1, 2048, (32, 8, 8), 128, 4, 4, 1), (2, 768, (6, 2), 64, 3, 2, 2),
    (1, 512, (4,), 128, 2, 2, 1), (3, 384, (12, 3, 3, 12), 64, 2, 3, 2), (1, 4096, (64, 8, 8, 64), 128, 8, 8, 1)])
def test_headctx_pack_n_equals_separate_packs(cuda_device, B, S, heads, d, cp, P, gather):
    """One launch over up to four tensors with their own head counts gives what
    separate loong_headctx_pack calls give, bit for bit, in both directions; the
    first tensor is also checked against the oracle's repack."""
    g = torch.Generator(device="cuda").manual_seed(S + sum(heads))
    xs = [torch.randn((B, S, h, d), generator=g, device="cuda").to(torch.bfloat16) for h in heads]
    s_local = S // (cp * P)
    ys = [torch.full((B * cp, P, S // cp, h // P, d), 3.0, dtype=torch.bfloat16, device="cuda") for h in heads]
    ops.loong_headctx_pack_n(xs, ys, B, cp, P, s_local, heads, d, 0, gather)
    for x, y in zip(xs, ys):
        assert torch.equal(y.view(torch.int16), ops.headctx_pack(x, cp, P, gather).view(torch.int16))
    placement = 1 if gather == 1 else 0
    xv = xs[0].view(torch.int16).cpu().numpy()
    want = np.concatenate([repack.headctx_pack(xv[b], cp, P, placement) for b in range(B)])
    assert np.array_equal(ys[0].view(torch.int16).cpu().numpy(), want)
    backs = [torch.full_like(x, 5.0) for x in xs]
    ops.loong_headctx_pack_n(ys, backs, B, cp, P, s_local, heads, d, 1, gather)
    for x, back in zip(xs, backs):
        assert torch.equal(back.view(torch.int16), x.view(torch.int16))
    assert ops.loong_get_device_status() == ops.LOONG_OK
