"""A seeded sweep over the descriptor's options on small problems: placement,
causal or not, FUSED / STEPWISE, head dimension, group size, head-parallel
degree, ring shape (inner x outer), batch and block lengths that leave ragged
tiles.  Every configuration is checked against the float64 oracle (O 2e-2,
LSE 1e-3, dQ/dK/dV 5e-2), and the rank-major layout against the natural one
(bit for bit, dQ up to its reduction order)."""
import numpy as np
import pytest
import torch

from head_context_attention_gb300 import inputs, ops
from oracle import attention
from tests.helpers import assert_close, to64
from tests.test_gpu_layout import _within_one_bf16_spacing

pytestmark = pytest.mark.gpu


def _configs(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([64, 128]))
        hkv = int(rng.choice([1, 2]))
        G = int(rng.choice([1, 2, 3, 4]))
        hq = hkv * G
        hp = int(rng.choice([p for p in (1, 2) if hkv % p == 0]))
        cp = int(rng.integers(1, 7))
        inner = int(rng.choice([i for i in range(1, cp + 1) if cp % i == 0]))
        placement = int(rng.integers(0, 2))
        nblocks = 2 * cp if placement == 1 else cp
        blk = int(rng.integers(8, 160)) * hp          # a multiple of hp; often not of 128
        S = nblocks * blk
        if S > 2048:
            continue
        out.append(dict(S=S, hq=hq, hkv=hkv, d=d, hp=hp, cp=cp, inner=inner, outer=cp // inner,
                        placement=placement, causal=bool(rng.integers(0, 2)), batch=int(rng.integers(1, 3)),
                        mode=int(rng.choice([ops.MODE_FUSED, ops.MODE_STEPWISE]))))
    return out


CONFIGS = _configs()


def _name(c):
    return (f"S{c['S']}-h{c['hq']}/{c['hkv']}-d{c['d']}-hp{c['hp']}-cp{c['cp']}({c['inner']}x{c['outer']})-"
            f"{'zz' if c['placement'] else 'ct'}-{'c' if c['causal'] else 'nc'}-b{c['batch']}-m{c['mode']}")


@pytest.mark.parametrize("c", CONFIGS, ids=[_name(c) for c in CONFIGS])
def test_sweep_matches_oracle_and_layouts_agree(cuda_device, c):
    w = inputs.Workload(_name(c), c["S"], c["hq"], c["hkv"], c["d"], c["hp"], c["cp"], c["inner"], c["outer"],
                        True, placement=c["placement"], batch=c["batch"], causal=c["causal"])
    assert ops.loong_attn_check(ops.make_desc(w, c["mode"])) == ops.LOONG_OK
    x = inputs.make_inputs(w, device="cuda")
    o, lse, o_res = ops.attn_fwd(w, x["q"], x["k"], x["v"], mode=c["mode"])
    dq, dk, dv = ops.attn_bwd(w, x["q"], x["k"], x["v"], o, lse, x["do"], o_res=o_res, mode=c["mode"])
    assert ops.loong_get_device_status() == ops.LOONG_OK
    for b in range(w.batch):
        q, k, v, do = (to64(x[n][b]) for n in ("q", "k", "v", "do"))
        want_o, want_lse = attention.attention_forward(q, k, v, causal=c["causal"])
        assert_close("O", to64(o[b]), want_o, 2e-2, 2e-2)
        assert_close("LSE", to64(lse[b]), want_lse, 1e-3, 0.0)
        g = attention.attention_backward(q, k, v, do, causal=c["causal"])[:3]
        for nm, got, exp in zip(("dQ", "dK", "dV"), (dq, dk, dv), g):
            assert_close(nm, to64(got[b]), exp, 5e-2, 5e-2)
    gather = 1 if c["placement"] == 1 else 2
    p = {n: ops.headctx_pack(x[n], w.cp, w.hp, gather) for n in ("q", "k", "v", "do")}
    rm = ops.LAYOUT_RANK_MAJOR
    o2, lse2, r2 = ops.attn_fwd(w, p["q"], p["k"], p["v"], mode=c["mode"], layout=rm)
    dq2, dk2, dv2 = ops.attn_bwd(w, p["q"], p["k"], p["v"], o2, lse2, p["do"], o_res=r2, mode=c["mode"], layout=rm)
    assert ops.loong_get_device_status() == ops.LOONG_OK
    un = lambda t: ops.headctx_unpack(t, w.batch, w.cp, w.hp, gather)
    assert torch.equal(lse2, lse)
    assert torch.equal(un(o2), o) and torch.equal(un(r2), o_res)
    assert torch.equal(un(dk2), dk) and torch.equal(un(dv2), dv)
    assert _within_one_bf16_spacing(un(dq2), dq)
