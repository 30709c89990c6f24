"""Seeded synthetic inputs for the ring-attention workloads.

This module holds only input generation: shapes, seeds and value
distributions.  It contains none of the attention arithmetic, imports nothing
else from this package, and serves both the CUDA path and its checks.

Recipe: every tensor is drawn as float32 N(0, 1) from its own seeded
``torch.Generator`` on the requested device and rounded to bf16; Q, K, V and
dO use seeds 1, 2, 3 and 4.  The peaky variant multiplies the K rows of
round(0.01 * S) token positions, drawn without replacement with seed 5, by 8
after the bf16 rounding (a power of two, so the scaling is exact).
Layout is [B, S, H, d], contiguous, natural token order.
"""
from dataclasses import dataclass, field, replace

import torch

SEED_Q, SEED_K, SEED_V, SEED_DO, SEED_PEAKY = 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Workload:
    name: str
    seqlen: int
    hq: int
    hkv: int
    head_dim: int
    hp: int
    cp: int
    ring_inner: int
    ring_outer: int
    backward: bool
    repack: bool = False
    peaky_keys: float = 0.0
    batch: int = 1
    placement: int = 1          # 1 paired blocks (zigzag), 0 contiguous
    causal: bool = True
    note: str = field(default="", compare=False)

    def with_(self, **kw):
        return replace(self, **kw)

    @property
    def fwd_flops(self):
        """Forward FLOPs: 2 GEMMs x 2 flops over the S^2/2 causal half (all S^2
        pairs when not causal)."""
        return (2 if self.causal else 4) * self.batch * self.seqlen * self.seqlen * self.hq * self.head_dim

    @property
    def flops(self):
        """fwd (+ bwd at 2.5x the forward, recompute of Q K^T included)."""
        f = self.fwd_flops
        return f * 3.5 if self.backward else f


WORKLOADS = {
    "tiny-gqa-s1k": Workload("tiny-gqa-s1k", 1024, 4, 2, 64, 2, 4, 4, 1, True,
                             note="tiny causal GQA, single ring"),
    "llama3-8b-s32k-fwd": Workload("llama3-8b-s32k-fwd", 32768, 32, 8, 128, 4, 8, 4, 2,
                                   False, note="Llama-3-8B attention layer, forward"),
    "llama3-8b-s128k": Workload("llama3-8b-s128k", 131072, 32, 8, 128, 8, 16, 8, 2, True,
                                note="Llama-3-8B attention layer, fwd+bwd"),
    "gqa-d64-s128k": Workload("gqa-d64-s128k", 131072, 32, 8, 64, 8, 16, 8, 2, True,
                              note="the same mesh and heads with head dimension 64, fwd+bwd"),
    "llama3-70b-s256k": Workload("llama3-70b-s256k", 262144, 64, 8, 128, 8, 32, 8, 4, True,
                                 repack=True,
                                 note="Llama-3-70B attention layer, fwd+bwd + Q/K/V repack"),
    "headgroup-s1m-peaky": Workload("headgroup-s1m-peaky", 1048576, 8, 1, 128, 1, 64, 8, 8,
                                    True, peaky_keys=0.01,
                                    note="one head group at 1M tokens, 1% keys x8"),
}


def _randn(shape, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def peaky_positions(seqlen, frac, device="cpu", seed=SEED_PEAKY):
    n = int(round(frac * seqlen))
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randperm(seqlen, generator=g, device=device)[:n]


def make_inputs(w, device="cpu", with_do=None, seed_offset=0):
    """Q, K, V (and dO) for workload ``w`` as bf16 [B, S, H, d] tensors."""
    if with_do is None:
        with_do = w.backward
    B, S, d = w.batch, w.seqlen, w.head_dim
    out = {
        "q": _randn((B, S, w.hq, d), SEED_Q + seed_offset, device),
        "k": _randn((B, S, w.hkv, d), SEED_K + seed_offset, device),
        "v": _randn((B, S, w.hkv, d), SEED_V + seed_offset, device),
    }
    if w.peaky_keys > 0:
        pos = peaky_positions(S, w.peaky_keys, device, SEED_PEAKY + seed_offset)
        out["k"][:, pos] *= 8
    if with_do:
        out["do"] = _randn((B, S, w.hq, d), SEED_DO + seed_offset, device)
    return out


def small(seqlen, hq, hkv, d, hp=1, cp=1, inner=None, outer=1, backward=True,
          placement=1, peaky=0.0, name=None):
    """An ad-hoc workload for parity cases (same recipe, other sizes)."""
    inner = cp if inner is None else inner
    return Workload(name or f"s{seqlen}-h{hq}x{hkv}-d{d}-hp{hp}-cp{cp}", seqlen, hq, hkv, d,
                    hp, cp, inner, outer, backward, placement=placement, peaky_keys=peaky)
