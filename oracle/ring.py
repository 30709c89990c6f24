"""Chunked oracle: the ring schedule walked block pair by block pair.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

This is a second float64 oracle, independent of ``attention``: it follows the
2D-Attention data flow literally.  Every emulated rank (ring rank c, head rank
h) owns the tokens of its paired blocks ([G] section 2) and the heads of its
head group ([G] "The Scalability Limits of DeepSpeed Ulysses"); at each ring
step it computes softmax attention of its queries against the K/V chunk it
holds at that step (``schedule.ring_source``), with the causal rule applied on
global token positions ([G] "The Communication Overhead and Causal Imbalance of
Ring Attention"), and folds the step's partial result into its running result
with the log-sum-exp merge (``merge.lse_merge2``).

Reading taken for the guide's ring step ([G] "Step 3", which masks only at
step 0 and computes full attention otherwise): that holds for step 0 of the
paired-block layout, but at later steps some block pairs lie wholly in the
future and must be skipped, so the mask is always taken from global token
positions.  The result equals plain attention for every step order; only
rounding depends on the order.
"""
import numpy as np

from . import merge, schedule


def _pair_partial(qc, kc, vc, qpos, kpos, scale):
    """Softmax attention of one query chunk over one key chunk.

    Returns (O_p [n, d], L_p [n]); rows that see no key get (0, -inf).
    """
    s = scale * (qc @ kc.T)
    s = np.where(kpos[None, :] > qpos[:, None], -np.inf, s)
    m = s.max(axis=1)
    seen = ~np.isneginf(m)
    m_safe = np.where(seen, m, 0.0)
    e = np.exp(s - m_safe[:, None])
    den = e.sum(axis=1)
    den_safe = np.where(seen, den, 1.0)
    o = (e / den_safe[:, None]) @ vc
    lse = np.where(seen, m_safe + np.log(den_safe), -np.inf)
    return o, lse


def ring_forward(q, k, v, hp, cp, inner, outer, placement=schedule.ZIGZAG,
                 scale=None, step_order=None):
    """Run every emulated rank's ring pass; returns (o [S,Hq,d], lse [Hq,S]).

    ``step_order`` optionally permutes the steps 0..cp-1 (each rank still sees
    every source once); it changes only rounding.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    if inner * outer != cp:
        raise ValueError("inner * outer must equal cp")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    steps = list(range(cp)) if step_order is None else list(step_order)
    o = np.zeros_like(q)
    lse = np.full((hq, S), -np.inf)
    for h in range(hp):
        qheads, _ = schedule.head_group(h, hq, hkv, hp)
        for c in range(cp):
            qpos = schedule.rank_tokens(S, cp, c, placement)
            for hh in qheads:
                acc_o = np.zeros((len(qpos), d))
                acc_l = np.full(len(qpos), -np.inf)
                for t in steps:
                    j = schedule.ring_source(c, t, inner, outer)
                    kpos = schedule.rank_tokens(S, cp, j, placement)
                    po, pl = _pair_partial(q[qpos, hh], k[kpos, hh // G],
                                           v[kpos, hh // G], qpos, kpos, scale)
                    acc_o, acc_l = merge.lse_merge2(acc_o, acc_l, po, pl)
                o[qpos, hh] = acc_o
                lse[hh, qpos] = acc_l
    return o, lse


def ring_backward(q, k, v, do, o, lse, hp, cp, inner, outer,
                  placement=schedule.ZIGZAG, scale=None):
    """Gradients accumulated pair by pair over the same schedule.

    Uses the final (o, lse) of the forward pass: P_ij = exp(s_ij - LSE_i),
    D_i = dO_i . O_i.  Each pair adds its share to dQ of the query rank and to
    dK, dV of the source rank (the traffic that travels back around the ring).
    """
    q, k, v, do, o, lse = (np.asarray(x, dtype=np.float64)
                           for x in (q, k, v, do, o, lse))
    S, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dvec = np.einsum("shd,shd->hs", do, o)
    for h in range(hp):
        qheads, _ = schedule.head_group(h, hq, hkv, hp)
        for c in range(cp):
            qpos = schedule.rank_tokens(S, cp, c, placement)
            for t in range(cp):
                j = schedule.ring_source(c, t, inner, outer)
                kpos = schedule.rank_tokens(S, cp, j, placement)
                for hh in qheads:
                    g = hh // G
                    s = scale * (q[qpos, hh] @ k[kpos, g].T)
                    s = np.where(kpos[None, :] > qpos[:, None], -np.inf, s)
                    p = np.exp(s - lse[hh, qpos][:, None])
                    dp = do[qpos, hh] @ v[kpos, g].T
                    ds = p * (dp - dvec[hh, qpos][:, None])
                    dq[qpos, hh] += scale * (ds @ k[kpos, g])
                    dk[kpos, g] += scale * (ds.T @ q[qpos, hh])
                    dv[kpos, g] += p.T @ do[qpos, hh]
    return dq, dk, dv
