"""Ulysses head-context repack and the zigzag gather, as index maps.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[G] "The Scalability Limits of DeepSpeed Ulysses": before attention an
all-to-all turns each rank's (S/P tokens, all H heads) into (all S tokens of
the group, H/P heads); after attention the inverse turns (S, H/P) back into
(S/P, H).  On one device the all-to-all is this permutation:
    out[n][p][q * s_local + t][h'] = in[n][q][t][p * (H/P) + h']
for group n, destination rank p, source rank q, local token t and head h'.
With 2D attention the group is the head-parallel group of one ring rank, so
the token axis is that ring rank's chunk (two paired blocks, [G] section 2).
"""
import numpy as np

from . import schedule


def ulysses_pack(x, P):
    """(S/P, H) -> (S, H/P): x [n, P, s_local, H, d] -> [n, P, P*s_local, H/P, d]."""
    x = np.asarray(x)
    n, p_in, s_local, H, d = x.shape
    if p_in != P or H % P:
        raise ValueError("bad shape for the repack")
    hp = H // P
    out = np.empty((n, P, P * s_local, hp, d), dtype=x.dtype)
    for b in range(n):
        for p in range(P):
            for q in range(P):
                out[b, p, q * s_local:(q + 1) * s_local] = \
                    x[b, q, :, p * hp:(p + 1) * hp]
    return out


def ulysses_unpack(y, P):
    """(S, H/P) -> (S/P, H): the inverse of ``ulysses_pack``."""
    y = np.asarray(y)
    n, p_in, s_tot, hp, d = y.shape
    if p_in != P or s_tot % P:
        raise ValueError("bad shape for the repack")
    s_local = s_tot // P
    out = np.empty((n, P, s_local, hp * P, d), dtype=y.dtype)
    for b in range(n):
        for p in range(P):
            for q in range(P):
                out[b, q, :, p * hp:(p + 1) * hp] = \
                    y[b, p, q * s_local:(q + 1) * s_local]
    return out


def zigzag_gather(x, cp, placement=schedule.ZIGZAG):
    """Natural order [S, H, d] -> per ring rank [cp, S/cp, H, d]."""
    x = np.asarray(x)
    S = x.shape[0]
    return np.stack([x[schedule.rank_tokens(S, cp, c, placement)]
                     for c in range(cp)])


def zigzag_scatter(y, placement=schedule.ZIGZAG):
    """Per ring rank [cp, S/cp, H, d] -> natural order [S, H, d]."""
    y = np.asarray(y)
    cp, sl = y.shape[0], y.shape[1]
    S = cp * sl
    out = np.empty((S,) + y.shape[2:], dtype=y.dtype)
    for c in range(cp):
        out[schedule.rank_tokens(S, cp, c, placement)] = y[c]
    return out


def headctx_pack(x_nat, cp, P, placement=schedule.ZIGZAG):
    """Natural [S, H, d] -> rank-major [cp, P, S/cp, H/P, d] (gather + pack)."""
    g = zigzag_gather(x_nat, cp, placement)
    cp_, sl, H, d = g.shape
    return ulysses_pack(g.reshape(cp, P, sl // P, H, d), P)


def headctx_unpack(y, cp, P, placement=schedule.ZIGZAG):
    """Rank-major [cp, P, S/cp, H/P, d] -> natural [S, H, d]."""
    u = ulysses_unpack(y, P)
    cp_, P_, s_local, H, d = u.shape
    return zigzag_scatter(u.reshape(cp, P * s_local, H, d), placement)
