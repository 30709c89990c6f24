"""Log-sum-exp merge of partial attention results.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages never state the merge (the guide's ring step returns a normalised
partial output with no log-sum-exp).  Reading taken: partial p over key set
K_p carries O_p = softmax-weighted mean of V over K_p and L_p = ln sum_{K_p}
exp(s).  For disjoint key sets, softmax over their union is
    L = ln sum_p exp(L_p),     O = sum_p exp(L_p - L) O_p,
which is evaluated with the largest L_p factored out.  A partial with an
empty key set has L_p = -inf and weight 0 (the identity of the merge); when
every part is empty the result is L = -inf, O = 0.
"""
import numpy as np


def lse_merge(o_parts, lse_parts):
    """Merge n partials: o_parts [n, rows, d], lse_parts [n, rows]."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.exp(lse_parts - m_safe[None, :])          # exp(-inf) = 0
    tot = w.sum(axis=0)
    lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, tot)))
    coef = np.where(empty[None, :], 0.0, w / np.where(empty, 1.0, tot)[None, :])
    o = np.einsum("nr,nrd->rd", coef, o_parts)
    return o, lse


def lse_merge2(o_a, lse_a, o_b, lse_b):
    """Two-way merge, the accumulate step of a ring pass."""
    return lse_merge(np.stack([o_a, o_b]), np.stack([lse_a, lse_b]))
