"""Plain float64 causal grouped-query attention, forward and backward.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Definition followed ([G] "The Communication Overhead and Causal Imbalance of
Ring Attention": query i sees key j only when j <= i; [G] "Step 3: Pipelined
Ring Attention Communication Kernel", ``forward_local_attention``: scores are
q.k^T times 1/sqrt(head_dim), softmax over keys, then the probability-weighted
sum of V rows; [G] "Best Practices", item 2, and "The Scalability Limits of
DeepSpeed Ulysses": Hq query heads share Hkv key/value heads).

Readings where the pages are silent:
  * GQA grouping is contiguous: query head i uses kv head i // (Hq // Hkv).
  * LSE is the natural log of the softmax denominator of the scaled logits,
    stored [Hq, S].
  * The backward pass is the exact gradient of the forward pass: with
    D_i = dO_i . O_i, dP = dO V^T, dS = P * (dP - D), dQ = scale dS K,
    dK = scale dS^T Q, dV = P^T dO, with dK and dV summed over the query heads
    that share a kv head.  Optionally (``d_from_bf16_o``) D is formed from O
    rounded to bf16: the reading for a backward that is given only the bf16
    output of the forward (with peaky logits this moves dQ by up to ~0.1 at
    keys scaled x8 and S = 1M).

Layouts: q [S, Hq, d], k and v [S, Hkv, d], o [S, Hq, d], lse [Hq, S].  The
batch dimension is handled by the caller (B = 1 in every workload).
"""
import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def round_bf16(x):
    """Round to the nearest bfloat16 value (ties to even), returned as float64.

    bfloat16 is the upper half of an IEEE-754 binary32: the value is first
    rounded to binary32 (numpy, ties to even), then its low 16 bits are
    removed with round-to-nearest-even on the bit pattern.  Inf and NaN pass
    through (no input here is either).
    """
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def _dvec(do, o, d_from_bf16_o):
    """D_i = dO_i . O_i; with ``d_from_bf16_o`` O is first rounded to bf16.

    Reading taken for the backward: D is formed from the output the forward
    returns, which is O rounded to bf16; ``d_from_bf16_o=False`` gives the
    exact gradient of the unrounded forward.
    """
    if d_from_bf16_o:
        o = round_bf16(o)
    return np.einsum("...d,...d->...", do, o)


def group_size(hq, hkv):
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return hq // hkv


def attention_forward(q, k, v, scale=None, causal=True):
    """Full forward: returns (o [S, Hq, d], lse [Hq, Sq]).

    Queries and keys share one position axis when ``causal`` (the causal rule
    j <= i on global positions).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    g = group_size(hq, hkv)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((sq, hq, d))
    lse = np.zeros((hq, sq))
    if causal:
        future = np.arange(sk)[None, :] > np.arange(sq)[:, None]
    for h in range(hq):
        kh, vh = k[:, h // g, :], v[:, h // g, :]
        s = scale * (q[:, h, :] @ kh.T)
        if causal:
            s = np.where(future, -np.inf, s)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True)
        lse[h] = (m + np.log(den))[:, 0]
        o[:, h, :] = (e / den) @ vh
    return o, lse


def attention_backward(q, k, v, do, scale=None, causal=True, d_from_bf16_o=False):
    """Full backward: returns (dq, dk, dv, o, lse, D) in float64.

    Recomputes the forward from its definition, then applies the chain rule
    through softmax (dS = P * (dP - D), D_i = sum_j P_ij dP_ij = dO_i . O_i).
    ``d_from_bf16_o``: see ``_dvec``.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    g = group_size(hq, hkv)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o, lse = attention_forward(q, k, v, scale, causal)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dvec = _dvec(do, o, d_from_bf16_o).T
    if causal:
        future = np.arange(sk)[None, :] > np.arange(sq)[:, None]
    for h in range(hq):
        kv = h // g
        kh, vh = k[:, kv, :], v[:, kv, :]
        s = scale * (q[:, h, :] @ kh.T)
        if causal:
            s = np.where(future, -np.inf, s)
        p = np.exp(s - lse[h][:, None])
        dp = do[:, h, :] @ vh.T
        ds = p * (dp - dvec[h][:, None])
        dq[:, h, :] = scale * (ds @ kh)
        dk[:, kv, :] += scale * (ds.T @ q[:, h, :])
        dv[:, kv, :] += p.T @ do[:, h, :]
    return dq, dk, dv, o, lse, dvec


def attention_rows(q, k, v, rows, heads, scale=None):
    """Causal forward for selected query rows of selected heads.

    Returns (o [len(heads), len(rows), d], lse [len(heads), len(rows)]).
    Each row i is softmax over keys 0..i exactly as in ``attention_forward``;
    rows are batched in groups only to bound memory (no blocking over keys).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    sq, hq, d = q.shape
    hkv = k.shape[1]
    g = group_size(hq, hkv)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.asarray(rows, dtype=np.int64)
    o = np.zeros((len(heads), len(rows), d))
    lse = np.zeros((len(heads), len(rows)))
    group = max(1, int(2 ** 25 // max(1, k.shape[0])))
    for a, h in enumerate(heads):
        kh = np.ascontiguousarray(k[:, h // g, :])
        vh = np.ascontiguousarray(v[:, h // g, :])
        for r0 in range(0, len(rows), group):
            rr = rows[r0:r0 + group]
            n = int(rr.max()) + 1
            s = scale * (q[rr, h, :] @ kh[:n].T)
            s = np.where(np.arange(n)[None, :] > rr[:, None], -np.inf, s)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            den = e.sum(axis=1, keepdims=True)
            lse[a, r0:r0 + group] = (m + np.log(den))[:, 0]
            o[a, r0:r0 + group] = (e / den) @ vh[:n]
    return o, lse


def attention_backward_rows(q, k, v, do, rows, heads, scale=None, d_from_bf16_o=False):
    """dQ for selected query rows of selected heads (causal).

    dQ_i = scale * sum_{j<=i} P_ij (dP_ij - D_i) k_j with D_i = dO_i . O_i,
    where O_i and LSE_i come from ``attention_rows``.
    Returns dq [len(heads), len(rows), d].
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    sq, hq, d = q.shape
    g = group_size(hq, k.shape[1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.asarray(rows, dtype=np.int64)
    o, lse = attention_rows(q, k, v, rows, heads, scale)
    dq = np.zeros((len(heads), len(rows), d))
    group = max(1, int(2 ** 25 // max(1, k.shape[0])))
    for a, h in enumerate(heads):
        kh = np.ascontiguousarray(k[:, h // g, :])
        vh = np.ascontiguousarray(v[:, h // g, :])
        for r0 in range(0, len(rows), group):
            rr = rows[r0:r0 + group]
            n = int(rr.max()) + 1
            s = scale * (q[rr, h, :] @ kh[:n].T)
            s = np.where(np.arange(n)[None, :] > rr[:, None], -np.inf, s)
            p = np.exp(s - lse[a, r0:r0 + group][:, None])
            dvec = _dvec(do[rr, h, :], o[a, r0:r0 + group], d_from_bf16_o)
            dp = do[rr, h, :] @ vh[:n].T
            ds = p * (dp - dvec[:, None])
            dq[a, r0:r0 + group] = scale * (ds @ kh[:n])
    return dq


def attention_backward_keys(q, k, v, do, keys, kv_head, scale=None, d_from_bf16_o=False):
    """dK and dV for selected key positions of one kv head (causal).

    dV_j = sum_{h in group} sum_{i>=j} P_ij dO_i and
    dK_j = scale * sum_{h in group} sum_{i>=j} dS_ij q_i.  Needs LSE_i and
    D_i for every query i >= min(keys); those rows are recomputed here with
    ``attention_rows``.  Returns (dk [len(keys), d], dv [len(keys), d]).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    sq, hq, d = q.shape
    g = group_size(hq, k.shape[1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    keys = np.asarray(keys, dtype=np.int64)
    i0 = int(keys.min())
    rows = np.arange(i0, sq)
    heads = list(range(kv_head * g, (kv_head + 1) * g))
    o, lse = attention_rows(q, k, v, rows, heads, scale)
    kj = k[keys, kv_head, :]
    vj = v[keys, kv_head, :]
    dk = np.zeros((len(keys), d))
    dv = np.zeros((len(keys), d))
    for a, h in enumerate(heads):
        qh = q[rows, h, :]
        doh = do[rows, h, :]
        dvec = _dvec(doh, o[a], d_from_bf16_o)
        s = scale * (qh @ kj.T)
        s = np.where(keys[None, :] > rows[:, None], -np.inf, s)
        p = np.exp(s - lse[a][:, None])
        dp = doh @ vj.T
        ds = p * (dp - dvec[:, None])
        dv += p.T @ doh
        dk += scale * (ds.T @ qh)
    return dk, dv
