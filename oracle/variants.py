"""fp64 oracle for programmable attention variants -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  Nothing here is shared with the CUDA path.

The pages describe two ways to vary the kernel (FlashAttention from
Scratch, sec. 12 "Programmable attention: FlexAttention meets FA4"): modify
a score before the softmax, S'_ij = f(S_ij, i, j), and restrict which
query-key pairs may attend.  The variants evaluated here, with the reading
taken for each:

* window (left, right): key j is allowed for query i iff
  c_i - left <= j <= c_i + right, where c_i = i + (Lk - Lq) is the query's
  position in the key sequence (bottom-right alignment, as for the causal
  mask); a negative bound is unlimited.  (-1, 0) is the causal mask, and a
  causal window of width w is (w - 1, 0).
* soft-capping (cap > 0): S' = cap * tanh(S / cap) on the scaled scores.
* ALiBi (one slope per query head): S' = S - slope_h * |c_i - j|, the
  positional bias proportional to the distance from the query's position.

The scale multiplies Q K^T first, the score modifier follows, the mask is
applied last; then softmax, O and the natural-log LSE as in the plain
definition (rows with no allowed key: O = 0, LSE = -inf).
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def variant_scores(q, k, scale, window=(-1, -1), softcap=0.0, slope=0.0, Lq=None, Lk=None, q_offset=0):
    """Modified and masked scores of one slice: q [n, d] are queries
    q_offset .. q_offset + n - 1 of a problem with Lq queries and Lk keys."""
    q, k = _f64(q), _f64(k)
    Lq = q.shape[0] if Lq is None else Lq
    Lk = k.shape[0] if Lk is None else Lk
    s = (q @ k.T) * scale
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    c = (np.arange(q.shape[0]) + q_offset + (Lk - Lq))[:, None]
    j = np.arange(k.shape[0])[None, :]
    if slope != 0.0:
        s = s - slope * np.abs(c - j)
    left, right = window
    allowed = np.ones(s.shape, dtype=bool)
    if left >= 0:
        allowed &= j >= c - left
    if right >= 0:
        allowed &= j <= c + right
    return np.where(allowed, s, -np.inf)


def _softmax_out(s, v):
    m = s.max(axis=1, keepdims=True)
    finite = np.isfinite(m)
    p = np.exp(s - np.where(finite, m, 0.0))
    ell = p.sum(axis=1, keepdims=True)
    o = np.where(ell > 0, (p @ v) / np.where(ell > 0, ell, 1.0), 0.0)
    lse = np.where(ell[:, 0] > 0, m[:, 0] + np.log(np.where(ell[:, 0] > 0, ell[:, 0], 1.0)), -np.inf)
    return o, lse


def attention_variant(q, k, v, scale: float, window=(-1, -1), softcap: float = 0.0, alibi_slopes=None,
                      rows=None, block: int = 1024):
    """Dense [B, H, L, D] inputs (GQA: query head h reads KV head h // (Hq/Hkv)).
    Returns (o [B, Hq, Lq, D], lse [B, Hq, Lq]) in float64, or, with rows
    (flat indices into B*Hq*Lq), (o [n, D], lse [n])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    r = Hq // Hkv
    slopes = np.zeros(Hq) if alibi_slopes is None else _f64(alibi_slopes).reshape(Hq)
    o = np.zeros((B, Hq, Lq, v.shape[-1]))
    lse = np.full((B, Hq, Lq), -np.inf)
    want = None if rows is None else np.asarray(rows).ravel()
    for b in range(B):
        for h in range(Hq):
            bh = b * Hq + h
            if want is not None:
                sel = want[(want >= bh * Lq) & (want < (bh + 1) * Lq)] - bh * Lq
                if sel.size == 0:
                    continue
            for i0 in range(0, Lq, block):
                i1 = min(Lq, i0 + block)
                if want is not None and not np.any((sel >= i0) & (sel < i1)):
                    continue
                s = variant_scores(q[b, h, i0:i1], k[b, h // r], scale, window, softcap, slopes[h], Lq, Lk, i0)
                o[b, h, i0:i1], lse[b, h, i0:i1] = _softmax_out(s, v[b, h // r])
    if want is not None:
        return o.reshape(-1, o.shape[-1])[want], lse.reshape(-1)[want]
    return o, lse


def attention_variant_varlen(q, k, v, cu_q, cu_k, scale: float, window=(-1, -1), softcap: float = 0.0,
                             alibi_slopes=None):
    """Packed [T, H, D] inputs with int prefix offsets: every sequence is an
    independent problem with its own bottom-right alignment.  Returns
    (o [Tq, Hq, D], lse [Hq, Tq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, Hq, D = q.shape
    o = np.zeros((Tq, Hq, v.shape[-1]))
    lse = np.full((Hq, Tq), -np.inf)
    cu_q, cu_k = np.asarray(cu_q), np.asarray(cu_k)
    for s_ in range(len(cu_q) - 1):
        a, b = int(cu_q[s_]), int(cu_q[s_ + 1])
        c, d = int(cu_k[s_]), int(cu_k[s_ + 1])
        if b == a:
            continue
        qs = q[a:b].transpose(1, 0, 2)[None]
        ks = k[c:d].transpose(1, 0, 2)[None]
        vs = v[c:d].transpose(1, 0, 2)[None]
        if d == c:
            continue  # no keys: O = 0, LSE = -inf
        os_, ls_ = attention_variant(qs, ks, vs, scale, window, softcap, alibi_slopes)
        o[a:b] = os_[0].transpose(1, 0, 2)
        lse[:, a:b] = ls_[0]
    return o, lse


def attention_variant_bwd(q, k, v, do, scale: float, window=(-1, -1), softcap: float = 0.0, alibi_slopes=None,
                          block: int = 1024):
    """Gradients (dq, dk, dv) of sum(O * do) for the variant forward above,
    dense [B, H, L, D] inputs.  With S the scaled scores and S' the modified
    ones (FlashAttention from Scratch, sec. 8 and sec. 12):
        P = softmax(S' masked), dV = P^T dO, dP = dO V^T,
        dS' = P * (dP - rowsum(P * dP)),
        dS = dS' * dS'/dS   (soft-capping: 1 - tanh(S / cap)^2; ALiBi and
                             windows: 1, the bias and the mask do not depend on S),
        dQ = scale dS K,  dK = scale dS^T Q."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    r = Hq // Hkv
    slopes = np.zeros(Hq) if alibi_slopes is None else _f64(alibi_slopes).reshape(Hq)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            K, V = k[b, h // r], v[b, h // r]
            for i0 in range(0, Lq, block):
                i1 = min(Lq, i0 + block)
                Q, G = q[b, h, i0:i1], do[b, h, i0:i1]
                s = variant_scores(Q, K, scale, window, softcap, slopes[h], Lq, Lk, i0)
                m = s.max(axis=1, keepdims=True)
                p = np.exp(s - np.where(np.isfinite(m), m, 0.0))
                ell = p.sum(axis=1, keepdims=True)
                p = np.where(ell > 0, p / np.where(ell > 0, ell, 1.0), 0.0)
                dp = G @ V.T
                ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
                if softcap > 0:
                    th = np.tanh((Q @ K.T) * scale / softcap)
                    ds = ds * (1.0 - th * th)
                dq[b, h, i0:i1] = scale * (ds @ K)
                dk[b, h // r] += scale * (ds.T @ Q)
                dv[b, h // r] += p.T @ G
    return dq, dk, dv


def attention_variant_bwd_varlen(q, k, v, do, cu_q, cu_k, scale: float, window=(-1, -1), softcap: float = 0.0,
                                 alibi_slopes=None):
    """Packed [T, H, D] version of :func:`attention_variant_bwd`: every
    sequence is an independent problem; returns (dq, dk, dv) in the packed
    layouts."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    cu_q, cu_k = np.asarray(cu_q), np.asarray(cu_k)
    for s_ in range(len(cu_q) - 1):
        a, b = int(cu_q[s_]), int(cu_q[s_ + 1])
        c, d = int(cu_k[s_]), int(cu_k[s_ + 1])
        if b == a or d == c:
            continue
        sl = lambda t, x, y: t[x:y].transpose(1, 0, 2)[None]
        g = attention_variant_bwd(sl(q, a, b), sl(k, c, d), sl(v, c, d), sl(do, a, b), scale, window, softcap,
                                  alibi_slopes)
        dq[a:b] = g[0][0].transpose(1, 0, 2)
        dk[c:d] = g[1][0].transpose(1, 0, 2)
        dv[c:d] = g[2][0].transpose(1, 0, 2)
    return dq, dk, dv
