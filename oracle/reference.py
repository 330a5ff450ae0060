"""Small fp64 numpy models of attention -- TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this module.  Nothing here is shared with the CUDA path.

Two models live here, both for one (batch, head) slice ``q [Nq, d]``,
``k [Nk, d]``, ``v [Nk, dv]`` with absolute token positions ``q_start`` and
``k_start`` (FlashAttention from Scratch, sec. 5: a causal pair is allowed iff
key position <= query position):

* :func:`dense_attention` -- the definition, with the full score matrix S and
  probability matrix P materialised (sec. 2 "Begin with one attention row").
* :func:`streaming_attention` -- the online-softmax recurrence in the order the
  pages give it: running maximum m, running sum l and unnormalised
  accumulator u per row, updated tile by tile (sec. 4.1 "Maintain three
  quantities"; FlashAttention Cheat Sheet, sec. 5 "Why online softmax is
  globally exact"), with the optional conditional rescale of sec. 11.3
  "Derive conditional rescaling correctly" (threshold ``tau``) and an
  arbitrary KV-tile visiting order.

:func:`merge_states` and :func:`merge_lse` combine partitions (sec. 4.3
"Merge independently computed partitions").
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def allowed_mask(nq: int, nk: int, causal: bool, q_start: int = 0, k_start: int = 0) -> np.ndarray:
    """Boolean [nq, nk]: True where the (query, key) pair may attend."""
    if not causal:
        return np.ones((nq, nk), dtype=bool)
    qi = np.arange(nq)[:, None] + q_start
    kj = np.arange(nk)[None, :] + k_start
    return kj <= qi


def scores(q, k, scale, causal=False, q_start=0, k_start=0):
    """S = scale * q k^T with -inf on disallowed pairs (fp64)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    s = (q @ k.T) * scale
    s = np.where(allowed_mask(q.shape[0], k.shape[0], causal, q_start, k_start), s, NEG_INF)
    return s


def softmax_rows(s):
    """Row softmax with the maximum subtracted; all-masked rows give zeros."""
    s = np.asarray(s, dtype=np.float64)
    m = s.max(axis=-1, keepdims=True)
    shift = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - shift)
    l = p.sum(axis=-1, keepdims=True)
    return np.where(l > 0, p / np.where(l > 0, l, 1.0), 0.0)


def dense_attention(q, k, v, scale=None, causal=False, q_start=0, k_start=0, return_p=False):
    """Materialised attention: returns (o [Nq, dv], lse [Nq]) and optionally P.

    Fully masked rows give o = 0 and lse = -inf (sec. 4.4).
    """
    q = np.asarray(q, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[1])
    s = scores(q, k, scale, causal, q_start, k_start)
    m = s.max(axis=-1)
    shift = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - shift[:, None])
    l = e.sum(axis=-1)
    p = np.where(l[:, None] > 0, e / np.where(l > 0, l, 1.0)[:, None], 0.0)
    o = p @ v
    lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)
    if return_p:
        return o, lse, p
    return o, lse


def _finish(ref, ell, u):
    """o = u / l and lse = ref + ln l; empty rows give 0 and -inf."""
    ok = ell > 0
    denom = np.where(ok, ell, 1.0)
    o = np.where(ok[:, None], u / denom[:, None], 0.0)
    lse = np.where(ok, ref + np.log(denom), NEG_INF)
    return o, lse


def streaming_attention(q, k, v, scale=None, block_q=32, block_k=64, causal=False,
                        q_start=0, k_start=0, tau=None, kv_order=None, trace=None):
    """Online-softmax attention over KV tiles; returns (o, lse).

    ``tau=None`` moves the reference to the new maximum whenever it rises
    (the plain recurrence).  A number keeps the reference while the tile
    maximum exceeds it by at most ``tau`` (natural-log units) and otherwise
    moves it to the new maximum.  ``kv_order`` permutes the KV tiles.
    ``trace`` (a list) receives (m, l, u) after every tile of query block 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[1])
    nk_tiles = (k.shape[0] + block_k - 1) // block_k
    order = list(range(nk_tiles)) if kv_order is None else list(kv_order)
    assert sorted(order) == list(range(nk_tiles))
    outs, lses = [], []
    for i0 in range(0, q.shape[0], block_q):
        qt = q[i0:i0 + block_q]
        ref = np.full(qt.shape[0], NEG_INF)
        ell = np.zeros(qt.shape[0])
        u = np.zeros((qt.shape[0], v.shape[1]))
        for t in order:
            j0 = t * block_k
            kt, vt = k[j0:j0 + block_k], v[j0:j0 + block_k]
            s = scores(qt, kt, scale, causal, q_start + i0, k_start + j0)
            tile_max = s.max(axis=-1)
            if tau is None:
                new_ref = np.maximum(ref, tile_max)
            else:
                keep = (tile_max - ref) <= tau  # False when ref is -inf and tile is not
                new_ref = np.where(keep, ref, np.maximum(ref, tile_max))
            # zero is a computational shift for rows that are still empty
            shift = np.where(np.isfinite(new_ref), new_ref, 0.0)
            alpha = np.where(np.isfinite(ref), np.exp(ref - shift), 0.0)
            p = np.exp(s - shift[:, None])
            ell = alpha * ell + p.sum(axis=-1)
            u = alpha[:, None] * u + p @ vt
            ref = new_ref
            if trace is not None and i0 == 0:
                trace.append((ref.copy(), ell.copy(), u.copy()))
        o, lse = _finish(ref, ell, u)
        outs.append(o)
        lses.append(lse)
    return np.concatenate(outs), np.concatenate(lses)


def partition_state(q, k, v, scale, causal=False, q_start=0, k_start=0):
    """(m, l, u) of one KV partition, computed directly from its scores."""
    s = scores(q, k, scale, causal, q_start, k_start)
    m = s.max(axis=-1)
    shift = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - shift[:, None])
    return m, p.sum(axis=-1), p @ np.asarray(v, dtype=np.float64)


def merge_states(a, b):
    """Merge (m, l, u) states of two disjoint key subsets (sec. 4.3)."""
    ma, la, ua = a
    mb, lb, ub = b
    m = np.maximum(ma, mb)
    shift = np.where(np.isfinite(m), m, 0.0)
    wa = np.where(np.isfinite(ma), np.exp(ma - shift), 0.0)
    wb = np.where(np.isfinite(mb), np.exp(mb - shift), 0.0)
    return m, wa * la + wb * lb, wa[:, None] * ua + wb[:, None] * ub


def merge_lse(oa, la, ob, lb):
    """Merge normalised partial outputs by their natural-log normalisers."""
    L = np.logaddexp(la, lb)
    ok = np.isfinite(L)
    Ls = np.where(ok, L, 0.0)
    wa = np.where(np.isfinite(la), np.exp(la - Ls), 0.0)
    wb = np.where(np.isfinite(lb), np.exp(lb - Ls), 0.0)
    o = wa[:, None] * oa + wb[:, None] * ob
    return np.where(ok[:, None], o, 0.0), np.where(ok, L, NEG_INF)
