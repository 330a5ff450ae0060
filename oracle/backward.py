"""fp64 oracle for the attention backward pass -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  Nothing here is shared with the CUDA path.

The loss is L = sum(O * dO) for a given upstream gradient dO (so dO is
dL/dO).  With the scale c, the mask M (0 or -inf) and, per (batch, query
head) slice, S = c Q K^T + M, P = row softmax of S, O = P V, the gradients are
the plain definitions (FlashAttention from Scratch, sec. 8 "Backward: spend
arithmetic to save memory"):

    dV = P^T dO
    dP = dO V^T
    delta_i = sum_t P_it dP_it = O_i . dO_i
    dS = P * (dP - delta)          (row-wise delta)
    dQ = c dS K,    dK = c dS^T Q

Grouped-query attention: the gradient of a KV head is the sum over the query
heads that read it (sec. 9.2).  Causal masking is bottom-right aligned, as in
the forward oracle.  Query rows with no allowed key have P = 0 and
contribute nothing.

:func:`attention_bwd` evaluates these definitions with materialised S and P,
one block of query rows at a time (numpy matrix products in fp64), and can
restrict the returned rows of dQ and of dK/dV to samples so that full-size
problems can be checked.  :func:`recomputed_backward` is a second model in
the recomputation style the pages describe (P rebuilt from the saved
natural-log normaliser instead of being kept, delta from the saved output),
organised the way a key-parallel GPU backward is: each key block owns its
dK and dV rows and sweeps every query block, while dQ collects partial
products from every key block.  The tests pin the two against each other,
against finite differences and against closed forms.
"""
from __future__ import annotations

import numpy as np

from .reference import allowed, exp_shifted, positions, probabilities, score_matrix


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def attention_bwd(q, k, v, do, scale: float, causal: bool = False, q_rows=None, k_rows=None,
                  block: int = 1024):
    """Gradients (dq, dk, dv) of sum(O * do) for dense [B, H, L, D] inputs.

    q [B, Hq, Lq, D]; k, v [B, Hkv, Lk, D]; do [B, Hq, Lq, D].  With q_rows
    (flat indices into B*Hq*Lq) dq is returned only for those rows, shape
    [n, D]; with k_rows (flat indices into B*Hkv*Lk) dk and dv only for those
    rows.  Without them the full tensors come back in float64.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    r = Hq // Hkv
    mask_all = allowed(positions(Lq, Lk - Lq), positions(Lk), causal)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    want_q = None if q_rows is None else set(int(x) for x in np.asarray(q_rows).ravel())
    want_kv_heads = None
    if k_rows is not None:
        kr = np.asarray(k_rows).ravel()
        want_kv_heads = set(int(x) for x in kr // Lk)
    for b in range(B):
        for h in range(Hq):
            hk = h // r
            bh = b * Hq + h
            need_q = want_q is None or any(bh * Lq <= x < (bh + 1) * Lq for x in want_q)
            need_kv = want_kv_heads is None or (b * Hkv + hk) in want_kv_heads
            if not (need_q or need_kv):
                continue
            K, V = k[b, hk], v[b, hk]
            for i0 in range(0, Lq, block):
                i1 = min(Lq, i0 + block)
                Q, G = q[b, h, i0:i1], do[b, h, i0:i1]
                s = (Q @ K.T) * scale
                s = np.where(mask_all[i0:i1], s, -np.inf)
                p = probabilities(s)
                o = p @ V
                delta = (o * G).sum(axis=1)
                dp = G @ V.T
                ds = p * (dp - delta[:, None])
                if need_q:
                    dq[b, h, i0:i1] = scale * (ds @ K)
                if need_kv:
                    dk[b, hk] += scale * (ds.T @ Q)
                    dv[b, hk] += p.T @ G
    if q_rows is not None:
        dq = dq.reshape(-1, D)[np.asarray(q_rows).ravel()]
    if k_rows is not None:
        idx = np.asarray(k_rows).ravel()
        dk = dk.reshape(-1, D)[idx]
        dv = dv.reshape(-1, v.shape[-1])[idx]
    return dq, dk, dv


def recomputed_backward(q, k, v, o, lse, do, scale: float, causal: bool = False, qpos=None,
                        kpos=None, query_blocks=None, key_blocks=None):
    """Gradients (dq, dk, dv) of sum(O * do) for one (batch, head) slice,
    from the saved forward results o [n, dv] and lse [n] (natural log).

    q [n, d], k [m, d], v [m, dv]; ``qpos``/``kpos`` are token positions
    for the causal mask (key position <= query position).  ``query_blocks``
    and ``key_blocks`` are (start, stop) ranges; each key block is finished
    (its dK, dV rows written) before the next one starts.
    """
    q, k, v, o, lse, do = (_f64(x) for x in (q, k, v, o, lse, do))
    n, m = q.shape[0], k.shape[0]
    qpos = positions(n) if qpos is None else np.asarray(qpos)
    kpos = positions(m) if kpos is None else np.asarray(kpos)
    query_blocks = [(0, n)] if query_blocks is None else list(query_blocks)
    key_blocks = [(0, m)] if key_blocks is None else list(key_blocks)
    # delta_i = sum_t P_it dP_it equals the row dot product of O and dO
    delta = np.einsum("id,id->i", o, do)
    dq_sum = np.zeros_like(q)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    for c0, c1 in key_blocks:
        kb, vb = k[c0:c1], v[c0:c1]
        dk_sum = np.zeros_like(kb)
        for r0, r1 in query_blocks:
            s = score_matrix(q[r0:r1], kb, scale, qpos[r0:r1], kpos[c0:c1], causal)
            # P_ij = exp(s_ij - lse_i); masked pairs (and rows with no key) give 0
            p = exp_shifted(s, lse[r0:r1, None])
            ds = p * (do[r0:r1] @ vb.T - delta[r0:r1, None])
            dv[c0:c1] += p.T @ do[r0:r1]
            dk_sum += ds.T @ q[r0:r1]
            dq_sum[r0:r1] += ds @ kb
        dk[c0:c1] = scale * dk_sum
    return scale * dq_sum, dk, dv


def attention_bwd_varlen(q, k, v, do, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool = False):
    """Gradients of sum(O * do) for a packed batch: q, do [Tq, Hq, D],
    k, v [Tk, Hkv, D]; sequence s owns query tokens cu_seqlens_q[s] ..
    cu_seqlens_q[s+1] - 1 and key tokens cu_seqlens_k[s] .. cu_seqlens_k[s+1] - 1.
    Every sequence is an independent problem (its own causal alignment), so
    the gradients are those of :func:`attention_bwd` on each sequence, placed
    back at the sequence's tokens; a sequence without query rows gives zero
    dK and dV, one without keys zero dQ."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    cq = [int(x) for x in np.asarray(cu_seqlens_q).tolist()]
    ck = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[s], cq[s + 1], ck[s], ck[s + 1]
        if q1 <= q0 or k1 <= k0:
            continue
        # [T, H, D] slices as [1, H, T, D] problems
        qs = q[q0:q1].transpose(1, 0, 2)[None]
        dos = do[q0:q1].transpose(1, 0, 2)[None]
        ks = k[k0:k1].transpose(1, 0, 2)[None]
        vs = v[k0:k1].transpose(1, 0, 2)[None]
        a, b, c = attention_bwd(qs, ks, vs, dos, scale, causal)
        dq[q0:q1] = a[0].transpose(1, 0, 2)
        dk[k0:k1] = b[0].transpose(1, 0, 2)
        dv[k0:k1] = c[0].transpose(1, 0, 2)
    return dq, dk, dv
