"""Pins of the fp64 backward oracle (oracle/backward.py) to things other than
itself: central finite differences of an independently written forward,
PyTorch autograd through an ordinary dense softmax, closed forms, exact
invariants of the gradients, and the pages' tile-by-tile recomputation order
(FlashAttention from Scratch, sec. 8 "Backward: spend arithmetic to save
memory", "A backward implementation you can check")."""
import math

import numpy as np
import pytest
import torch

from oracle.backward import attention_bwd, attention_bwd_varlen, recomputed_backward
from oracle.reference import blocks, definition, positions


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _loss_direct(q, k, v, do, scale, causal):
    """sum(O * dO), written with explicit loops (no shared helpers)."""
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    r = Hq // Hkv
    total = 0.0
    for b in range(B):
        for h in range(Hq):
            for i in range(Lq):
                sc = []
                for j in range(Lk):
                    if causal and j > i + (Lk - Lq):
                        continue
                    sc.append((j, scale * float(np.dot(q[b, h, i], k[b, h // r, j]))))
                if not sc:
                    continue
                m = max(x for _, x in sc)
                w = [(j, math.exp(x - m)) for j, x in sc]
                z = sum(x for _, x in w)
                o = sum(x / z * v[b, h // r, j] for j, x in w)
                total += float(np.dot(o, do[b, h, i]))
    return total


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(3, 5), (5, 3), (4, 4)])
def test_finite_differences(causal, Lq, Lk):
    B, Hq, Hkv, D = 1, 2, 1, 3
    q = _rand((B, Hq, Lq, D), 1)
    k = _rand((B, Hkv, Lk, D), 2)
    v = _rand((B, Hkv, Lk, D), 3)
    do = _rand((B, Hq, Lq, D), 4)
    scale = 0.7
    dq, dk, dv = attention_bwd(q, k, v, do, scale, causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            fp = _loss_direct(q, k, v, do, scale, causal)
            x[idx] = old - h
            fm = _loss_direct(q, k, v, do, scale, causal)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(g, num, atol=1e-7, rtol=1e-6, err_msg=name)


def _autograd(q, k, v, do, scale, causal):
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    r = q.shape[1] // k.shape[1]
    kr, vr = kt.repeat_interleave(r, dim=1), vt.repeat_interleave(r, dim=1)
    s = torch.einsum("bhid,bhjd->bhij", qt, kr) * scale
    Lq, Lk = q.shape[2], k.shape[2]
    if causal:
        allowed = torch.arange(Lk)[None, :] <= torch.arange(Lq)[:, None] + (Lk - Lq)
        s = s.masked_fill(~allowed, float("-inf"))
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)  # rows with no key: P = 0
    o = torch.einsum("bhij,bhjd->bhid", p, vr)
    return torch.autograd.grad(o, (qt, kt, vt), torch.tensor(do))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,D", [(2, 4, 2, 37, 53, 16), (1, 3, 3, 64, 40, 8), (1, 4, 1, 20, 20, 32)])
def test_matches_autograd(causal, B, Hq, Hkv, Lq, Lk, D):
    q = _rand((B, Hq, Lq, D), 5)
    k = _rand((B, Hkv, Lk, D), 6)
    v = _rand((B, Hkv, Lk, D), 7)
    do = _rand((B, Hq, Lq, D), 8)
    scale = 1 / math.sqrt(D)
    got = attention_bwd(q, k, v, do, scale, causal, block=16)
    ref = _autograd(q, k, v, do, scale, causal)
    for g, e, n in zip(got, ref, "qkv"):
        np.testing.assert_allclose(g, e.numpy(), atol=1e-11, rtol=1e-9, err_msg=n)


def test_single_key_closed_form():
    """One key: P = 1 for every row, so dQ = dK = 0 and dV = sum of dO over
    the rows (and heads) that read it."""
    B, Hq, Hkv, Lq, D = 2, 4, 2, 7, 8
    q, k, v, do = _rand((B, Hq, Lq, D), 9), _rand((B, Hkv, 1, D), 10), _rand((B, Hkv, 1, D), 11), \
        _rand((B, Hq, Lq, D), 12)
    dq, dk, dv = attention_bwd(q, k, v, do, 0.3, False)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    expect = do.reshape(B, Hkv, Hq // Hkv, Lq, D).sum(axis=(2, 3))
    np.testing.assert_allclose(dv[:, :, 0], expect, atol=1e-12)


def test_constant_values_give_no_score_gradient():
    """All value rows equal: O = v whatever P is, so dQ = dK = 0."""
    q, k, do = _rand((1, 2, 9, 4), 13), _rand((1, 2, 11, 4), 14), _rand((1, 2, 9, 4), 15)
    v = np.broadcast_to(_rand((4,), 16), (1, 2, 11, 4)).copy()
    dq, dk, dv = attention_bwd(q, k, v, do, 0.5, True)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.abs(dv).max() > 0.1


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    """Rows of dS sum to zero, so sum_j dK_j = 0; rows of P sum to one, so
    sum_j dV_j = sum of dO over the rows that see at least one key."""
    B, Hq, Hkv, Lq, Lk, D = 1, 4, 2, 30, 25, 6
    q, k, v, do = (_rand(s, 17 + i, 2.0) for i, s in
                   enumerate([(B, Hq, Lq, D), (B, Hkv, Lk, D), (B, Hkv, Lk, D), (B, Hq, Lq, D)]))
    dq, dk, dv = attention_bwd(q, k, v, do, 0.4, causal)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-10)
    seen = np.ones(Lq, dtype=bool) if not causal else (np.arange(Lq) + (Lk - Lq) >= 0)
    expect = (do[:, :, seen].reshape(B, Hkv, Hq // Hkv, -1, D)).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(axis=2), expect, atol=1e-10)


def test_gqa_equals_repeated_heads_summed():
    B, Hq, Hkv, Lq, Lk, D = 1, 6, 2, 12, 17, 4
    q, k, v, do = _rand((B, Hq, Lq, D), 30), _rand((B, Hkv, Lk, D), 31), _rand((B, Hkv, Lk, D), 32), \
        _rand((B, Hq, Lq, D), 33)
    dq, dk, dv = attention_bwd(q, k, v, do, 0.5, True)
    r = Hq // Hkv
    dq2, dk2, dv2 = attention_bwd(q, np.repeat(k, r, axis=1), np.repeat(v, r, axis=1), do, 0.5, True)
    np.testing.assert_allclose(dq, dq2, atol=1e-12)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, r, Lk, D).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, r, Lk, D).sum(axis=2), atol=1e-12)


@pytest.mark.parametrize("block_q,block_k", [(1, 1), (3, 4), (32, 64), (5, 2)])
def test_recomputation_matches_definition(block_q, block_k):
    """The pages' case: five queries at the end of a nine-key sequence, causal,
    recomputed tile by tile from the saved output and log-sum-exp."""
    q, k, v, do = _rand((5, 7), 40), _rand((9, 7), 41), _rand((9, 3), 42), _rand((5, 3), 43)
    scale = 1 / math.sqrt(7)
    o, lse = definition(q, k, v, scale=scale, causal=True, qpos=positions(5, 4))[2:]
    got = recomputed_backward(q, k, v, o, lse, do, scale, causal=True, qpos=positions(5, 4),
                              query_blocks=blocks(5, block_q), key_blocks=blocks(9, block_k))
    ref = attention_bwd(q[None, None], k[None, None], v[None, None], do[None, None], scale, True)
    for g, e in zip(got, ref):
        np.testing.assert_allclose(g, e[0, 0], atol=1e-12)


def test_recomputation_handles_rows_without_keys():
    """q_start = -2: the first two queries precede every key (LSE = -inf)."""
    q, k, v, do = _rand((6, 4), 50), _rand((5, 4), 51), _rand((5, 4), 52), _rand((6, 4), 53)
    o, lse = definition(q, k, v, scale=0.5, causal=True, qpos=positions(6, -2))[2:]
    assert np.isneginf(lse[:2]).all()
    dq, dk, dv = recomputed_backward(q, k, v, o, lse, do, 0.5, causal=True, qpos=positions(6, -2),
                                     query_blocks=blocks(6, 4), key_blocks=blocks(5, 2))
    assert np.all(np.isfinite(dq)) and np.abs(dq[:2]).max() == 0.0
    # same problem in the dense layout: Lq = 6 > Lk = 5 puts the offset at -1,
    # so compare with the matching bottom-right case instead
    o2, lse2 = definition(q, k, v, scale=0.5, causal=True, qpos=positions(6, -1))[2:]
    ref = attention_bwd(q[None, None], k[None, None], v[None, None], do[None, None], 0.5, True)
    got = recomputed_backward(q, k, v, o2, lse2, do, 0.5, causal=True, qpos=positions(6, -1),
                              query_blocks=blocks(6, 4), key_blocks=blocks(5, 2))
    for g, e in zip(got, ref):
        np.testing.assert_allclose(g, e[0, 0], atol=1e-12)


def test_sampled_rows_equal_full_result():
    B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 50, 70, 8
    q, k, v, do = _rand((B, Hq, Lq, D), 60), _rand((B, Hkv, Lk, D), 61), _rand((B, Hkv, Lk, D), 62), \
        _rand((B, Hq, Lq, D), 63)
    full = attention_bwd(q, k, v, do, 0.35, True, block=8)
    qr = np.array([0, 49, 50, 123, 399])
    kr = np.array([0, 69, 70, 200, 279])
    dq, dk, dv = attention_bwd(q, k, v, do, 0.35, True, q_rows=qr, k_rows=kr, block=16)
    np.testing.assert_allclose(dq, full[0].reshape(-1, D)[qr], atol=1e-12)
    np.testing.assert_allclose(dk, full[1].reshape(-1, D)[kr], atol=1e-12)
    np.testing.assert_allclose(dv, full[2].reshape(-1, D)[kr], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_autograd_per_sequence(causal):
    # packed sequences with Lq != Lk, an empty query sequence and an empty key
    # sequence; each sequence is checked against PyTorch autograd through a
    # dense softmax of that sequence alone (bottom-right causal alignment)
    lq, lk = [5, 0, 9, 3, 7], [8, 4, 9, 0, 2]
    Hq, Hkv, D = 4, 2, 6
    cq = np.concatenate([[0], np.cumsum(lq)])
    ck = np.concatenate([[0], np.cumsum(lk)])
    q = _rand((cq[-1], Hq, D), 1)
    k = _rand((ck[-1], Hkv, D), 2)
    v = _rand((ck[-1], Hkv, D), 3)
    do = _rand((cq[-1], Hq, D), 4)
    scale = 0.4
    dq, dk, dv = attention_bwd_varlen(q, k, v, do, cq, ck, scale, causal)
    r = Hq // Hkv
    for s in range(len(lq)):
        q0, q1, k0, k1 = cq[s], cq[s + 1], ck[s], ck[s + 1]
        if q1 == q0 or k1 == k0:
            # no pairs: the sequence's gradients stay zero
            assert np.all(dq[q0:q1] == 0) and np.all(dk[k0:k1] == 0) and np.all(dv[k0:k1] == 0)
            continue
        Q = torch.tensor(q[q0:q1].transpose(1, 0, 2), requires_grad=True)
        K = torch.tensor(k[k0:k1].transpose(1, 0, 2), requires_grad=True)
        V = torch.tensor(v[k0:k1].transpose(1, 0, 2), requires_grad=True)
        G = torch.tensor(do[q0:q1].transpose(1, 0, 2))
        Lq_, Lk_ = q1 - q0, k1 - k0
        S = scale * Q @ K.repeat_interleave(r, 0).transpose(1, 2)
        if causal:
            allowed = torch.arange(Lk_)[None, :] <= torch.arange(Lq_)[:, None] + (Lk_ - Lq_)
            S = S.masked_fill(~allowed, float("-inf"))
        P = torch.softmax(S, dim=-1)
        P = torch.nan_to_num(P, nan=0.0)  # rows without an allowed key
        O = P @ V.repeat_interleave(r, 0)
        (O * G).sum().backward()
        assert np.allclose(dq[q0:q1], Q.grad.numpy().transpose(1, 0, 2), atol=1e-12)
        assert np.allclose(dk[k0:k1], K.grad.numpy().transpose(1, 0, 2), atol=1e-12)
        assert np.allclose(dv[k0:k1], V.grad.numpy().transpose(1, 0, 2), atol=1e-12)
