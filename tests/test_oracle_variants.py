"""Pins of the variant oracle (oracle/variants.py) to the plain oracle, to
brute force written independently, and to closed forms (FlashAttention from
Scratch, sec. 12 "Programmable attention: FlexAttention meets FA4")."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.variants import attention_variant, attention_variant_varlen, variant_scores


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _bf16_triple(B, Hq, Hkv, Lq, Lk, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, Lq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Lk, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Lk, D), generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("Lq,Lk", [(37, 37), (20, 53), (53, 20)])
def test_window_reduces_to_causal_and_full(Lq, Lk):
    q, k, v = _bf16_triple(1, 4, 2, Lq, Lk, 16, Lq + Lk)
    for window, causal in (((-1, 0), True), ((-1, -1), False), ((10 ** 6, 10 ** 6), False)):
        o, lse = attention_variant(q, k, v, 0.25, window=window)
        ref_o, ref_lse = oracle.attention(q, k, v, scale=0.25, causal=causal)
        np.testing.assert_allclose(o, ref_o, atol=1e-12)
        np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
        fin = np.isfinite(ref_lse)
        np.testing.assert_allclose(lse[fin], ref_lse[fin], atol=1e-12)


def test_causal_window_worked_example():
    """A causal window of width 2 over five tokens: each query sees itself
    and the key before it."""
    s = variant_scores(np.eye(5, 3), np.eye(5, 3), 1.0, window=(1, 0))
    allowed = np.isfinite(s)
    expect = np.array([[1, 0, 0, 0, 0],
                       [1, 1, 0, 0, 0],
                       [0, 1, 1, 0, 0],
                       [0, 0, 1, 1, 0],
                       [0, 0, 0, 1, 1]], dtype=bool)
    np.testing.assert_array_equal(allowed, expect)


def _brute(q, k, v, scale, window, cap, slope, Lq, Lk):
    """Loop form for one slice, with no shared helpers."""
    o = np.zeros((Lq, v.shape[1]))
    lse = np.full(Lq, -np.inf)
    for i in range(Lq):
        c = i + Lk - Lq
        terms = []
        for j in range(Lk):
            if window[0] >= 0 and j < c - window[0]:
                continue
            if window[1] >= 0 and j > c + window[1]:
                continue
            s = scale * sum(q[i, d] * k[j, d] for d in range(q.shape[1]))
            if cap > 0:
                s = cap * math.tanh(s / cap)
            s -= slope * abs(c - j)
            terms.append((j, s))
        if not terms:
            continue
        m = max(x for _, x in terms)
        z = sum(math.exp(x - m) for _, x in terms)
        o[i] = sum(math.exp(x - m) / z * v[j] for j, x in terms)
        lse[i] = m + math.log(z)
    return o, lse


@pytest.mark.parametrize("window,cap,slope", [((2, 1), 0.0, 0.0), ((-1, 0), 3.0, 0.0), ((4, -1), 0.0, 0.3),
                                              ((0, 0), 0.0, 0.0), ((1, 2), 2.0, 0.0), ((-1, -1), 0.0, 0.7),
                                              ((-1, 0), 3.0, 0.3), ((3, 2), 1.5, 0.5)])  # cap, then the bias
@pytest.mark.parametrize("Lq,Lk", [(6, 6), (4, 9), (9, 4)])
def test_brute_force(window, cap, slope, Lq, Lk):
    q, k, v = _rand((1, 2, Lq, 3), 1, 1.5), _rand((1, 1, Lk, 3), 2, 1.5), _rand((1, 1, Lk, 2), 3)
    slopes = np.array([slope, 2 * slope])
    o, lse = attention_variant(q, k, v, 0.8, window, cap, slopes)
    for h in range(2):
        bo, bl = _brute(q[0, h], k[0, 0], v[0, 0], 0.8, window, cap, slopes[h], Lq, Lk)
        np.testing.assert_allclose(o[0, h], bo, atol=1e-12)
        np.testing.assert_array_equal(np.isneginf(lse[0, h]), np.isneginf(bl))
        fin = np.isfinite(bl)
        np.testing.assert_allclose(lse[0, h][fin], bl[fin], atol=1e-12)


def test_softcap_limits_and_two_key_closed_form():
    q, k, v = _rand((1, 1, 5, 4), 4, 3.0), _rand((1, 1, 7, 4), 5, 3.0), _rand((1, 1, 7, 4), 6)
    plain = attention_variant(q, k, v, 0.5)
    big = attention_variant(q, k, v, 0.5, softcap=1e9)
    np.testing.assert_allclose(big[0], plain[0], atol=1e-9)
    # two keys: p1 / p2 = exp(cap tanh(s1/cap) - cap tanh(s2/cap)); capped scores lie in (-cap, cap)
    s1, s2, cap = 7.0, -3.0, 2.5
    qv = np.array([[[[1.0]]]])
    kv = np.array([[[[s1], [s2]]]])
    vv = np.array([[[[1.0], [0.0]]]])
    o, lse = attention_variant(qv, kv, vv, 1.0, softcap=cap)
    a, b = cap * math.tanh(s1 / cap), cap * math.tanh(s2 / cap)
    assert abs(o[0, 0, 0, 0] - math.exp(a) / (math.exp(a) + math.exp(b))) < 1e-14
    assert abs(lse[0, 0, 0] - math.log(math.exp(a) + math.exp(b))) < 1e-14


def test_alibi_zero_slope_and_equal_keys_closed_form():
    q, k, v = _rand((1, 2, 6, 4), 7), _rand((1, 2, 9, 4), 8), _rand((1, 2, 9, 3), 9)
    np.testing.assert_allclose(attention_variant(q, k, v, 0.5, alibi_slopes=np.zeros(2))[0],
                               attention_variant(q, k, v, 0.5)[0], atol=1e-14)
    # identical keys: every raw score of a row is equal, so the weights are
    # exp(-slope |c - j|) normalised; c = i + (Lk - Lq)
    kk = np.broadcast_to(_rand((4,), 10), (1, 1, 9, 4)).copy()
    vv = _rand((1, 1, 9, 3), 11)
    o, _ = attention_variant(q[:, :1], kk, vv, 0.5, alibi_slopes=np.array([0.4]))
    for i in range(6):
        w = np.exp(-0.4 * np.abs(i + 3 - np.arange(9)))
        np.testing.assert_allclose(o[0, 0, i], (w[:, None] * vv[0, 0]).sum(0) / w.sum(), atol=1e-13)


def test_rows_and_varlen_agree_with_dense():
    q, k, v = _bf16_triple(2, 4, 2, 33, 33, 8, 12)
    full = attention_variant(q, k, v, 0.3, (5, 2), 0.0, np.array([0.1, 0.2, 0.3, 0.4]))
    rows = np.array([0, 32, 33, 100, 263])
    o, l = attention_variant(q, k, v, 0.3, (5, 2), 0.0, np.array([0.1, 0.2, 0.3, 0.4]), rows=rows)
    np.testing.assert_allclose(o, full[0].reshape(-1, 8)[rows], atol=1e-14)
    np.testing.assert_allclose(l, full[1].reshape(-1)[rows], atol=1e-14)
    # varlen of the two batch entries equals the dense batch
    qp = torch.cat([q[0].transpose(0, 1), q[1].transpose(0, 1)])
    kp = torch.cat([k[0].transpose(0, 1), k[1].transpose(0, 1)])
    vp = torch.cat([v[0].transpose(0, 1), v[1].transpose(0, 1)])
    cu = np.array([0, 33, 66])
    ov, lv = attention_variant_varlen(qp, kp, vp, cu, cu, 0.3, (5, 2), 0.0, np.array([0.1, 0.2, 0.3, 0.4]))
    for b in range(2):
        np.testing.assert_allclose(ov[33 * b:33 * (b + 1)].transpose(1, 0, 2), full[0][b], atol=1e-14)
        np.testing.assert_allclose(lv[:, 33 * b:33 * (b + 1)], full[1][b], atol=1e-14)


# ------------------------------------------------------------------ backward

def _torch_variant_grads(q, k, v, do, scale, window, softcap, slopes):
    """PyTorch autograd through an independently written variant forward."""
    Q = torch.tensor(q, requires_grad=True)
    K = torch.tensor(k, requires_grad=True)
    V = torch.tensor(v, requires_grad=True)
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    r = Hq // Hkv
    Kr, Vr = K.repeat_interleave(r, 1), V.repeat_interleave(r, 1)
    S = scale * Q @ Kr.transpose(-1, -2)
    if softcap > 0:
        S = softcap * torch.tanh(S / softcap)
    pos = torch.arange(Lq)[:, None] + (Lk - Lq)
    key = torch.arange(Lk)[None, :]
    if slopes is not None:
        S = S - torch.tensor(slopes)[None, :, None, None] * (pos - key).abs()
    ok = torch.ones(Lq, Lk, dtype=torch.bool)
    if window[0] >= 0:
        ok &= key >= pos - window[0]
    if window[1] >= 0:
        ok &= key <= pos + window[1]
    P = torch.nan_to_num(torch.softmax(S.masked_fill(~ok, float("-inf")), dim=-1), nan=0.0)
    (P @ Vr * torch.tensor(do)).sum().backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("window,softcap,alibi", [((5, 0), 0.0, False), ((3, 4), 0.0, False), ((-1, -1), 2.0, False),
                                                 ((6, 0), 1.5, False), ((-1, -1), 0.0, True), ((4, 2), 0.0, True),
                                                 ((-1, -1), 2.0, True), ((6, 0), 1.5, True)])
@pytest.mark.parametrize("Lq,Lk", [(13, 13), (9, 17), (17, 9)])
def test_variant_backward_matches_autograd(window, softcap, alibi, Lq, Lk):
    from oracle.variants import attention_variant_bwd
    rng = np.random.default_rng(Lq * 7 + Lk)
    B, Hq, Hkv, D = 1, 4, 2, 8
    q = rng.standard_normal((B, Hq, Lq, D))
    k = rng.standard_normal((B, Hkv, Lk, D))
    v = rng.standard_normal((B, Hkv, Lk, D))
    do = rng.standard_normal((B, Hq, Lq, D))
    slopes = np.array([0.5, 0.25, 0.125, 0.0625]) if alibi else None
    got = attention_variant_bwd(q, k, v, do, 0.4, window, softcap, slopes, block=5)
    ref = _torch_variant_grads(q, k, v, do, 0.4, window, softcap, slopes)
    for g, e, n in zip(got, ref, "qkv"):
        np.testing.assert_allclose(g, e, atol=1e-11, rtol=1e-9, err_msg=n)


def test_variant_backward_varlen_equals_dense_per_sequence():
    from oracle.variants import attention_variant_bwd, attention_variant_bwd_varlen
    rng = np.random.default_rng(3)
    lq, lk, H, D = [7, 0, 12], [9, 5, 12], 2, 8
    cq, ck = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q, do = rng.standard_normal((cq[-1], H, D)), rng.standard_normal((cq[-1], H, D))
    k, v = rng.standard_normal((ck[-1], H, D)), rng.standard_normal((ck[-1], H, D))
    dq, dk, dv = attention_variant_bwd_varlen(q, k, v, do, cq, ck, 0.3, (4, 1), 3.0)
    for s in (0, 2):
        sl = lambda t, c, i: t[c[i]:c[i + 1]].transpose(1, 0, 2)[None]
        g = attention_variant_bwd(sl(q, cq, s), sl(k, ck, s), sl(v, ck, s), sl(do, cq, s), 0.3, (4, 1), 3.0)
        assert np.array_equal(dq[cq[s]:cq[s + 1]], g[0][0].transpose(1, 0, 2))
        assert np.array_equal(dk[ck[s]:ck[s + 1]], g[1][0].transpose(1, 0, 2))
    assert np.all(dk[ck[1]:ck[2]] == 0) and np.all(dv[ck[1]:ck[2]] == 0)  # no query rows
