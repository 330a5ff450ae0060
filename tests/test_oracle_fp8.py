"""Pins of the FP8 oracle (oracle/fp8.py): the rotation is orthogonal and
leaves scores unchanged, e4m3 rounding hits known values, the quantisation
error stays within the format's bound, scales follow the definition, and
incoherent processing lowers the error on inputs with outlier features
(FlashAttention from Scratch, sec. 10.3; FlashAttention 1-4, FA3 item 3)."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.fp8 import (E4M3_MAX, attention_fp8_inputs, dequantize, hadamard, prepare, rotation, round_e4m3)


def _signs(d, seed):
    return np.where(np.random.default_rng(seed).random(d) < 0.5, -1.0, 1.0)


def test_hadamard_and_rotation_are_orthogonal():
    for d in (2, 8, 64, 128):
        h = hadamard(d)
        assert set(np.unique(h)) == {-1.0, 1.0}
        np.testing.assert_allclose(h @ h.T, d * np.eye(d), atol=0)
        m = rotation(_signs(d, d))
        np.testing.assert_allclose(m @ m.T, np.eye(d), atol=1e-14)
    # Sylvester recursion: H_4 from H_2
    h2 = np.array([[1, 1], [1, -1]], dtype=float)
    np.testing.assert_array_equal(hadamard(4), np.kron(h2, h2))


def test_rotation_leaves_scores_unchanged():
    q, k = np.random.default_rng(1).standard_normal((9, 128)), np.random.default_rng(2).standard_normal((7, 128))
    m = rotation(_signs(128, 3))
    np.testing.assert_allclose((q @ m) @ (k @ m).T, q @ k.T, atol=1e-12)


def test_e4m3_known_values():
    x = np.array([0.0, 1.0, -1.0, 448.0, 0.1, 2.0 ** -9, 2.0 ** -6, 1.0625, 1.1875, 300.0, 17.0])
    expect = np.array([0.0, 1.0, -1.0, 448.0, 0.1015625, 2.0 ** -9, 2.0 ** -6, 1.0, 1.25, 288.0, 16.0])
    np.testing.assert_array_equal(round_e4m3(x), expect)


def test_quantisation_error_bound_and_scales():
    g = torch.Generator().manual_seed(0)
    q = torch.randn((2, 3, 300, 128), generator=g).to(torch.bfloat16)
    k = torch.randn((2, 1, 200, 128), generator=g).to(torch.bfloat16)
    v = torch.randn((2, 1, 200, 128), generator=g).to(torch.bfloat16)
    prep = prepare(q, k, v, _signs(128, 5))
    assert prep["sq"].shape == (2, 3, 3) and prep["sk"].shape == (2, 1, 2) and prep["sv"].shape == (2, 1)
    qr = q.double().numpy() @ rotation(_signs(128, 5))
    # scale = amax / 448 per 128-row tile; codes within [-448, 448]
    np.testing.assert_allclose(prep["sq"][1, 2, 0], np.abs(qr[1, 2, :128]).max() / E4M3_MAX, rtol=1e-15)
    np.testing.assert_allclose(prep["sq"][0, 0, 2], np.abs(qr[0, 0, 256:]).max() / E4M3_MAX, rtol=1e-15)
    assert np.abs(prep["qc"]).max() <= E4M3_MAX
    dq, dk, dv = dequantize(prep)
    # e4m3: 3 mantissa bits (relative step 2^-3, rounding error <= 2^-4) above
    # 2^-6, absolute step 2^-9 (error <= 2^-10) below, in units of the scale
    sc = np.repeat(prep["sq"], 128, axis=2)[:, :, :300, None]
    bound = np.maximum(2.0 ** -4 * np.abs(qr), 2.0 ** -10 * sc) * (1 + 1e-12)
    assert np.all(np.abs(dq - qr) <= bound)
    assert np.all(np.abs(dv - v.double().numpy()) <= np.maximum(2.0 ** -4 * np.abs(v.double().numpy()),
                                                                2.0 ** -10 * prep["sv"][:, :, None, None]) * (1 + 1e-12))


def test_fp8_inputs_attention_close_to_exact_and_rotation_helps_on_outliers():
    """Exact attention of the dequantised inputs is close to exact attention;
    with outlier feature channels, incoherent processing lowers the error (the
    pages report 2.6x lower RMSE on such inputs)."""
    g = torch.Generator().manual_seed(1)
    B, H, L, D = 1, 2, 256, 128
    q = torch.randn((B, H, L, D), generator=g)
    k = torch.randn((B, H, L, D), generator=g)
    v = torch.randn((B, H, L, D), generator=g)
    scale = 1 / math.sqrt(D)
    ref_o, _ = oracle.attention(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), scale=scale)
    prep = prepare(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), _signs(D, 7))
    o, _ = attention_fp8_inputs(prep, scale)
    rel = np.linalg.norm(o - ref_o) / np.linalg.norm(ref_o)
    assert rel < 0.05
    # outliers: a few channels 30x larger in Q and K
    q2, k2 = q.clone(), k.clone()
    q2[..., :4] *= 30.0
    k2[..., :4] *= 30.0
    q2, k2, vb = q2.to(torch.bfloat16), k2.to(torch.bfloat16), v.to(torch.bfloat16)
    ref2, _ = oracle.attention(q2, k2, vb, scale=scale / 30)
    err = {}
    for rot in (True, False):
        pr = prepare(q2, k2, vb, _signs(D, 7), rotate=rot)
        o2, _ = attention_fp8_inputs(pr, scale / 30)
        err[rot] = np.sqrt(np.mean((o2 - ref2) ** 2))
    assert err[True] < 0.7 * err[False], err
