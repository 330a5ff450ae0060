"""GPU parity of the attention backward (fa_bwd) against the fp64 oracle.

The CUDA path runs fa_fwd, then fa_bwd with the forward's own O and LSE; the
oracle computes the exact gradients of sum(O * dO) from the same bf16 inputs
(oracle/backward.py).  The pages state no tolerance for gradients; the bar
below follows from the arithmetic: P and dS enter the tensor cores rounded to
bf16 (unit roundoff u = 2^-8, relative RMS error about u / sqrt(3) each), so
every gradient carries a relative RMS error of a few 1e-3.  Bar per gradient
tensor: relative RMS <= 1e-2 and max |error| <= 2e-2 * max |reference|.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_07_gb300 as fa
from oracle.backward import attention_bwd
from workloads import grad_output, random_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
REL_RMS = 1e-2
MAX_REL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.load_library()


def run_bwd(q, k, v, do, causal, scale=None):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fa_fwd(qd, kd, vd, causal=causal, softmax_scale=scale)
    dq, dk, dv = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=causal, softmax_scale=scale)
    fa.fa_check()
    assert fa.fa_last_launch_count() == 2
    return dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy()


def compare_grads(got, ref, what):
    floor = 1e-3 * max(np.abs(r).max() for r in ref)  # for gradients that are exactly zero
    for g, r, n in zip(got, ref, ("dq", "dk", "dv")):
        g = np.asarray(g, dtype=np.float64)
        assert g.shape == r.shape, f"{what} {n} shape"
        assert np.isfinite(g).all(), f"{what} {n}: non-finite"
        denom = np.linalg.norm(r)
        err = np.abs(g - r).max() if g.size else 0.0
        if denom <= floor:
            assert err <= floor, f"{what} {n}: |err| {err:.3e} on a zero gradient"
            continue
        rel = np.linalg.norm(g - r) / denom
        assert rel <= REL_RMS, f"{what} {n}: relRMS {rel:.3e}"
        assert err <= MAX_REL * np.abs(r).max(), f"{what} {n}: max err {err:.3e} vs max|ref| {np.abs(r).max():.3e}"


CASES = [
    # B, Hq, Hkv, Lq, Lk, causal, q_mult
    (1, 2, 2, 256, 256, False, 1.0),
    (1, 2, 2, 256, 256, True, 1.0),
    (2, 4, 2, 300, 300, True, 1.0),      # GQA r = 2, ragged tail tile
    (1, 2, 1, 200, 520, True, 1.0),      # Lq < Lk, bottom-right causal
    (1, 2, 1, 520, 200, True, 1.0),      # Lq > Lk: leading rows see no key
    (1, 8, 2, 513, 513, True, 3.0),      # GQA r = 4, sharper softmax
    (1, 2, 2, 1, 1000, False, 1.0),      # one query row
    (1, 1, 1, 1, 1, False, 1.0),         # one key: dQ = dK = 0
    (1, 4, 1, 700, 257, False, 1.0),     # MQA
    (2, 2, 2, 1100, 1100, True, 1.0),
    (1, 2, 2, 640, 640, False, 20.0),    # very sharp softmax
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,causal,qm", CASES)
def test_bwd_full_compare(B, Hq, Hkv, Lq, Lk, causal, qm):
    _bwd_case(B, Hq, Hkv, Lq, Lk, causal, qm, 128)


CASES_D64 = [
    # head dimension 64: dQ formed untransposed (lanes = query rows)
    (1, 2, 2, 256, 256, False, 1.0),
    (2, 4, 2, 300, 300, True, 1.0),
    (1, 2, 1, 200, 520, True, 1.0),
    (1, 2, 1, 520, 200, True, 1.0),
    (1, 8, 2, 513, 513, True, 3.0),
    (1, 1, 1, 1, 1, False, 1.0),
    (4, 4, 4, 1024, 1024, True, 1.0),   # the D = 64 forward workload's shape
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,causal,qm", CASES_D64)
def test_bwd_d64_full_compare(B, Hq, Hkv, Lq, Lk, causal, qm):
    _bwd_case(B, Hq, Hkv, Lq, Lk, causal, qm, 64)


def _bwd_case(B, Hq, Hkv, Lq, Lk, causal, qm, D):
    seed = B * 7 + Hq + Lq + 3 * Lk + D
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=seed, q_mult=qm)
    do = grad_output((B, Hq, Lq, D), seed)
    got = run_bwd(q, k, v, do, causal)
    ref = attention_bwd(q, k, v, do, 1 / math.sqrt(D), causal)
    compare_grads(got, ref, f"bwd {B,Hq,Hkv,Lq,Lk,causal,qm}")


def test_bwd_custom_scale_and_repeat_calls():
    q, k, v = random_inputs((1, 4, 333, 128), (1, 2, 333, 128), seed=77)
    do = grad_output((1, 4, 333, 128), 77)
    a = run_bwd(q, k, v, do, True, scale=0.05)
    b = run_bwd(q, k, v, do, True, scale=0.05)
    # dK and dV come out of tensor memory in a fixed order: bit-identical;
    # dQ is summed with atomics in arrival order
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert np.abs(a[0] - b[0]).max() <= 1e-4 * np.abs(a[0]).max()
    ref = attention_bwd(q, k, v, do, 0.05, True)
    compare_grads(a, ref, "scale 0.05")


def test_bwd_timed_out_wait_is_reported_and_context_survives():
    q, k, v = random_inputs((1, 2, 256, 128), (1, 2, 256, 128), seed=5)
    do = grad_output((1, 2, 256, 128), 5)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fa_fwd(qd, kd, vd, causal=False)
    fa.fa_check()
    fa.load_library().fa_test_inject_fault(1)
    fa.fa_bwd(qd, kd, vd, o, lse, dod)
    with pytest.raises(fa.FAError) as ei:
        fa.fa_check()
    assert ei.value.status == fa.FA_ERR_TIMEOUT
    got = run_bwd(q, k, v, do, False)
    compare_grads(got, attention_bwd(q, k, v, do, 1 / math.sqrt(128), False), "after timeout")


# ------------------------------------------------------------------ packed batches

VARLEN_CASES = [
    # query lengths, key lengths, Hq, Hkv, causal
    ([1, 127, 128, 129, 300, 5], [1, 127, 128, 129, 300, 5], 4, 2, True),
    ([1, 127, 128, 129, 300, 5], [1, 127, 128, 129, 300, 5], 4, 2, False),
    ([50, 700, 3, 256], [90, 650, 3, 300], 4, 4, True),      # Lq != Lk per sequence
    ([200, 0, 100, 64], [200, 40, 0, 64], 2, 1, True),       # no query rows / no keys
    ([513, 7, 1024], [513, 7, 1024], 8, 2, False),
]


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("lq,lk,Hq,Hkv,causal", VARLEN_CASES)
def test_bwd_varlen_full_compare(lq, lk, Hq, Hkv, causal, D):
    from oracle.backward import attention_bwd_varlen
    Tq, Tk = sum(lq), sum(lk)
    seed = Tq + 3 * Tk + Hq
    q, k, v = random_inputs((Tq, Hq, D), (Tk, Hkv, D), seed=seed)
    do = grad_output((Tq, Hq, D), seed)
    cq = torch.tensor([0] + np.cumsum(lq).tolist(), dtype=torch.int32, device=DEV)
    ck = torch.tensor([0] + np.cumsum(lk).tolist(), dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fa_fwd_varlen(qd, kd, vd, cq, ck, max(lq), max(max(lk), 1), causal=causal)
    # outputs start as NaN: every element must be written
    dq = torch.full((Tq, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    dk = torch.full((Tk, Hkv, D), float("nan"), dtype=torch.float32, device=DEV)
    dv = torch.full((Tk, Hkv, D), float("nan"), dtype=torch.float32, device=DEV)
    fa.fa_bwd_varlen(qd, kd, vd, o, lse, dod, cq, ck, max(lq), max(max(lk), 1), causal=causal,
                     dq=dq, dk=dk, dv=dv)
    fa.fa_check()
    assert fa.fa_last_launch_count() == 3
    ref = attention_bwd_varlen(q, k, v, do, cq.cpu().numpy(), ck.cpu().numpy(), 1 / math.sqrt(D), causal)
    compare_grads((dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy()), ref, f"varlen bwd {lq} {lk}")


def test_bwd_varlen_single_sequence_equals_dense():
    # one packed sequence is the dense problem with B = 1 (layouts transposed)
    Hq, Hkv, L, D = 4, 2, 333, 128
    q, k, v = random_inputs((1, Hq, L, D), (1, Hkv, L, D), seed=21)
    do = grad_output((1, Hq, L, D), 21)
    a = run_bwd(q, k, v, do, True)
    pk = [t[0].permute(1, 0, 2).contiguous().to(DEV) for t in (q, k, v, do)]
    cu = torch.tensor([0, L], dtype=torch.int32, device=DEV)
    o, lse = fa.fa_fwd_varlen(pk[0], pk[1], pk[2], cu, cu, L, L, causal=True)
    dq, dk, dv = fa.fa_bwd_varlen(pk[0], pk[1], pk[2], o, lse, pk[3], cu, cu, L, L, causal=True)
    fa.fa_check()
    # dK and dV have the same summation order in both layouts: bit-identical
    assert np.array_equal(dk.cpu().numpy(), a[1][0].transpose(1, 0, 2))
    assert np.array_equal(dv.cpu().numpy(), a[2][0].transpose(1, 0, 2))
    assert np.abs(dq.cpu().numpy() - a[0][0].transpose(1, 0, 2)).max() <= 1e-4 * np.abs(a[0]).max()


# ------------------------------------------------------------------ variants (windows, soft-capping, ALiBi)

BWD_VARIANT_CASES = [
    # B, Hq, Hkv, Lq, Lk, window, cap, alibi, Q multiplier
    (1, 2, 2, 384, 384, (127, 0), 0.0, False, 1.0),     # causal window of width 128
    (1, 2, 1, 513, 513, (300, 0), 0.0, False, 1.0),     # window edge inside tiles, GQA
    (1, 2, 2, 300, 700, (200, 50), 0.0, False, 1.0),    # two-sided, Lq < Lk
    (1, 2, 2, 700, 300, (64, 64), 0.0, False, 1.0),     # Lq > Lk: rows without keys
    (1, 2, 2, 256, 256, (-1, 0), 0.0, False, 1.0),      # plain causal as a window
    (2, 4, 2, 333, 333, (-1, -1), 0.0, True, 1.0),      # ALiBi, full
    (1, 4, 4, 400, 400, (255, 0), 0.0, True, 1.0),      # ALiBi inside a causal window
    (1, 2, 2, 384, 384, (-1, -1), 5.0, False, 4.0),     # soft cap 5, scores ~ N(0, 16): tanh saturates
    (1, 4, 2, 333, 517, (-1, 0), 30.0, False, 6.0),     # soft cap 30, causal, GQA, ragged, Lq < Lk
    (2, 2, 2, 300, 300, (100, 20), 2.0, False, 3.0),    # soft cap 2 inside a two-sided window
    (2, 4, 2, 400, 400, (-1, -1), 4.0, True, 3.0),     # soft-capping, then ALiBi
    (1, 4, 4, 333, 517, (-1, 0), 6.0, True, 4.0),       # both modifiers, causal, ragged, Lq < Lk
]


BWD_VARIANT_CASES_D64 = [
    (1, 2, 1, 513, 513, (300, 0), 0.0, False, 1.0),     # window edge inside tiles, GQA
    (1, 4, 2, 333, 517, (-1, 0), 30.0, False, 6.0),     # soft cap 30, causal, GQA, ragged, Lq < Lk
    (1, 4, 4, 400, 400, (255, 0), 0.0, True, 1.0),      # ALiBi inside a causal window
    (1, 4, 2, 400, 400, (-1, 0), 4.0, True, 3.0),       # soft-capping, then ALiBi, causal
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,window,cap,alibi,qm,D",
                         [c + (128,) for c in BWD_VARIANT_CASES] + [c + (64,) for c in BWD_VARIANT_CASES_D64])
def test_bwd_variant_full_compare(B, Hq, Hkv, Lq, Lk, window, cap, alibi, qm, D):
    from oracle.variants import attention_variant_bwd
    seed = Lq + 2 * Lk + Hq + (7 if alibi else 0) + int(cap)
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=seed, q_mult=qm)
    do = grad_output((B, Hq, Lq, D), seed)
    slopes = torch.tensor([2.0 ** (-(h + 1)) for h in range(Hq)], dtype=torch.float32) if alibi else None
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    sd = slopes.to(DEV) if alibi else None
    o, lse = fa.fa_fwd_variant(qd, kd, vd, window=window, softcap=cap, alibi_slopes=sd)
    dq = torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
    dk = torch.full(k.shape, float("nan"), dtype=torch.float32, device=DEV)
    dv = torch.full(k.shape, float("nan"), dtype=torch.float32, device=DEV)
    fa.fa_bwd_variant(qd, kd, vd, o, lse, dod, window=window, softcap=cap, alibi_slopes=sd, dq=dq, dk=dk, dv=dv)
    fa.fa_check()
    ref = attention_variant_bwd(q, k, v, do, 1 / math.sqrt(D), window, cap,
                                slopes.numpy() if alibi else None)
    compare_grads((dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy()), ref,
                  f"bwd variant {window} cap {cap} alibi {alibi}")


def test_bwd_causal_window_equals_causal():
    # window (-1, 0) is the causal mask: same gradients as the causal kernel
    q, k, v = random_inputs((1, 4, 300, 128), (1, 2, 300, 128), seed=44)
    do = grad_output((1, 4, 300, 128), 44)
    a = run_bwd(q, k, v, do, True)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fa_fwd_variant(qd, kd, vd, window=(-1, 0))
    b = fa.fa_bwd_variant(qd, kd, vd, o, lse, dod, window=(-1, 0))
    fa.fa_check()
    assert np.array_equal(b[1].cpu().numpy(), a[1]) and np.array_equal(b[2].cpu().numpy(), a[2])
    assert np.abs(b[0].cpu().numpy() - a[0]).max() <= 1e-4 * np.abs(a[0]).max()


@pytest.mark.parametrize("window,cap,qm,D", [((100, 0), 0.0, 1.0, 128), ((-1, 0), 8.0, 4.0, 128),
                                             ((100, 0), 0.0, 1.0, 64)])
def test_bwd_varlen_variant_full_compare(window, cap, qm, D):
    from oracle.variants import attention_variant_bwd_varlen
    lq, lk, Hq, Hkv = [200, 5, 400, 129], [260, 5, 400, 129], 4, 2
    Tq, Tk = sum(lq), sum(lk)
    q, k, v = random_inputs((Tq, Hq, D), (Tk, Hkv, D), seed=61, q_mult=qm)
    do = grad_output((Tq, Hq, D), 61)
    cq = torch.tensor([0] + np.cumsum(lq).tolist(), dtype=torch.int32, device=DEV)
    ck = torch.tensor([0] + np.cumsum(lk).tolist(), dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fa_fwd_varlen_variant(qd, kd, vd, cq, ck, max(lq), max(lk), window=window, softcap=cap)
    dq, dk, dv = fa.fa_bwd_varlen_variant(qd, kd, vd, o, lse, dod, cq, ck, max(lq), max(lk), window=window,
                                          softcap=cap)
    fa.fa_check()
    ref = attention_variant_bwd_varlen(q, k, v, do, cq.cpu().numpy(), ck.cpu().numpy(), 1 / math.sqrt(D), window,
                                       cap)
    compare_grads((dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy()), ref, f"varlen bwd window cap {cap}")
