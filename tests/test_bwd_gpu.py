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
    D = 128
    seed = B * 7 + Hq + Lq + 3 * Lk
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
