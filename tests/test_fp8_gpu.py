"""GPU parity of the FP8 forward (fa_fp8_prepare + fa_fwd_fp8) against the
FP8 oracle (oracle/fp8.py).

Tolerance, derived (the pages give none for FP8): beyond the quantised
inputs, the kernel rounds P to e4m3 (3 mantissa bits, relative step 2^-3)
for the P.V product.  Simulating exactly that rounding on N(0,1) inputs of
512-2048 keys gives O a relative RMS error of 2.2-2.6e-2 and a max error of
2-3 % of max|O|.  Bar against the oracle of the quantised inputs: O relative
RMS <= 5e-2, O max |error| <= 5e-2 * max(1, max|O|), LSE max |error| <=
5e-3 (the LSE is summed from unrounded p).  Codes are compared element by
element: the device rounds its fp32 rotation, the oracle its fp64 rotation,
so a code may differ by one e4m3 step where the value sits on a rounding
boundary; anything else must agree.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_07_gb300 as fa
import oracle
from oracle.fp8 import attention_fp8_inputs, prepare
from workloads import WORKLOADS, dense_inputs, fp8_signs, random_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.load_library()


def _section(buf, sec, name, dtype):
    off, nbytes, shape = sec[name]
    raw = buf[off:off + nbytes].cpu()
    if dtype == "e4m3":
        return raw.view(torch.float8_e4m3fn).float().numpy().reshape(shape)
    return raw.view(torch.float32).numpy().reshape(shape)


def _e4m3_neighbours(x):
    """The e4m3 values adjacent to each value of x (as float64)."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    vals = np.unique(codes[np.isfinite(codes)])
    idx = np.searchsorted(vals, x)
    lo = vals[np.clip(idx - 1, 0, len(vals) - 1)]
    hi = vals[np.clip(idx + 1, 0, len(vals) - 1)]
    return lo, hi


def run_fp8(q, k, v, causal, signs):
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    buf = fa.fp8_prepare(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(signs).float().to(DEV))
    o, lse = fa.fa_fwd_fp8(buf, B, Hq, Hkv, Lq, Lk, causal=causal)
    fa.fa_check()
    return buf, o.cpu().numpy(), lse.cpu().numpy()


def check_codes(buf, q, k, v, signs):
    B, Hq, Lq, _ = q.shape
    _, Hkv, Lk, _ = k.shape
    sec = fa.fp8_sections(B, Hq, Hkv, Lq, Lk)
    ref = prepare(q, k, v, signs)
    for name, rname in (("sq", "sq"), ("sk", "sk"), ("sv", "sv")):
        np.testing.assert_allclose(_section(buf, sec, name, "f32"), ref[rname], rtol=2e-6, err_msg=name)
    vt = _section(buf, sec, "vt", "e4m3")
    got = {"qc": _section(buf, sec, "qc", "e4m3"), "kc": _section(buf, sec, "kc", "e4m3"),
           "vc": vt[..., :Lk].transpose(0, 1, 3, 2)}
    assert np.all(vt[..., Lk:] == 0)  # padding keys
    for name in ("qc", "kc", "vc"):
        g, r = got[name], ref[name]
        diff = g != r
        frac = diff.mean()
        assert frac < 5e-3, f"{name}: {frac:.2e} of the codes differ"
        lo, hi = _e4m3_neighbours(r[diff])
        assert np.all((g[diff] == lo) | (g[diff] == hi)), f"{name}: a code differs by more than one step"
    return ref


def compare_fp8(o, lse, ref_o, ref_lse, what):
    empty = ~np.isfinite(ref_lse)
    assert np.array_equal(~np.isfinite(lse), empty), what
    assert np.all(o[empty] == 0)
    rel = np.linalg.norm(o - ref_o) / np.linalg.norm(ref_o)
    err = np.abs(o - ref_o).max()
    lerr = np.abs(lse[~empty] - ref_lse[~empty]).max() if (~empty).any() else 0.0
    assert rel <= 5e-2, f"{what}: relRMS {rel:.3e}"
    assert err <= 5e-2 * max(1.0, np.abs(ref_o).max()), f"{what}: max err {err:.3e}"
    assert lerr <= 5e-3, f"{what}: LSE err {lerr:.3e}"
    return rel


CASES = [
    # B, Hq, Hkv, Lq, Lk, causal, q_mult
    (1, 2, 2, 256, 256, False, 1.0),
    (1, 2, 2, 384, 384, True, 1.0),
    (2, 4, 2, 300, 300, True, 1.0),     # GQA, ragged tail tiles
    (1, 2, 1, 200, 520, True, 1.0),     # Lq < Lk
    (1, 2, 1, 520, 200, True, 1.0),     # Lq > Lk: leading rows see no key
    (1, 8, 2, 513, 513, True, 3.0),     # sharper softmax
    (1, 2, 2, 1, 700, False, 1.0),      # one query row
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,causal,qm", CASES)
def test_fp8_against_quantised_input_oracle(B, Hq, Hkv, Lq, Lk, causal, qm):
    D = 128
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=Lq + 3 * Lk + Hq, q_mult=qm)
    signs = fp8_signs(D, seed=Lq)
    buf, o, lse = run_fp8(q, k, v, causal, signs)
    ref = check_codes(buf, q, k, v, signs)
    ref_o, ref_lse = attention_fp8_inputs(ref, 1 / math.sqrt(D), causal)
    compare_fp8(o, lse, ref_o, ref_lse, f"fp8 {B,Hq,Hkv,Lq,Lk,causal,qm}")
    # and the distance to the exact bf16 attention stays within the FP8 budget
    ex_o, _ = oracle.attention(q, k, v, scale=1 / math.sqrt(D), causal=causal)
    assert np.linalg.norm(o - ex_o) / np.linalg.norm(ex_o) < 8e-2


def test_fp8_outlier_channels():
    """Inputs with a few 30x outlier channels in Q and K: the device result is
    as close to exact attention as the oracle's FP8 simulation (which, with
    the rotation, beats per-tile quantisation without it: oracle pins)."""
    D = 128
    q, k, v = random_inputs((1, 2, 512, D), (1, 2, 512, D), seed=21)
    q, k = q.float(), k.float()
    q[..., :4] *= 30.0
    k[..., :4] *= 30.0
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    signs = fp8_signs(D, seed=9)
    scale = 1 / (30 * math.sqrt(D))
    buf = fa.fp8_prepare(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(signs).float().to(DEV))
    o, lse = fa.fa_fwd_fp8(buf, 1, 2, 2, 512, 512, softmax_scale=scale)
    fa.fa_check()
    ex_o, _ = oracle.attention(q, k, v, scale=scale)
    sim_o, _ = attention_fp8_inputs(prepare(q, k, v, signs), scale)
    dev_err = np.sqrt(np.mean((o.cpu().numpy() - ex_o) ** 2))
    sim_err = np.sqrt(np.mean((sim_o - ex_o) ** 2))
    assert dev_err <= 2.0 * sim_err + 1e-4, (dev_err, sim_err)


def test_fp8_timed_out_wait_is_reported():
    q, k, v = random_inputs((1, 2, 256, 128), (1, 2, 256, 128), seed=2)
    signs = fp8_signs(128, seed=1)
    buf = fa.fp8_prepare(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(signs).float().to(DEV))
    fa.fa_check()
    fa.load_library().fa_test_inject_fault(1)
    fa.fa_fwd_fp8(buf, 1, 2, 2, 256, 256)
    with pytest.raises(fa.FAError) as ei:
        fa.fa_check()
    assert ei.value.status == fa.FA_ERR_TIMEOUT


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if w.fp8])
def test_fp8_workload_sampled(name):
    w = WORKLOADS[name]
    q, k, v = dense_inputs(w)
    signs = fp8_signs(w.D, seed=w.seed)
    buf = fa.fp8_prepare(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(signs).float().to(DEV))
    o, lse = fa.fa_fwd_fp8(buf, w.B, w.Hq, w.Hkv, w.Lq, w.Lk, causal=w.causal)
    fa.fa_check()
    rows = np.unique(np.concatenate([[0, w.B * w.Hq * w.Lq - 1],
                                     np.random.default_rng(4).integers(0, w.B * w.Hq * w.Lq, 200)]))
    ref = prepare(q, k, v, signs)
    ref_o, ref_lse = attention_fp8_inputs(ref, w.scale, w.causal, rows=rows)
    idx = torch.from_numpy(rows).to(DEV)
    compare_fp8(o.reshape(-1, w.D)[idx].cpu().numpy(), lse.reshape(-1)[idx].cpu().numpy(), ref_o, ref_lse, name)
