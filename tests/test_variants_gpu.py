"""GPU parity of the programmable forward variants (key windows, soft-capping,
ALiBi) against the fp64 variant oracle (FlashAttention from Scratch, sec. 12).
Same tolerance as the plain forward."""
import math

import numpy as np
import pytest
import torch

import exact_attention_07_gb300 as fa
import oracle
from oracle.variants import attention_variant, attention_variant_varlen
from parity import compare
from workloads import WORKLOADS, dense_inputs, random_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.load_library()


def alibi(H):
    """Geometric slopes, the usual ALiBi choice: 2^(-8 (h+1) / H)."""
    return np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=np.float32)


CASES = [
    # B, Hq, Hkv, Lq, Lk, window, softcap, alibi, q_mult
    (1, 2, 2, 384, 384, (-1, 0), 0.0, False, 1.0),       # the causal mask as a window
    (1, 2, 2, 700, 700, (127, 0), 0.0, False, 1.0),      # causal sliding window of width 128
    (2, 4, 2, 1000, 1000, (300, 0), 0.0, False, 1.0),    # width 301, GQA, ragged
    (1, 2, 1, 300, 900, (64, 64), 0.0, False, 1.0),      # two-sided window, Lq < Lk
    (1, 2, 1, 900, 300, (100, 5), 0.0, False, 1.0),      # Lq > Lk: leading rows see nothing
    (1, 2, 2, 513, 513, (0, 0), 0.0, False, 1.0),        # only the aligned key
    (1, 2, 2, 640, 640, (-1, -1), 30.0, False, 3.0),     # soft-capping, full attention
    (1, 4, 2, 777, 777, (-1, 0), 5.0, False, 4.0),       # tight cap, causal, GQA
    (1, 4, 4, 600, 600, (-1, -1), 0.0, True, 1.0),       # ALiBi, full attention
    (2, 8, 2, 529, 529, (255, 0), 0.0, True, 1.0),       # ALiBi with a causal window, GQA
    (2, 4, 2, 600, 600, (-1, -1), 5.0, True, 4.0),       # soft-capping, then ALiBi, full attention
    (1, 4, 4, 777, 777, (300, 0), 8.0, True, 3.0),       # both modifiers inside a causal window
]


CASES_D64 = [
    (1, 2, 2, 700, 700, (127, 0), 0.0, False, 1.0),      # causal sliding window of width 128
    (1, 2, 1, 300, 900, (64, 64), 0.0, False, 1.0),      # two-sided window, Lq < Lk
    (1, 4, 2, 777, 777, (-1, 0), 5.0, False, 4.0),       # tight cap, causal, GQA
    (2, 8, 2, 529, 529, (255, 0), 0.0, True, 1.0),       # ALiBi with a causal window, GQA
    (1, 4, 2, 600, 600, (-1, 0), 5.0, True, 4.0),        # soft-capping, then ALiBi, causal
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,window,cap,use_alibi,qm,D",
                         [c + (128,) for c in CASES] + [c + (64,) for c in CASES_D64])
def test_variant_full_compare(B, Hq, Hkv, Lq, Lk, window, cap, use_alibi, qm, D):
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=Lq + Lk + Hq, q_mult=qm)
    slopes = alibi(Hq) if use_alibi else None
    o, lse = fa.fa_fwd_variant(q.to(DEV), k.to(DEV), v.to(DEV), window=window, softcap=cap,
                               alibi_slopes=torch.from_numpy(slopes).to(DEV) if use_alibi else None)
    fa.fa_check()
    ref_o, ref_lse = attention_variant(q, k, v, 1 / math.sqrt(D), window, cap, slopes)
    compare(o.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, f"variant {window} cap={cap} alibi={use_alibi}")


@pytest.mark.parametrize("D", [64, 128])
def test_causal_window_equals_plain_causal_kernel(D):
    q, k, v = random_inputs((1, 4, 1000, D), (1, 4, 1000, D), seed=3)
    a = fa.fa_fwd_variant(q.to(DEV), k.to(DEV), v.to(DEV), window=(-1, 0))
    b = fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    fa.fa_check()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("D", [64, 128])
def test_varlen_variant(D):
    lens_q, lens_k = [300, 1, 700, 129], [300, 50, 700, 400]
    Hq, Hkv = 4, 2
    q, k, v = random_inputs((sum(lens_q), Hq, D), (sum(lens_k), Hkv, D), seed=11)
    cq = torch.tensor([0] + np.cumsum(lens_q).tolist(), dtype=torch.int32)
    ck = torch.tensor([0] + np.cumsum(lens_k).tolist(), dtype=torch.int32)
    slopes = alibi(Hq)
    for window, cap, sl in (((127, 0), 0.0, None), ((-1, 0), 10.0, None), ((200, 3), 0.0, slopes),
                            ((-1, 0), 6.0, slopes)):
        o, lse = fa.fa_fwd_varlen_variant(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV), max(lens_q),
                                          max(lens_k), window=window, softcap=cap,
                                          alibi_slopes=torch.from_numpy(sl).to(DEV) if sl is not None else None)
        fa.fa_check()
        ref_o, ref_lse = attention_variant_varlen(q, k, v, cq.numpy(), ck.numpy(), 1 / math.sqrt(D), window, cap, sl)
        compare(o.cpu().numpy().transpose(1, 0, 2), lse.cpu().numpy(), ref_o.transpose(1, 0, 2), ref_lse,
                f"varlen variant {window} {cap}")


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if w.window is not None])
def test_variant_workload_sampled(name):
    w = WORKLOADS[name]
    q, k, v = dense_inputs(w)
    o, lse = fa.fa_fwd_variant(q.to(DEV), k.to(DEV), v.to(DEV), window=w.window)
    fa.fa_check()
    n_total = w.B * w.Hq * w.Lq
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 4095, 4096, 4097, n_total - 1], rng.integers(0, n_total, 300)]))
    ref_o, ref_lse = attention_variant(q, k, v, w.scale, w.window, rows=rows)
    idx = torch.from_numpy(rows).to(DEV)
    compare(o.reshape(-1, w.D)[idx].cpu().numpy(), lse.reshape(-1)[idx].cpu().numpy(), ref_o, ref_lse, name)
