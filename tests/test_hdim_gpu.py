"""GPU parity of the forward with a value head dimension different from the
query/key one: (D, Dv) = (192, 128), the asymmetric case of the
FlashAttention-4 benchmarks (FlashAttention-4: Blackwell Attention Kernel
Co-Design, "How we know").  Compared with the fp64 oracle element by element;
same tolerances as the other forward tests."""
import math

import numpy as np
import pytest
import torch

import exact_attention_07_gb300 as fa
import oracle
from parity import compare
from workloads import random_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
D, DV = 192, 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.load_library()


def run_hdim(q, k, v, causal, scale=None):
    """fa_fwd_hdim with guard bands around O and LSE; checks the guards."""
    B, Hq, Lq, _ = q.shape
    Dv = v.shape[3]
    G = 4096
    n_o = B * Hq * Lq * Dv
    o_buf = torch.full((n_o + 2 * G,), float("nan"), dtype=torch.float32, device=DEV)
    l_buf = torch.full((B * Hq * Lq + 2 * G,), 12345.0, dtype=torch.float32, device=DEV)
    o = o_buf[G:G + n_o].view(B, Hq, Lq, Dv)
    lse = l_buf[G:G + B * Hq * Lq].view(B, Hq, Lq)
    fa.fa_fwd_hdim(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, softmax_scale=scale, out=o, lse=lse)
    fa.fa_check()
    assert torch.isnan(o_buf[:G]).all() and torch.isnan(o_buf[-G:]).all(), "O guard band written"
    assert (l_buf[:G] == 12345.0).all() and (l_buf[-G:] == 12345.0).all(), "LSE guard band written"
    return o.cpu().numpy(), lse.cpu().numpy()


CASES = [
    # B, Hq, Hkv, Lq, Lk, causal, q_mult
    (1, 2, 2, 384, 384, False, 1.0),    # several tiles, half-empty second Q tile
    (1, 2, 2, 384, 384, True, 1.0),
    (2, 3, 3, 300, 300, False, 1.0),    # ragged tail
    (2, 3, 3, 300, 300, True, 1.0),
    (1, 2, 1, 200, 517, True, 1.0),     # Lq < Lk, bottom-right causal
    (1, 2, 1, 517, 200, True, 1.0),     # Lq > Lk: leading rows see no key
    (1, 8, 2, 513, 513, True, 3.0),     # GQA r = 4, sharper softmax
    (1, 2, 2, 1, 1000, False, 1.0),     # one query row, long key range
    (1, 2, 2, 640, 640, False, 20.0),   # very sharp softmax: rescales
    (1, 4, 4, 1500, 1500, False, 1.0),  # 12 KV tiles: the K-tail ring wraps many times
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,causal,qm", CASES)
def test_hdim_192_128_full_compare(B, Hq, Hkv, Lq, Lk, causal, qm):
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=B * 5 + Lq + Lk, q_mult=qm,
                            shape_v=(B, Hkv, Lk, DV))
    o, lse = run_hdim(q, k, v, causal)
    ref_o, ref_lse = oracle.attention(q, k, v, scale=1.0 / math.sqrt(D), causal=causal)
    compare(o, lse, ref_o, ref_lse, f"hdim {B,Hq,Hkv,Lq,Lk,causal,qm}")


def test_hdim_equal_dims_match_fa_fwd():
    # fa_fwd_hdim with Dv = D runs the same kernel as fa_fwd: identical bits
    q, k, v = random_inputs((1, 4, 333, 128), (1, 2, 333, 128), seed=12)
    o1, l1 = fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    o2, l2 = fa.fa_fwd_hdim(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    fa.fa_check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_hdim_varlen_full_compare(causal):
    lq = [1, 127, 128, 129, 300, 5, 700]
    lk = [1, 127, 128, 129, 300, 5, 650] if causal else [9, 200, 128, 1, 300, 64, 700]
    Hq, Hkv = 4, 2
    Tq, Tk = sum(lq), sum(lk)
    q, k, v = random_inputs((Tq, Hq, D), (Tk, Hkv, D), seed=8, shape_v=(Tk, Hkv, DV))
    cq = torch.tensor([0] + np.cumsum(lq).tolist(), dtype=torch.int32)
    ck = torch.tensor([0] + np.cumsum(lk).tolist(), dtype=torch.int32)
    o = torch.full((Tq, Hq, DV), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((Hq, Tq), 12345.0, dtype=torch.float32, device=DEV)
    fa.fa_fwd_varlen_hdim(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV), max(lq), max(lk),
                          causal=causal, out=o, lse=lse)
    fa.fa_check()
    ref_o, ref_lse = oracle.attention_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=1 / math.sqrt(D),
                                             causal=causal)
    compare(o.cpu().numpy().transpose(1, 0, 2), lse.cpu().numpy(), ref_o.transpose(1, 0, 2), ref_lse,
            f"hdim varlen causal={causal}")


def test_hdim_varlen_split_across_launches():
    """(192, 128) launches schedule at most 64 sequences each: 150 sequences
    take three launches, every row compared in full."""
    rng = np.random.default_rng(192)
    n = 150
    lq = rng.integers(0, 300, n).tolist()
    lk = [x + int(rng.integers(0, 50)) for x in lq]
    Hq, Hkv = 2, 1
    Tq, Tk = sum(lq), sum(lk)
    q, k, v = random_inputs((Tq, Hq, D), (Tk, Hkv, D), seed=9, shape_v=(Tk, Hkv, DV))
    cq = torch.tensor([0] + np.cumsum(lq).tolist(), dtype=torch.int32)
    ck = torch.tensor([0] + np.cumsum(lk).tolist(), dtype=torch.int32)
    o = torch.full((Tq, Hq, DV), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((Hq, Tq), 12345.0, dtype=torch.float32, device=DEV)
    fa.fa_fwd_varlen_hdim(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV), max(lq), max(lk),
                          causal=True, out=o, lse=lse)
    assert fa.fa_last_launch_count() == 3
    fa.fa_check()
    ref_o, ref_lse = oracle.attention_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=1 / math.sqrt(D), causal=True)
    compare(o.cpu().numpy().transpose(1, 0, 2), lse.cpu().numpy(), ref_o.transpose(1, 0, 2), ref_lse,
            "hdim varlen split")


def test_hdim_unsupported_pairs_raise():
    q, k, _ = random_inputs((1, 2, 64, 192), (1, 2, 64, 192), seed=1)
    v = torch.zeros((1, 2, 64, 192), dtype=torch.bfloat16)
    with pytest.raises(fa.FAError) as ei:
        fa.fa_fwd_hdim(q.to(DEV), k.to(DEV), v.to(DEV))
    assert ei.value.status == fa.FA_ERR_UNSUPPORTED
