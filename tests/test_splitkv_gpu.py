"""GPU parity of the split-KV (decode) forward against the fp64 oracle.

The split-KV path computes the same attention as the dense forward: each
(batch, KV head) key range is cut into partitions, every partition yields a
normalised partial output and its log-sum-exp, and a merge kernel combines
them (FlashAttention from Scratch, sec. 9.1 and sec. 4.3).  Whatever the
partition count, the result must equal the plain definition, so every case
here is compared element by element with the oracle, which knows nothing of
partitions.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_07_gb300 as fa
import oracle
from parity import compare
from workloads import WORKLOADS, dense_inputs, random_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.load_library()


def run_splitkv(q, k, v, causal, num_splits=0, scale=None):
    """fa_fwd_splitkv with guard bands around O and LSE; checks the guards."""
    B, Hq, Lq, D = q.shape
    G = 4096
    o_buf = torch.full((B * Hq * Lq * D + 2 * G,), float("nan"), dtype=torch.float32, device=DEV)
    l_buf = torch.full((B * Hq * Lq + 2 * G,), 12345.0, dtype=torch.float32, device=DEV)
    o = o_buf[G:G + B * Hq * Lq * D].view(B, Hq, Lq, D)
    lse = l_buf[G:G + B * Hq * Lq].view(B, Hq, Lq)
    fa.fa_fwd_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, softmax_scale=scale, num_splits=num_splits,
                      out=o, lse=lse)
    fa.fa_check()
    assert torch.isnan(o_buf[:G]).all() and torch.isnan(o_buf[-G:]).all(), "O guard band written"
    assert (l_buf[:G] == 12345.0).all() and (l_buf[-G:] == 12345.0).all(), "LSE guard band written"
    return o.cpu().numpy(), lse.cpu().numpy()


CASES = [
    # B, Hq, Hkv, Lq, Lk, D, causal, num_splits, q_mult
    (2, 32, 8, 1, 4096, 128, False, 0, 1.0),    # GQA r = 4 single-token decode, automatic partitions
    (2, 32, 8, 1, 4100, 128, True, 0, 1.0),     # ragged last tile
    (1, 8, 8, 1, 1000, 64, False, 3, 1.0),      # MHA: one row per KV head
    (3, 16, 1, 1, 777, 128, False, 5, 1.0),     # MQA: 16 rows share the only KV head
    (2, 8, 2, 4, 1500, 128, True, 7, 1.0),      # 4 new tokens per head (speculative decode), causal
    (1, 8, 2, 4, 1500, 64, True, 0, 1.0),       # same at D = 64
    (1, 4, 2, 3, 2, 64, True, 0, 1.0),          # Lq > Lk: the first row sees no key
    (1, 2, 1, 1, 1, 128, False, 0, 1.0),        # a single key
    (1, 4, 4, 2, 3200, 64, True, 50, 1.0),      # one tile per partition
    (1, 4, 2, 1, 640, 128, False, 1000, 1.0),   # more partitions asked than tiles: reduced
    (2, 16, 4, 1, 2048, 128, False, 4, 20.0),   # very sharp softmax
    (1, 6, 2, 2, 3000, 128, True, 6, 1.0),      # 6 rows: padded row slots in the kernel
    (1, 12, 4, 1, 999, 64, False, 2, 1.0),      # 3 rows at D = 64
    (2, 32, 8, 1, 4100, 64, True, 0, 1.0),      # GQA r = 4 at D = 64 on the tensor cores, ragged last tile
    (1, 16, 1, 1, 3000, 64, False, 5, 20.0),    # MQA, 16 rows, sharp softmax, D = 64
    (4, 8, 8, 1, 65, 128, True, 1, 1.0),        # one partition: no merge launch
    (1, 16, 2, 1, 2500, 64, True, 0, 1.0),      # 8 rows: the softmax carries exactly 8
    (1, 10, 2, 1, 1999, 128, False, 3, 1.0),    # 5 rows in the 8-row softmax
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,D,causal,splits,qm", CASES)
def test_splitkv_full_compare(B, Hq, Hkv, Lq, Lk, D, causal, splits, qm):
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=B + Hq + Lq * 3 + Lk + D, q_mult=qm)
    o, lse = run_splitkv(q, k, v, causal, splits)
    _, used = fa.splitkv_workspace(B, Hq, Hkv, Lq, Lk, D, splits)
    assert fa.fa_last_launch_count() == (2 if used > 1 else 1)
    assert 1 <= used <= math.ceil(Lk / 64)  # partitions hold whole tiles (64 or 128 keys)
    ref_o, ref_lse = oracle.attention(q, k, v, scale=1 / math.sqrt(D), causal=causal)
    compare(o, lse, ref_o, ref_lse, f"splitkv {B,Hq,Hkv,Lq,Lk,D,causal,splits,qm}")
    if (Hq // Hkv) * Lq == 1:
        # one row per KV head runs the FP32-pipe kernel, which keeps P in fp32:
        # far inside the bf16-P tolerance
        fin = np.isfinite(ref_lse)
        assert np.abs(o - ref_o).max() <= 1e-3
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-4 if fin.any() else True


def test_partition_count_does_not_change_the_result_beyond_rounding():
    B, Hq, Hkv, Lq, Lk, D = 1, 16, 4, 1, 5000, 128
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=31)
    ref_o, ref_lse = oracle.attention(q, k, v, scale=1 / math.sqrt(D), causal=False)
    outs = []
    for splits in (1, 2, 3, 8, 79, 0):
        o, lse = run_splitkv(q, k, v, False, splits)
        compare(o, lse, ref_o, ref_lse, f"splits={splits}")
        outs.append(o)
    # P is rounded to bf16 against each partition's own running reference, so
    # partition counts differ by bf16 rounding of P (about 2^-9 relative)
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-3


def test_custom_scale_and_repeat_calls_identical():
    q, k, v = random_inputs((2, 8, 2, 128), (2, 2, 2500, 128), seed=8)
    o1, l1 = run_splitkv(q, k, v, True, 0, scale=0.03)
    o2, l2 = run_splitkv(q, k, v, True, 0, scale=0.03)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ref_o, ref_lse = oracle.attention(q, k, v, scale=0.03, causal=True)
    compare(o1, l1, ref_o, ref_lse, "scale 0.03")


def test_workspace_too_small_is_rejected():
    q, k, v = (t.to(DEV) for t in random_inputs((1, 4, 1, 128), (1, 1, 4096, 128), seed=2))
    nbytes, used = fa.splitkv_workspace(1, 4, 1, 1, 4096, 128, 8)
    assert used == 8 and nbytes > 0
    ws = torch.empty(nbytes - 256, dtype=torch.uint8, device=DEV)
    o = torch.empty((1, 4, 1, 128), dtype=torch.float32, device=DEV)
    lse = torch.empty((1, 4, 1), dtype=torch.float32, device=DEV)
    lib = fa.load_library()
    st = lib.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 4, 1, 1,
                            4096, 128, 0, 0.1, 8, ws.data_ptr(), ws.numel(), None)
    assert st == fa.FA_ERR_INVALID_ARG
    st = lib.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 4, 1, 1,
                            4096, 128, 0, 0.1, 8, None, 0, None)
    assert st == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("Hq,D", [(4, 128), (4, 64), (1, 64)])  # tensor-core (D = 128, 64) and FP32-pipe kernels
def test_timed_out_wait_is_reported_and_context_survives(Hq, D):
    """The test hook drops the first K/V tile of every CTA: the bounded wait
    runs out, the launch retires with FA_ERR_TIMEOUT, the next call works."""
    q, k, v = random_inputs((1, Hq, 1, D), (1, 1, 1024, D), seed=4)
    fa.load_library().fa_test_inject_fault(1)
    fa.fa_fwd_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), num_splits=2)
    with pytest.raises(fa.FAError) as ei:
        fa.fa_check()
    assert ei.value.status == fa.FA_ERR_TIMEOUT
    o, lse = run_splitkv(q, k, v, False, 2)
    ref_o, ref_lse = oracle.attention(q, k, v, scale=1 / math.sqrt(D), causal=False)
    compare(o, lse, ref_o, ref_lse, "after timeout")


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if w.decode])
def test_decode_workload_sampled(name):
    """Full-size decode workload in the launch configuration the benchmark
    times (automatic partitions), checked on sampled rows."""
    w = WORKLOADS[name]
    q, k, v = dense_inputs(w)
    o, lse = fa.fa_fwd_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal)
    fa.fa_check()
    n_total = w.B * w.Hq * w.Lq
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, n_total - 1], rng.integers(0, n_total, 96)]))
    ref_o, ref_lse = oracle.attention(q, k, v, scale=w.scale, causal=w.causal, rows=rows)
    o_s = o.reshape(-1, w.D)[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    l_s = lse.reshape(-1)[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    compare(o_s, l_s, ref_o, ref_lse, name)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
