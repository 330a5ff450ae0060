"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small and ragged shapes are compared element by element over every output;
the benchmark workloads at full size are compared on sampled rows, in the
same launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_07_gb300 as fa
import oracle
from parity import compare, sample_rows
from workloads import WORKLOADS, dense_inputs, random_inputs, varlen_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.load_library()


def run_dense(q, k, v, causal, scale=None, canary=True):
    """Run fa_fwd with guard bands around O and LSE; check the guards."""
    B, Hq, Lq, D = q.shape
    G = 4096
    o_buf = torch.full((B * Hq * Lq * D + 2 * G,), float("nan"), dtype=torch.float32, device=DEV)
    l_buf = torch.full((B * Hq * Lq + 2 * G,), 12345.0, dtype=torch.float32, device=DEV)
    o = o_buf[G:G + B * Hq * Lq * D].view(B, Hq, Lq, D)
    lse = l_buf[G:G + B * Hq * Lq].view(B, Hq, Lq)
    fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, softmax_scale=scale, out=o, lse=lse)
    fa.fa_check()
    if canary:
        assert torch.isnan(o_buf[:G]).all() and torch.isnan(o_buf[-G:]).all(), "O guard band written"
        assert (l_buf[:G] == 12345.0).all() and (l_buf[-G:] == 12345.0).all(), "LSE guard band written"
    return o.float().cpu().numpy(), lse.cpu().numpy()


DENSE_CASES = [
    # B, Hq, Hkv, Lq, Lk, D, causal, q_mult
    (1, 1, 1, 128, 128, 64, False, 1.0),     # the 128-token, D = 64 workload
    (1, 2, 2, 384, 384, 128, False, 1.0),    # several tiles, half-empty second Q tile
    (1, 2, 2, 384, 384, 128, True, 1.0),
    (2, 3, 3, 300, 300, 64, True, 1.0),      # ragged tail
    (2, 3, 3, 300, 300, 128, False, 1.0),
    (1, 2, 1, 200, 520, 128, True, 1.0),     # Lq < Lk, bottom-right causal
    (1, 2, 1, 520, 200, 64, True, 1.0),      # Lq > Lk: leading rows see no key
    (1, 1, 1, 1, 1, 64, False, 1.0),         # single element
    (1, 2, 2, 1, 1000, 128, True, 1.0),      # one query row, long key range
    (1, 8, 2, 513, 513, 128, True, 3.0),     # GQA r = 4, sharper softmax
    (1, 4, 1, 257, 700, 64, False, 1.0),     # MQA
    (1, 2, 2, 640, 640, 128, False, 20.0),   # very sharp softmax: exercises rescales
    (3, 2, 2, 1100, 1100, 64, True, 1.0),
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,D,causal,qm", DENSE_CASES)
def test_dense_small_full_compare(B, Hq, Hkv, Lq, Lk, D, causal, qm):
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=B * 7 + Lq + Lk + D, q_mult=qm)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_dense(q, k, v, causal)
    ref_o, ref_lse = oracle.attention(q, k, v, scale=scale, causal=causal)
    compare(o, lse, ref_o, ref_lse, f"dense {B,Hq,Hkv,Lq,Lk,D,causal,qm}")


def test_custom_scale_and_repeat_calls_identical():
    q, k, v = random_inputs((2, 4, 333, 128), (2, 4, 333, 128), seed=77)
    o1, l1 = run_dense(q, k, v, True, scale=0.05)
    o2, l2 = run_dense(q, k, v, True, scale=0.05)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2), "repeat calls must be bit-identical"
    ref_o, ref_lse = oracle.attention(q, k, v, scale=0.05, causal=True)
    compare(o1, l1, ref_o, ref_lse, "scale 0.05")


@pytest.mark.parametrize("mode", ["plain", "causal", "window", "alibi"])
def test_batch_equals_one_batch_at_a_time(mode):
    """A dense batch is launched as one list of (batch, head) slabs, each of
    its work tiles computed by one CTA with no cross-tile arithmetic, so every
    batch entry must come out bit-identical to a call on that entry alone;
    GQA (r = 4) checks that query head h of batch b reads KV head
    b * Hkv + h / r.  ALiBi slopes are per query head of one batch entry."""
    B, Hq, Hkv, L, D = 3, 8, 2, 700, 128
    q, k, v = random_inputs((B, Hq, L, D), (B, Hkv, L, D), seed=91)
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    slopes = torch.tensor([2.0 ** (-(i + 1)) for i in range(Hq)], dtype=torch.float32, device=DEV)

    def call(a, b, c):
        if mode in ("plain", "causal"):
            return fa.fa_fwd(a, b, c, causal=mode == "causal")
        if mode == "window":
            return fa.fa_fwd_variant(a, b, c, window=(300, 0))
        return fa.fa_fwd_variant(a, b, c, alibi_slopes=slopes)

    o, lse = call(qd, kd, vd)
    fa.fa_check()
    for b in range(B):
        ob, lb = call(qd[b:b + 1].contiguous(), kd[b:b + 1].contiguous(), vd[b:b + 1].contiguous())
        fa.fa_check()
        assert torch.equal(o[b:b + 1], ob) and torch.equal(lse[b:b + 1], lb), f"{mode}: batch entry {b}"


VARLEN_CASES = [
    ([1, 127, 128, 129, 300, 5], [1, 127, 128, 129, 300, 5], 4, 2, 128, True),
    ([1, 127, 128, 129, 300, 5], [1, 127, 128, 129, 300, 5], 4, 2, 64, False),
    ([50, 700, 3, 256], [90, 650, 3, 300], 8, 8, 128, True),     # Lq != Lk per sequence
    ([200, 0, 100], [200, 40, 0], 2, 1, 64, True),               # empty query / empty key sequences
]


def run_varlen(lq, lk, Hq, Hkv, D, causal, seed=5):
    Tq, Tk = sum(lq), sum(lk)
    q, k, v = random_inputs((Tq, Hq, D), (Tk, Hkv, D), seed=seed)
    cq = torch.tensor([0] + np.cumsum(lq).tolist(), dtype=torch.int32)
    ck = torch.tensor([0] + np.cumsum(lk).tolist(), dtype=torch.int32)
    o = torch.full((Tq, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((Hq, Tq), 12345.0, dtype=torch.float32, device=DEV)
    fa.fa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV), max(lq), max(max(lk), 1),
                     causal=causal, out=o, lse=lse)
    fa.fa_check()
    return q, k, v, cq, ck, o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("lq,lk,Hq,Hkv,D,causal", VARLEN_CASES)
def test_varlen_small_full_compare(lq, lk, Hq, Hkv, D, causal):
    q, k, v, cq, ck, o, lse = run_varlen(lq, lk, Hq, Hkv, D, causal)
    ref_o, ref_lse = oracle.attention_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=1 / math.sqrt(D), causal=causal)
    # O is [T, H, D] and LSE [H, T]: compare per head
    compare(o.transpose(1, 0, 2), lse, ref_o.transpose(1, 0, 2), ref_lse, f"varlen {lq} {lk}")


@pytest.mark.parametrize("D", [64, 128])
def test_varlen_batch_split_across_launches(D):
    """More sequences than one launch schedules: consecutive launches of
    FA_VARLEN_SEQS_PER_LAUNCH sequences, every row still compared in full."""
    rng = np.random.default_rng(100 + D)
    n = fa.VARLEN_SEQS_PER_LAUNCH + 70
    lq = rng.integers(0, 40, n).tolist()
    lk = [x + int(rng.integers(0, 9)) for x in lq]
    q, k, v, cq, ck, o, lse = run_varlen(lq, lk, 2, 1, D, True, seed=D)
    assert fa.fa_last_launch_count() == 2
    ref_o, ref_lse = oracle.attention_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=1 / math.sqrt(D), causal=True)
    compare(o.transpose(1, 0, 2), lse, ref_o.transpose(1, 0, 2), ref_lse, f"varlen split D={D}")


_CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8  # CUmemPool_attribute in cuda.h


def _default_pool_high(reset: bool) -> int:
    """High-water mark of the current device's stream-ordered memory pool
    (what cudaMallocAsync draws from), read through the driver API."""
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    dev = ctypes.c_int()
    assert cu.cuCtxGetDevice(ctypes.byref(dev)) == 0
    pool = ctypes.c_void_p()
    assert cu.cuDeviceGetDefaultMemPool(ctypes.byref(pool), dev) == 0
    val = ctypes.c_uint64(0)
    if reset:
        assert cu.cuMemPoolSetAttribute(pool, _CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(val)) == 0
    assert cu.cuMemPoolGetAttribute(pool, _CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(val)) == 0
    return int(val.value)


def test_varlen_allocates_no_device_memory():
    """fa_fwd_varlen obtains no device memory per call: the stream-ordered pool
    stays unused, torch's allocator serves no request, and the device's free
    memory is the same before and after the calls."""
    lens = [300, 1, 777, 128, 64, 2000]
    Hq, Hkv, D = 4, 2, 128
    T = sum(lens)
    q, k, v = (x.to(DEV) for x in random_inputs((T, Hq, D), (T, Hkv, D), seed=17))
    cu = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32, device=DEV)
    o = torch.empty((T, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=DEV)
    fa.fa_fwd_varlen(q, k, v, cu, cu, max(lens), max(lens), causal=True, out=o, lse=lse)  # loads the kernels
    torch.cuda.synchronize()
    fa.fa_check()
    assert _default_pool_high(reset=True) == 0
    allocs = torch.cuda.memory_stats()["allocation.all.allocated"]
    free0, _ = torch.cuda.mem_get_info()
    for causal in (True, False, True):
        fa.fa_fwd_varlen(q, k, v, cu, cu, max(lens), max(lens), causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    fa.fa_check()
    assert _default_pool_high(reset=False) == 0, "a stream-ordered allocation was made"
    assert torch.cuda.memory_stats()["allocation.all.allocated"] == allocs
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_varlen_invalid_offsets_latch_error():
    Hq, D = 2, 64
    q, k, v = random_inputs((300, Hq, D), (300, Hq, D), seed=3)
    bad = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device=DEV)  # decreasing
    o = torch.zeros((300, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.zeros((Hq, 300), dtype=torch.float32, device=DEV)
    fa.fa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), bad, bad, 300, 300, causal=True, out=o, lse=lse)
    with pytest.raises(fa.FAError) as ei:
        fa.fa_check()
    assert ei.value.status == fa.FA_ERR_INVALID_ARG
    fa.fa_check()  # latch cleared


# ------------------------------------------------------------------ benchmark workloads, full size

def _dense_workload(name):
    w = WORKLOADS[name]
    q, k, v = dense_inputs(w)
    if w.Dv != w.D:
        o, lse = fa.fa_fwd_hdim(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal)
    else:
        o, lse = fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal)
    fa.fa_check()
    return w, q, k, v, o, lse


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items()
                                  if not (w.varlen or w.bwd or w.fp8 or w.window is not None)])
def test_benchmark_workload_sampled(name):
    w, q, k, v, o, lse = _dense_workload(name)
    rows_per_slab = w.Lq
    n_total = w.B * w.Hq * w.Lq
    rng = np.random.default_rng(0)
    slabs = [0, w.B * w.Hq - 1, (w.B * w.Hq) // 2]
    rows = np.arange(n_total) if n_total <= 4096 else sample_rows(n_total, rows_per_slab, slabs, rng)
    ref_o, ref_lse = oracle.attention(q, k, v, scale=w.scale, causal=w.causal, rows=rows)
    o_s = o.float().reshape(-1, w.Dv)[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    l_s = lse.reshape(-1)[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    compare(o_s, l_s, ref_o, ref_lse, name)
    # properties that hold for every row at any size
    assert torch.isfinite(o.float()).all()
    assert torch.isfinite(lse).all()


def test_benchmark_varlen_workload_sampled():
    w = WORKLOADS["varlen8_h32x8_d128_causal"]
    q, k, v, cq, ck = varlen_inputs(w)
    o, lse = fa.fa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV), max(w.seqlens),
                              max(w.seqlens), causal=True)
    fa.fa_check()
    Tq = q.shape[0]
    rng = np.random.default_rng(1)
    picks = set(rng.integers(0, w.Hq * Tq, 1500).tolist())
    starts = cq.tolist()
    for s in range(len(starts) - 1):  # both ends of every sequence, a few heads
        for h in (0, 5, w.Hq - 1):
            for t in (starts[s], starts[s] + 1, starts[s + 1] - 1, starts[s] + 255, starts[s] + 256):
                if starts[s] <= t < starts[s + 1]:
                    picks.add(h * Tq + t)
    rows = np.array(sorted(picks), dtype=np.int64)
    ref_o, ref_lse = oracle.attention_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=w.scale, causal=True, rows=rows)
    h, t = rows // Tq, rows % Tq
    o_s = o.float()[torch.from_numpy(t).to(DEV), torch.from_numpy(h).to(DEV)].cpu().numpy()
    l_s = lse[torch.from_numpy(h).to(DEV), torch.from_numpy(t).to(DEV)].cpu().numpy()
    compare(o_s, l_s, ref_o, ref_lse, "varlen benchmark workload")
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


# ------------------------------------------------------------------ failure detection and limits

def test_timed_out_wait_is_reported_and_context_survives():
    """A wait that never completes (the test hook drops a K tile) ends the
    launch after its time limit with FA_ERR_TIMEOUT; the next call works."""
    q, k, v = random_inputs((1, 4, 512, 128), (1, 4, 512, 128), seed=99)
    lib = fa.load_library()
    lib.fa_test_inject_fault(1)
    fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    with pytest.raises(fa.FAError) as ei:
        fa.fa_check()
    assert ei.value.status == fa.FA_ERR_TIMEOUT
    o, lse = run_dense(q, k, v, True)  # same process, same context
    ref_o, ref_lse = oracle.attention(q, k, v, scale=1 / math.sqrt(128), causal=True)
    compare(o, lse, ref_o, ref_lse, "after timeout")


def test_long_key_range_large_indices():
    """Lk = 131072 keys (K and V 64 MiB each per head pair): 64-bit indexing
    and long KV loops; Lq < Lk with bottom-right causal alignment."""
    B, Hq, Hkv, Lq, Lk, D = 1, 2, 1, 256, 131072, 128
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=7)
    for causal in (False, True):
        o, lse = run_dense(q, k, v, causal)
        ref_o, ref_lse = oracle.attention(q, k, v, scale=1 / math.sqrt(D), causal=causal)
        compare(o, lse, ref_o, ref_lse, f"Lk=131072 causal={causal}")
