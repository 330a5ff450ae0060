"""fa_fwd_varlen_noalloc: the packed forward for callers that cannot call
cudaMalloc on the hot path (a process whose device memory all belongs to its
own allocator, a server that must not allocate while serving).  It sorts the
whole batch into a fixed array inside the library and runs one attention
launch over it.

Each case is checked twice: against fa_fwd_varlen on the same inputs and
against the fp64 oracle.  This file is collected last so that a run stopping
at the first failure has already run every other test.  It builds what it
needs itself, so it passes alone in a fresh process as well as after the rest
of the suite.
"""
import ctypes
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


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return fa.load_library()


def _packed(lens_q, lens_k, Hq, Hkv, D, seed):
    q, k, v = random_inputs((sum(lens_q), Hq, D), (sum(lens_k), Hkv, D), seed=seed)
    cq = torch.tensor([0] + np.cumsum(lens_q).tolist(), dtype=torch.int32)
    ck = torch.tensor([0] + np.cumsum(lens_k).tolist(), dtype=torch.int32)
    return q, k, v, cq, ck


def _noalloc_abi(lib, q, k, v, cq, ck, max_q, max_k, causal):
    """The entry point called through the C ABI directly."""
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    o = torch.full((Tq, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((Hq, Tq), 12345.0, dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.fa_fwd_varlen_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   cq.data_ptr(), ck.data_ptr(), cq.numel() - 1, Tq, Tk, max_q, max_k, Hq, Hkv, D,
                                   int(causal), ctypes.c_float(1.0 / D ** 0.5), stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    fa.fa_check()
    return o, lse


def _noalloc_python(q, k, v, cq, ck, max_q, max_k, causal):
    """The same entry point through the Python binding."""
    Tq, Hq, D = q.shape
    o = torch.full((Tq, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((Hq, Tq), 12345.0, dtype=torch.float32, device=DEV)
    fa.fa_fwd_varlen_noalloc(q, k, v, cq, ck, max_q, max_k, o, lse, causal=causal)
    fa.fa_check()
    return o, lse


def _short_batch(n, seed):
    rng = np.random.default_rng(seed)
    lq = rng.integers(0, 9, n).tolist()
    lk = [x + int(rng.integers(0, 4)) for x in lq]
    return lq, lk


CASES = [
    # lengths of queries and keys, Hq, Hkv, D, causal, seed, call through the binding
    ([300, 1, 777, 128, 64], [300, 1, 777, 128, 64], 4, 2, 128, True, 21, False),
    ([5, 1000, 256, 0, 33, 129, 7], [5, 1000, 300, 40, 33, 129, 70], 8, 8, 64, False, 22, True),
    # more sequences than the schedule kernel sorts (4096): the batch keeps its
    # order, and the upper part of the fixed array is written and read
    (*_short_batch(5000, 23), 2, 1, 64, True, 23, False),
]


def test_noalloc_matches_existing_entry_point_and_oracle_on_calls_in_a_row(lib):
    # consecutive calls with different batches share the fixed schedule
    # array; each must agree with fa_fwd_varlen and with the fp64 oracle
    for lens_q, lens_k, Hq, Hkv, D, causal, seed, python in CASES:
        q, k, v, cq, ck = _packed(lens_q, lens_k, Hq, Hkv, D, seed)
        qd, kd, vd, cqd, ckd = (x.to(DEV) for x in (q, k, v, cq, ck))
        max_q, max_k = max(max(lens_q), 1), max(max(lens_k), 1)
        ref_o, ref_lse = fa.fa_fwd_varlen(qd, kd, vd, cqd, ckd, max_q, max_k, causal=causal)
        fa.fa_check()
        if python:
            o, lse = _noalloc_python(qd, kd, vd, cqd, ckd, max_q, max_k, causal)
        else:
            o, lse = _noalloc_abi(lib, qd, kd, vd, cqd, ckd, max_q, max_k, causal)
        assert fa.fa_last_launch_count() == 2  # schedule kernel + one attention launch
        o = o.cpu().numpy().transpose(1, 0, 2)
        lse = lse.cpu().numpy()
        ro = ref_o.cpu().numpy().astype(np.float64).transpose(1, 0, 2)
        rl = ref_lse.cpu().numpy().astype(np.float64)
        compare(o, lse, ro, rl, f"noalloc vs fa_fwd_varlen, {len(lens_q)} sequences")
        oo, ol = oracle.attention_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=1 / math.sqrt(D), causal=causal)
        compare(o, lse, oo.transpose(1, 0, 2), ol, f"noalloc vs oracle, {len(lens_q)} sequences")


def test_noalloc_rejects_batches_beyond_its_limit(lib):
    n = fa.NOALLOC_MAX_SEQS + 1
    st = lib.fa_fwd_varlen_noalloc(16, 16, 16, 16, 16, 32, 32, n, n, n, 1, 1, 2, 2, 128, 1,
                                   ctypes.c_float(0.1), None)
    assert st == fa.FA_ERR_INVALID_ARG
