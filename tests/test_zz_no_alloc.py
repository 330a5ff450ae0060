"""fa_fwd_varlen_noalloc: the variable-length forward for callers that cannot
allocate device memory (for example work recorded into a CUDA graph, or a
process whose device memory all belongs to its own allocator).  It keeps the
sequence schedule in a fixed array inside the library instead of obtaining a
buffer per call.

This file is collected last so that a run stopping at the first failure has
already run every other test.  It builds what it needs itself, so it passes
alone in a fresh process as well as after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_07_gb300 as fa
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
    return q.to(DEV), k.to(DEV), v.to(DEV), cq.to(DEV), ck.to(DEV)


def _noalloc(lib, q, k, v, cq, ck, max_q, max_k, causal):
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


CASES = [
    # lengths of queries and keys, Hq, Hkv, D, causal, seed
    ([300, 1, 777, 128, 64], [300, 1, 777, 128, 64], 4, 2, 128, True, 21),
    ([5, 1000, 256, 0, 33, 129, 7], [5, 1000, 300, 40, 33, 129, 70], 8, 8, 64, False, 22),
]


def test_noalloc_matches_existing_entry_point_on_two_calls_in_a_row(lib):
    # two consecutive calls with different batches share the fixed schedule
    # array; each must agree with fa_fwd_varlen on the same inputs
    for lens_q, lens_k, Hq, Hkv, D, causal, seed in CASES:
        q, k, v, cq, ck = _packed(lens_q, lens_k, Hq, Hkv, D, seed)
        max_q, max_k = max(lens_q), max(max(lens_k), 1)
        ref_o, ref_lse = fa.fa_fwd_varlen(q, k, v, cq, ck, max_q, max_k, causal=causal)
        fa.fa_check()
        o, lse = _noalloc(lib, q, k, v, cq, ck, max_q, max_k, causal)
        assert fa.fa_last_launch_count() == 2
        ro = ref_o.cpu().numpy().astype(np.float64).transpose(1, 0, 2)
        rl = ref_lse.cpu().numpy().astype(np.float64)
        compare(o.cpu().numpy().transpose(1, 0, 2), lse.cpu().numpy(), ro, rl, f"noalloc {lens_q}")


def test_noalloc_rejects_batches_beyond_its_limit(lib):
    n = fa.NOALLOC_MAX_SEQS + 1
    st = lib.fa_fwd_varlen_noalloc(16, 16, 16, 16, 16, 32, 32, n, n, n, 1, 1, 2, 2, 128, 1,
                                   ctypes.c_float(0.1), None)
    assert st == fa.FA_ERR_INVALID_ARG
