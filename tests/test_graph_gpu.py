"""The entry points inside CUDA graphs.

Short problems are dominated by the host side of a call (tens of
microseconds against a few of kernel time), so callers capture their calls
into a CUDA graph and replay it.  Every entry point here takes caller-owned
buffers, launches only kernels and copies nothing back to the host, so a
captured call must replay to exactly what the same call computes eagerly, on
whatever the captured input buffers hold at replay time.  The forward
kernels, the split-KV partials and merge, and the backward's dK and dV are
deterministic and must match bit for bit; dQ is summed by reduce-adds in an
order that varies from run to run and must match to rounding.
"""
import numpy as np
import pytest
import torch

import exact_attention_07_gb300 as fa
from workloads import grad_output, random_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.load_library()


def capture(fn):
    """Runs fn once on a side stream (the first call on a device sets up the
    library's per-device state), then captures it into a graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def refill(dst, src):
    dst.copy_(src.to(DEV))


def test_dense_forward_graph_replays_eager_results():
    q, k, v = random_inputs((2, 4, 300, 128), (2, 2, 300, 128), seed=71)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o = torch.empty((2, 4, 300, 128), dtype=torch.float32, device=DEV)
    lse = torch.empty((2, 4, 300), dtype=torch.float32, device=DEV)
    g = capture(lambda: fa.fa_fwd(qd, kd, vd, causal=True, out=o, lse=lse))
    for seed in (72, 73):  # new inputs in the captured buffers
        q2, k2, v2 = random_inputs((2, 4, 300, 128), (2, 2, 300, 128), seed=seed)
        for d, s in ((qd, q2), (kd, k2), (vd, v2)):
            refill(d, s)
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        fa.fa_check()
        o_ref, l_ref = fa.fa_fwd(qd, kd, vd, causal=True)
        fa.fa_check()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_varlen_forward_graph_replays_eager_results():
    lens = [130, 7, 400]
    T, Hq, Hkv, D = sum(lens), 4, 2, 128
    q, k, v = random_inputs((T, Hq, D), (T, Hkv, D), seed=74)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    cu = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32, device=DEV)
    o = torch.empty((T, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=DEV)
    g = capture(lambda: fa.fa_fwd_varlen(qd, kd, vd, cu, cu, max(lens), max(lens), causal=True, out=o, lse=lse))
    q2, k2, v2 = random_inputs((T, Hq, D), (T, Hkv, D), seed=75)
    for d, s in ((qd, q2), (kd, k2), (vd, v2)):
        refill(d, s)
    o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    fa.fa_check()
    o_ref, l_ref = fa.fa_fwd_varlen(qd, kd, vd, cu, cu, max(lens), max(lens), causal=True)
    fa.fa_check()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_splitkv_decode_graph_replays_eager_results():
    B, Hq, Hkv, Lk, D = 2, 8, 2, 5000, 128
    q, k, v = random_inputs((B, Hq, 1, D), (B, Hkv, Lk, D), seed=76)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    nbytes, _ = fa.splitkv_workspace(B, Hq, Hkv, 1, Lk, D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o = torch.empty((B, Hq, 1, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=DEV)
    g = capture(lambda: fa.fa_fwd_splitkv(qd, kd, vd, out=o, lse=lse, workspace=ws))
    q2, _, _ = random_inputs((B, Hq, 1, D), (B, Hkv, 1, D), seed=77)
    refill(qd, q2)  # a new query token against the same cache
    o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    fa.fa_check()
    o_ref, l_ref = fa.fa_fwd_splitkv(qd, kd, vd, workspace=ws)
    fa.fa_check()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_backward_graph_replays_eager_results():
    B, Hq, Hkv, L, D = 1, 4, 2, 333, 128
    q, k, v = random_inputs((B, Hq, L, D), (B, Hkv, L, D), seed=78)
    do = grad_output((B, Hq, L, D), 78)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fa_fwd(qd, kd, vd, causal=True)
    ws = torch.empty(fa.bwd_workspace(B, Hq, L), dtype=torch.uint8, device=DEV)
    dq = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    dk = torch.empty(k.shape, dtype=torch.float32, device=DEV)
    dv = torch.empty(k.shape, dtype=torch.float32, device=DEV)
    g = capture(lambda: fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws))
    refill(dod, grad_output((B, Hq, L, D), 79))  # a new upstream gradient
    for t in (dq, dk, dv):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    fa.fa_check()
    rq, rk, rv = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True, workspace=ws)
    fa.fa_check()
    assert torch.equal(dk, rk) and torch.equal(dv, rv)
    assert torch.isfinite(dq).all()
    assert (dq - rq).abs().max().item() <= 1e-5 * rq.abs().max().item()
