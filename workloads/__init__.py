"""Seeded synthetic inputs for exact attention forward.

This module holds no attention arithmetic: it only draws random tensors and
packs them.  Both the fp64 oracle (test infrastructure) and the CUDA path are
fed from here, so the two sides always see identical bf16 inputs.

Recipe (the pages only say "i.i.d. N(0,1) from seed 0"; this is the reading
taken): a CPU ``torch.Generator`` seeded with ``seed`` draws Q, then K, then V
with ``torch.randn(..., dtype=float32)``; Q is multiplied by ``q_mult``; all
three are then rounded to bf16 (round-to-nearest-even).  The oracle consumes
the rounded bf16 values, so input quantisation is not counted as error.

Variable-length batches draw their lengths with
``torch.randint(lo, hi + 1, (n,))`` from a generator seeded with ``seed``
("uniform on [lo, hi]", read as inclusive) and pack sequences token-major,
``[total_tokens, heads, D]``, with int32 prefix offsets ``cu_seqlens``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    """One attention-forward problem: shapes, mask and input recipe."""

    name: str
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    D: int
    causal: bool
    q_mult: float = 1.0
    seed: int = 0
    # variable-length batches: per-sequence lengths (Lq/Lk above are unused)
    seqlens: tuple[int, ...] | None = None
    # decode-shaped problem (few query rows per KV head, long key range) that
    # runs through the split-KV forward
    decode: bool = False
    # the backward pass (fa_bwd) of this problem instead of the forward
    bwd: bool = False
    # key window (left, right) around each query's aligned position, run
    # through the variant forward (-1 = unlimited)
    window: tuple[int, int] | None = None
    # the FP8 forward (e4m3 inputs after the Hadamard rotation)
    fp8: bool = False
    # value head dimension when it differs from the query/key one D
    dv: int | None = None

    @property
    def Dv(self) -> int:
        return self.D if self.dv is None else self.dv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def varlen(self) -> bool:
        return self.seqlens is not None

    def flops(self) -> float:
        """Matrix FLOPs of the forward: 2*Lq*Lk*(D + Dv) per head (4*Lq*Lk*D
        when Dv = D), halved when causal.

        Multiply and add are counted separately; the causal half ignores the
        diagonal's extra half tile.
        """
        dd = 2.0 * (self.D + self.Dv)
        if self.varlen:
            total = sum(dd * self.Hq * L * L for L in self.seqlens)
        else:
            total = dd * self.B * self.Hq * self.Lq * self.Lk
        if self.window is not None:  # count only the pairs the window allows
            import numpy as np
            c = np.arange(self.Lq, dtype=np.int64) + (self.Lk - self.Lq)
            lo = np.maximum(0, c - self.window[0]) if self.window[0] >= 0 else np.zeros_like(c)
            hi = np.minimum(self.Lk - 1, c + self.window[1]) if self.window[1] >= 0 else np.full_like(c, self.Lk - 1)
            pairs = float(np.maximum(hi - lo + 1, 0).sum())
            return dd * self.B * self.Hq * pairs * (2.5 if self.bwd else 1.0)
        if self.bwd:  # five matrix products instead of two (S, dP, dV, dQ, dK)
            total *= 2.5
        return total / 2 if self.causal else total

    def hbm_bytes(self) -> float:
        """Least device-memory traffic of one forward: Q, K, V read once (bf16),
        O (fp32) and LSE (fp32) written once."""
        assert not self.varlen
        qo = self.B * self.Hq * self.Lq
        return (2.0 * qo * self.D + 2.0 * self.B * self.Hkv * self.Lk * (self.D + self.Dv) + 4.0 * qo * self.Dv
                + 4.0 * qo)


def varlen_lengths(n: int = 8, lo: int = 512, hi: int = 8192, seed: int = 0) -> list[int]:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def dense_inputs(w: Workload):
    """Q [B,Hq,Lq,D], K [B,Hkv,Lk,D] and V [B,Hkv,Lk,Dv], bf16 on the CPU."""
    assert not w.varlen
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.B, w.Hq, w.Lq, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Hkv, w.Lk, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, w.Lk, w.Dv), generator=g, dtype=torch.float32)
    if w.q_mult != 1.0:
        q = q * w.q_mult
    return _bf16(q), _bf16(k), _bf16(v)


def varlen_inputs(w: Workload):
    """Packed Q [Tq,Hq,D], K and V [Tk,Hkv,D] (bf16) and int32 cu_seqlens.

    Query and key lengths are equal per sequence (self-attention prefill).
    """
    assert w.varlen
    lens = list(w.seqlens)
    total = sum(lens)
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((total, w.Hq, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((total, w.Hkv, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((total, w.Hkv, w.D), generator=g, dtype=torch.float32)
    if w.q_mult != 1.0:
        q = q * w.q_mult
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return _bf16(q), _bf16(k), _bf16(v), cu, cu.clone()


def random_inputs(shape_q, shape_k, seed: int, q_mult: float = 1.0, shape_v=None):
    """Generic seeded bf16 triple for edge-case tests with arbitrary shapes;
    V has shape ``shape_v`` (default: the shape of K)."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(shape_q, generator=g, dtype=torch.float32) * q_mult
    k = torch.randn(shape_k, generator=g, dtype=torch.float32)
    v = torch.randn(shape_k if shape_v is None else shape_v, generator=g, dtype=torch.float32)
    return _bf16(q), _bf16(k), _bf16(v)


def grad_output(shape, seed: int):
    """Seeded upstream gradient dO for the backward pass: N(0,1) from its own
    generator (seed + 1000, so it never repeats the Q/K/V stream), bf16."""
    g = torch.Generator().manual_seed(seed + 1000)
    return _bf16(torch.randn(shape, generator=g, dtype=torch.float32))


def fp8_signs(d: int, seed: int):
    """The random +-1 signs of the FP8 rotation diag(signs) H / sqrt(d): a
    seeded draw, passed to both the kernel and the oracle (float64 array)."""
    import numpy as np
    g = torch.Generator().manual_seed(seed + 2000)
    return np.where(torch.rand(d, generator=g).numpy() < 0.5, -1.0, 1.0)


_VARLEN_LENS = tuple(varlen_lengths(8, 512, 8192, seed=0))

# The five workloads of the headline benchmark.  Names say what they are.
WORKLOADS: dict[str, Workload] = {
    "b1_h1_l128_d64": Workload("b1_h1_l128_d64", 1, 1, 1, 128, 128, 64, False),
    "b4_h16_l1024_d64": Workload("b4_h16_l1024_d64", 4, 16, 16, 1024, 1024, 64, False),
    "b4_h16_l1024_d64_causal": Workload("b4_h16_l1024_d64_causal", 4, 16, 16, 1024, 1024, 64, True),
    "gqa_b2_h32x8_l4096_d128_causal_q3": Workload(
        "gqa_b2_h32x8_l4096_d128_causal_q3", 2, 32, 8, 4096, 4096, 128, True, q_mult=3.0),
    "b1_h16_l16384_d128": Workload("b1_h16_l16384_d128", 1, 16, 16, 16384, 16384, 128, False),
    "b1_h16_l16384_d128_causal": Workload("b1_h16_l16384_d128_causal", 1, 16, 16, 16384, 16384, 128, True),
    "varlen8_h32x8_d128_causal": Workload(
        "varlen8_h32x8_d128_causal", 8, 32, 8, 0, 0, 128, True, seqlens=_VARLEN_LENS),
}

# A smaller case of the headline kernel for detailed profiler captures: Q, K,
# V and O still exceed the 126 MiB L2 (32 + 32 + 32 + 64 MiB), so DRAM
# counters stay meaningful, while one launch lasts about half a millisecond.
PROFILE_WORKLOADS: dict[str, Workload] = {
    "b1_h16_l8192_d128": Workload("b1_h16_l8192_d128", 1, 16, 16, 8192, 8192, 128, False),
}
WORKLOADS.update(PROFILE_WORKLOADS)

# Decode through the split-KV forward: one new token per sequence, GQA with
# four query heads per KV head, a 32768-token KV cache per sequence (K and V
# together 1 GiB, eight times the L2).  Shaped after the single-token GQA
# decode the pages discuss; no causal flag, since with one query row at the
# end of the cache every key is visible either way.
DECODE_WORKLOADS: dict[str, Workload] = {
    "decode_b8_h32x8_l32768_d128": Workload("decode_b8_h32x8_l32768_d128", 8, 32, 8, 1, 32768, 128, False,
                                            decode=True),
    "decode_b8_h32x8_l32768_d64": Workload("decode_b8_h32x8_l32768_d64", 8, 32, 8, 1, 32768, 64, False,
                                           decode=True),
}
WORKLOADS.update(DECODE_WORKLOADS)

# Backward of the long-sequence workloads (same shapes and seeds; dO drawn by
# grad_output), and a smaller case for profiler captures (Q, K, V, dO, O, dQ,
# dK, dV total 288 MiB, above the L2).
BWD_WORKLOADS: dict[str, Workload] = {
    "bwd_b1_h16_l16384_d128": Workload("bwd_b1_h16_l16384_d128", 1, 16, 16, 16384, 16384, 128, False, bwd=True),
    "bwd_b1_h16_l16384_d128_causal": Workload("bwd_b1_h16_l16384_d128_causal", 1, 16, 16, 16384, 16384, 128, True,
                                              bwd=True),
    "bwd_gqa_b2_h32x8_l4096_d128_causal_q3": Workload(
        "bwd_gqa_b2_h32x8_l4096_d128_causal_q3", 2, 32, 8, 4096, 4096, 128, True, q_mult=3.0, bwd=True),
    "bwd_b1_h16_l4096_d128": Workload("bwd_b1_h16_l4096_d128", 1, 16, 16, 4096, 4096, 128, False, bwd=True),
    # the sliding-window forward workload through the variant backward
    "bwd_swa4096_b1_h16_l16384_d128": Workload("bwd_swa4096_b1_h16_l16384_d128", 1, 16, 16, 16384, 16384, 128,
                                               False, window=(4095, 0), bwd=True),
    # the D = 64 forward workload's shape through the backward
    "bwd_b4_h16_l1024_d64": Workload("bwd_b4_h16_l1024_d64", 4, 16, 16, 1024, 1024, 64, False, bwd=True),
    # the packed forward workload's batch through the packed backward
    "bwd_varlen8_h32x8_d128_causal": Workload(
        "bwd_varlen8_h32x8_d128_causal", 8, 32, 8, 0, 0, 128, True, seqlens=_VARLEN_LENS, bwd=True),
}
WORKLOADS.update(BWD_WORKLOADS)

# Causal sliding window of width 4096 over the long-sequence shape (the
# variant forward skips KV tiles outside every row's window; FLOPs count the
# allowed pairs only).
VARIANT_WORKLOADS: dict[str, Workload] = {
    "swa4096_b1_h16_l16384_d128": Workload("swa4096_b1_h16_l16384_d128", 1, 16, 16, 16384, 16384, 128, False,
                                           window=(4095, 0)),
}
WORKLOADS.update(VARIANT_WORKLOADS)

# The long-sequence shape through the FP8 forward (inputs prepared once).
FP8_WORKLOADS: dict[str, Workload] = {
    "fp8_b1_h16_l16384_d128": Workload("fp8_b1_h16_l16384_d128", 1, 16, 16, 16384, 16384, 128, False, fp8=True),
}
WORKLOADS.update(FP8_WORKLOADS)

# Query/key head dimension 192 with value head dimension 128 (the asymmetric
# case of the FlashAttention-4 benchmarks) on the long-sequence shape.
HDIM_WORKLOADS: dict[str, Workload] = {
    "d192_b1_h16_l16384": Workload("d192_b1_h16_l16384", 1, 16, 16, 16384, 16384, 192, False, dv=128),
    "d192_b1_h16_l16384_causal": Workload("d192_b1_h16_l16384_causal", 1, 16, 16, 16384, 16384, 192, True, dv=128),
}
WORKLOADS.update(HDIM_WORKLOADS)

# The configuration the throughput metric is quoted on.
HEADLINE = "b1_h16_l16384_d128"
