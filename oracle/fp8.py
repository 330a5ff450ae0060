"""fp64 oracle for the FP8 forward (block quantisation with incoherent
processing) -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  Nothing here is shared with the CUDA path.

Method (FlashAttention from Scratch, sec. 10.3 "Treat FP8 as a second
lesson"; FlashAttention 1-4, FA3 item 3 "FP8 with block quantization and
incoherent processing"):

1. Incoherent processing: Q and K are multiplied by the same orthogonal
   matrix M = diag(signs) H / sqrt(d), with H the Sylvester Hadamard matrix
   and a random sign vector (drawn by the caller and passed in), so that
   (QM)(KM)^T = QK^T in exact arithmetic while outlier coordinates are spread
   over all d coordinates.
2. Block quantisation: one FP8 (e4m3) scale per tile of 128 rows of a
   (batch, head) slice of QM and KM, scale = amax(tile) / 448 (448 is the
   largest finite e4m3 value; an all-zero tile gets scale 1).  V is not
   rotated (the rotation would have to be undone on O); it gets one scale per
   (batch, KV head).  Codes are round-to-nearest-even of x / scale.
3. Attention runs on the dequantised inputs code * scale.

:func:`prepare` returns the codes (as their fp32 values) and scales;
:func:`attention_fp8_inputs` is the exact (fp64) attention of the
dequantised inputs -- what the FP8 kernel computes apart from rounding P to
e4m3 for the P.V product.
"""
from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0
TILE = 128


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (a power of two), entries +-1."""
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    assert h.shape[0] == d, "d must be a power of two"
    return h


def rotation(signs) -> np.ndarray:
    """M = diag(signs) H / sqrt(d): orthogonal."""
    s = _f64(signs).ravel()
    d = s.size
    return (s[:, None] * hadamard(d)) / np.sqrt(d)


def round_e4m3(x) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even) through PyTorch's
    float8_e4m3fn conversion, after rounding to fp32 as the device does;
    |x| must not exceed 448."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def quantize_tiles(x: np.ndarray, rows_per_tile: int = TILE):
    """x [S, L, D] (S slices): per slice, per tile of rows, scale = amax/448.
    Returns (codes as float64 values, scales [S, ceil(L/tile)])."""
    S, L, D = x.shape
    nt = (L + rows_per_tile - 1) // rows_per_tile
    codes = np.zeros_like(x)
    scales = np.ones((S, nt))
    for s in range(S):
        for t in range(nt):
            blk = x[s, t * rows_per_tile:(t + 1) * rows_per_tile]
            amax = np.abs(blk).max() if blk.size else 0.0
            sc = amax / E4M3_MAX if amax > 0 else 1.0
            scales[s, t] = sc
            codes[s, t * rows_per_tile:(t + 1) * rows_per_tile] = round_e4m3(blk / sc)
    return codes, scales


def prepare(q, k, v, signs, rotate: bool = True, block_q: bool = True):
    """Quantised inputs of the FP8 forward.  q [B, Hq, Lq, D], k/v [B, Hkv, Lk, D].

    Returns a dict with the codes (float64 values) and scales:
    qc [B, Hq, Lq, D], sq [B, Hq, nq]; kc [B, Hkv, Lk, D], sk [B, Hkv, nk];
    vc [B, Hkv, Lk, D], sv [B, Hkv].  rotate=False skips step 1, block_q=False
    uses one scale per (batch, head) for Q and K instead of per tile (both for
    comparisons only).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    if rotate:
        m = rotation(signs)
        q = q @ m
        k = k @ m
    tile_q = TILE if block_q else max(Lq, 1)
    tile_k = TILE if block_q else max(Lk, 1)
    qc, sq = quantize_tiles(q.reshape(B * Hq, Lq, D), tile_q)
    kc, sk = quantize_tiles(k.reshape(B * Hkv, Lk, D), tile_k)
    vc, sv = quantize_tiles(v.reshape(B * Hkv, Lk, D), max(Lk, 1))
    return {"qc": qc.reshape(B, Hq, Lq, D), "sq": sq.reshape(B, Hq, -1), "tile_q": tile_q,
            "kc": kc.reshape(B, Hkv, Lk, D), "sk": sk.reshape(B, Hkv, -1), "tile_k": tile_k,
            "vc": vc.reshape(B, Hkv, Lk, D), "sv": sv.reshape(B, Hkv)}


def dequantize(prep):
    """(q, k, v) rebuilt from codes and scales (float64)."""
    def expand(c, s, tile):
        rows = np.arange(c.shape[2]) // tile
        return c * s[:, :, rows][..., None]
    q = expand(prep["qc"], prep["sq"], prep["tile_q"])
    k = expand(prep["kc"], prep["sk"], prep["tile_k"])
    v = prep["vc"] * prep["sv"][:, :, None, None]
    return q, k, v


def attention_fp8_inputs(prep, scale: float, causal: bool = False, rows=None):
    """Exact attention (fp64, C oracle) of the dequantised inputs."""
    import oracle
    q, k, v = dequantize(prep)
    return oracle.attention(torch.from_numpy(q.astype(np.float32)), torch.from_numpy(k.astype(np.float32)),
                            torch.from_numpy(v.astype(np.float32)), scale=scale, causal=causal, rows=rows)
