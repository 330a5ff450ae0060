"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances (bf16 inputs, fp32 accumulation and output): O max-abs <= 1e-2 and
relative RMS <= 5e-3 against the fp64 oracle; LSE max-abs <= 1e-3 on rows
with at least one allowed key, and exactly -inf (with O == 0) on rows with
none.
"""
import numpy as np

O_MAX_ABS = 1e-2
O_REL_RMS = 5e-3
LSE_MAX_ABS = 1e-3


def compare(o, lse, ref_o, ref_lse, what=""):
    """o/lse: GPU results as float64 numpy arrays with the oracle's shapes."""
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert o.shape == ref_o.shape and lse.shape == ref_lse.shape, what
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    empty = ~np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf LSE pattern differs"
    assert np.all(lse[~empty] == lse[~empty]), f"{what}: NaN LSE"
    err = np.abs(o - ref_o).max() if o.size else 0.0
    denom = np.linalg.norm(ref_o)
    rel = np.linalg.norm(o - ref_o) / denom if denom > 0 else np.linalg.norm(o)
    lerr = np.abs(lse[~empty] - ref_lse[~empty]).max() if (~empty).any() else 0.0
    if empty.any():
        assert np.all(o[empty] == 0.0), f"{what}: empty rows must be zero"
    assert err <= O_MAX_ABS, f"{what}: max|dO| {err:.3e} > {O_MAX_ABS}"
    assert rel <= O_REL_RMS, f"{what}: relRMS {rel:.3e} > {O_REL_RMS}"
    assert lerr <= LSE_MAX_ABS, f"{what}: max|dLSE| {lerr:.3e} > {LSE_MAX_ABS}"
    return err, rel, lerr


def sample_rows(n_total, rows_per_slab, n_slabs, rng, n_random=600):
    """Flat row ids covering both ends of every 128-row tile of a few slabs
    plus random rows."""
    picks = set()
    for s in n_slabs:
        base = s * rows_per_slab
        for t in range(0, rows_per_slab, 128):
            for r in (t, t + 1, t + 63, t + 64, t + 126, t + 127):
                if r < rows_per_slab:
                    picks.add(base + r)
        picks.add(base + rows_per_slab - 1)
    picks.update(rng.integers(0, n_total, n_random).tolist())
    return np.array(sorted(picks), dtype=np.int64)
