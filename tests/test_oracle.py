"""Pins of the fp64 oracle to the pages and to mathematics (CPU only).

Every test here checks the oracle against something other than itself: a
number printed on the pages, an invariant the pages state, a special case that
reduces to a smaller problem, or an independent brute-force evaluation in
multi-precision arithmetic.
"""
import math
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import reference as R
from workloads import random_inputs


def c_oracle_1head(q, k, v, scale, causal=False):
    """C oracle on one head given [Nq,d], [Nk,d], [Nk,dv] lists (dv == d)."""
    q = torch.tensor(q, dtype=torch.float32)[None, None]
    k = torch.tensor(k, dtype=torch.float32)[None, None]
    v = torch.tensor(v, dtype=torch.float32)[None, None]
    o, lse = oracle.attention(q, k, v, scale=scale, causal=causal)
    return o[0, 0], lse[0, 0]


def printed(x, value, decimals):
    """True when x agrees with a number the page prints to ``decimals`` places.

    The pages round some numbers and truncate others, so the check allows
    one unit in the last printed digit.
    """
    return abs(float(x) - value) <= 10.0 ** (-decimals) * (1 + 1e-9)


def scalar_problem(scores, values):
    """d = 1 problem whose scores are exactly ``scores``: q = 1, k_j = s_j."""
    q = [[1.0]]
    k = [[float(s)] for s in scores]
    v = [[float(x)] for x in values]
    return q, k, v


# ----------------------------------------------------------------- worked examples

def test_three_scores_dense(golden):
    g = golden["three_scores"]
    q, k, v = scalar_problem(g["scores"], g["values"])
    o, lse = c_oracle_1head(q, k, v, scale=1.0)
    assert printed(o[0, 0], g["output"], g["output_decimals"])
    o2 = R.definition(q, k, v, scale=1.0).o
    assert printed(o2[0, 0], g["output"], g["output_decimals"])
    # LSE is the natural-log normaliser of the row: exp(lse) sums the weights
    assert math.isclose(math.exp(float(lse[0])), sum(math.exp(s) for s in g["scores"]), rel_tol=1e-14)


def test_three_scores_online(golden):
    g = golden["three_scores"]
    q, k, v = scalar_problem(g["scores"], g["values"])
    hist = []
    o, _ = R.online(q, k, v, scale=1.0, key_blocks=R.blocks(3, 2), history=hist)
    assert printed(o[0, 0], g["output"], g["output_decimals"])
    # the maximum rises from 2 to 3 on the second tile: alpha = e^(2-3)
    m1, m2 = hist[0].top, hist[1].top
    assert float(m1[0]) == 2.0 and float(m2[0]) == 3.0
    assert math.isclose(math.exp(float(m1[0] - m2[0])), math.exp(-1.0), rel_tol=0, abs_tol=0)


def test_two_tile_example_intermediates(golden):
    g = golden["two_tiles"]
    dec = g["decimals"]
    q, k, v = scalar_problem(g["scores"], g["values"])
    hist = []
    o, _ = R.online(q, k, v, scale=1.0, key_blocks=R.blocks(len(k), g["tile_size"]), history=hist)
    (m1, l1, A1), (m2, l2, A2) = ((h.top, h.mass, h.acc) for h in hist)
    assert float(m1[0]) == g["m1"] and float(m2[0]) == g["m2"]
    assert printed(l1[0], g["l1"], dec["l1"])
    assert printed(A1[0, 0], g["A1"], dec["A1"])
    assert printed(math.exp(float(m1[0] - m2[0])), g["alpha"], dec["alpha"])
    assert printed(l2[0], g["l2"], dec["l2"])
    assert printed(A2[0, 0], g["A2"], dec["A2"])
    assert printed(o[0, 0], g["output"], dec["output"])
    # "identical to one global softmax over all four scores"
    oc, _ = c_oracle_1head(q, k, v, scale=1.0)
    assert abs(float(oc[0, 0]) - float(o[0, 0])) < 1e-12
    assert printed(oc[0, 0], g["output"], dec["output"])


def test_conditional_rescale_keeps_reference(golden):
    g2 = golden["two_tiles"]
    c = golden["conditional_rescale"]
    tau = c["tau_log2"] * math.log(2.0)  # 8 in base 2 is 8 ln 2 in natural units
    assert math.isclose(math.exp(tau), c["factor"], rel_tol=1e-12)
    q, k, v = scalar_problem(g2["scores"], g2["values"])
    hist = []
    o_lazy, lse_lazy = R.online(q, k, v, scale=1.0, key_blocks=R.blocks(4, 2), tau=tau, history=hist)
    o_eager, lse_eager = R.online(q, k, v, scale=1.0, key_blocks=R.blocks(4, 2))
    # max 2 -> 3 is within the threshold: the reference stays at 2
    assert float(hist[1].top[0]) == 2.0
    assert abs(float(o_lazy[0, 0] - o_eager[0, 0])) < 1e-12
    assert abs(float(lse_lazy[0] - lse_eager[0])) < 1e-12
    # a jump larger than the threshold does move the reference
    q, k, v = scalar_problem([0.0, 1.0, 20.0, 3.0], [1.0, 2.0, 3.0, 4.0])
    hist = []
    R.online(q, k, v, scale=1.0, key_blocks=R.blocks(4, 2), tau=tau, history=hist)
    assert float(hist[0].top[0]) == 1.0 and float(hist[1].top[0]) == 20.0


# ---------------------------------------------------------------------- invariants

def test_shift_by_1000_leaves_output_unchanged():
    base = [1.0, 2.0, 3.0]
    vals = [10.0, 20.0, 30.0]
    # d = 2: q = (1, 1) and k_j = (s_j, shift) give scores s_j + shift
    for shift in (0.0, 1000.0):
        q = [[1.0, 1.0]]
        k = [[s, shift] for s in base]
        v = [[x, -x] for x in vals]
        o, lse = c_oracle_1head(q, k, v, scale=1.0)
        if shift == 0.0:
            o0, lse0 = o, lse
    assert np.all(np.isfinite(o))  # a missing max-subtraction overflows here
    assert np.max(np.abs(o - o0)) < 1e-12
    assert abs(float(lse[0] - lse0[0]) - 1000.0) < 1e-9


def test_masking_renormalises_remaining_keys(golden):
    g = golden["three_scores"]
    # two query rows against three keys, bottom-right causal: row 0 may see keys 0..1
    q = [[1.0], [1.0]]
    k = [[s] for s in g["scores"]]
    v = [[x] for x in g["values"]]
    o, lse = c_oracle_1head(q, k, v, scale=1.0, causal=True)
    o_first_two, _ = c_oracle_1head([[1.0]], k[:2], v[:2], scale=1.0)
    assert abs(float(o[0, 0] - o_first_two[0, 0])) < 1e-12
    # setting the old third weight to zero without renormalising is a different answer
    w = np.exp(np.array(g["scores"]) - 3.0)
    w /= w.sum()
    zeroed = w[0] * 10 + w[1] * 20
    assert abs(float(o[0, 0]) - zeroed) > 1.0
    # row 1 sees all three keys
    full, _ = c_oracle_1head([[1.0]], k, v, scale=1.0)
    assert abs(float(o[1, 0] - full[0, 0])) < 1e-12


def test_rectangular_causal_alignment_matches_table(golden):
    t = golden["rectangular_causal"]
    nq, nk = len(t["query_positions"]), len(t["key_positions"])
    rng = np.random.default_rng(3)
    q = rng.standard_normal((nq, 4)).astype(np.float32)
    k = rng.standard_normal((nk, 4)).astype(np.float32)
    v = rng.standard_normal((nk, 4)).astype(np.float32)
    o0, _ = c_oracle_1head(q.tolist(), k.tolist(), v.tolist(), scale=0.5, causal=True)
    allowed = np.zeros((nq, nk), dtype=int)
    for j in range(nk):
        v2 = v.copy()
        v2[j] += 100.0  # a key influences a row iff its value moves that row
        o1, _ = c_oracle_1head(q.tolist(), k.tolist(), v2.tolist(), scale=0.5, causal=True)
        allowed[:, j] = (np.abs(o1 - o0).max(axis=1) > 1e-9).astype(int)
    assert allowed.tolist() == t["allowed"]


def test_probability_rows_sum_to_one():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((9, 8))
    k = rng.standard_normal((13, 8)) * 3
    v = rng.standard_normal((13, 8))
    for causal in (False, True):
        p = R.definition(q, k, v, causal=causal, qpos=R.positions(9, 4)).p
        assert np.all(p >= 0)
        assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-15 * 16


# --------------------------------------------------------------- brute force (mpmath)

def brute_force_mp(q, k, v, scale, causal, dps=40):
    """Independent multi-precision evaluation, one scalar at a time."""
    import mpmath
    mpmath.mp.dps = dps
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    Dv = v.shape[3]
    r = Hq // Hkv
    O = np.zeros((B, Hq, Lq, Dv))
    L = np.zeros((B, Hq, Lq))
    for b in range(B):
        for h in range(Hq):
            hk = h // r
            for i in range(Lq):
                w = []
                for j in range(Lk):
                    if causal and j > i + (Lk - Lq):
                        continue
                    dot = mpmath.fsum(mpmath.mpf(float(q[b, h, i, d])) * mpmath.mpf(float(k[b, hk, j, d]))
                                      for d in range(D))
                    w.append((j, mpmath.mpf(scale) * dot))
                if not w:
                    L[b, h, i] = -np.inf
                    continue
                z = mpmath.fsum(mpmath.e ** s for _, s in w)
                for d in range(Dv):
                    O[b, h, i, d] = float(mpmath.fsum(mpmath.e ** s * mpmath.mpf(float(v[b, hk, j, d]))
                                                      for j, s in w) / z)
                L[b, h, i] = float(mpmath.log(z))
    return O, L


@pytest.mark.parametrize("Lq,Lk,causal", [(5, 7, False), (5, 7, True), (7, 4, True), (3, 3, True)])
def test_c_oracle_against_mpmath_brute_force(Lq, Lk, causal):
    B, Hq, Hkv, D = 2, 4, 2, 3
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=11 + Lq + Lk, q_mult=2.0)
    scale = 0.7
    o, lse = oracle.attention(q, k, v, scale=scale, causal=causal)
    qf, kf, vf = q.float().numpy(), k.float().numpy(), v.float().numpy()
    O, L = brute_force_mp(qf, kf, vf, scale, causal)
    assert np.max(np.abs(o - O)) < 1e-13
    fin = np.isfinite(L)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - L[fin])) < 1e-13
    assert np.all(lse[~fin] == -np.inf) and np.all(o[~fin] == 0.0)
    if causal and Lq > Lk:
        assert (~fin).sum() == B * Hq * (Lq - Lk)  # rows i < Lq - Lk see no key


@pytest.mark.parametrize("D,Dv,causal", [(3, 5, False), (6, 2, True)])
def test_c_oracle_value_width_against_mpmath(D, Dv, causal):
    # values (and outputs) with Dv elements per row while queries and keys
    # have D, as in the (192, 128) head-dimension case
    B, Hq, Hkv, Lq, Lk = 1, 4, 2, 6, 9
    q, k, v = random_inputs((B, Hq, Lq, D), (B, Hkv, Lk, D), seed=31 + D, shape_v=(B, Hkv, Lk, Dv))
    o, lse = oracle.attention(q, k, v, scale=0.6, causal=causal)
    assert o.shape == (B, Hq, Lq, Dv)
    O, L = brute_force_mp(q.float().numpy(), k.float().numpy(), v.float().numpy(), 0.6, causal)
    assert np.max(np.abs(o - O)) < 1e-13 and np.max(np.abs(lse - L)) < 1e-13


def test_value_columns_are_independent():
    # every output column uses only its own value column, and the normaliser
    # does not involve V at all: splitting V by columns splits O exactly and
    # leaves the LSE unchanged
    q, k, v = random_inputs((2, 4, 21, 12), (2, 2, 30, 12), seed=4, shape_v=(2, 2, 30, 8))
    o, lse = oracle.attention(q, k, v, scale=0.3, causal=True)
    for a, b in ((0, 3), (3, 8)):
        o2, lse2 = oracle.attention(q, k, v[..., a:b].contiguous(), scale=0.3, causal=True)
        assert np.array_equal(o2, o[..., a:b]) and np.array_equal(lse2, lse)


# ------------------------------------------------------------------ reductions

def test_gqa_equals_mha_with_repeated_kv():
    B, Hq, Hkv, L, D = 2, 8, 2, 33, 16
    q, k, v = random_inputs((B, Hq, L, D), (B, Hkv, L, D), seed=5)
    o, lse = oracle.attention(q, k, v, scale=0.25, causal=True)
    kr = k.repeat_interleave(Hq // Hkv, dim=1)
    vr = v.repeat_interleave(Hq // Hkv, dim=1)
    o2, lse2 = oracle.attention(q, kr, vr, scale=0.25, causal=True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # a wrong head map (h % Hkv instead of h // r) would differ
    kw = k.repeat(1, Hq // Hkv, 1, 1)
    vw = v.repeat(1, Hq // Hkv, 1, 1)
    o3, _ = oracle.attention(q, kw, vw, scale=0.25, causal=True)
    assert np.max(np.abs(o3 - o)) > 1e-3


def test_varlen_equals_independent_dense_calls():
    lens_q = [5, 1, 17, 9]
    lens_k = [5, 3, 17, 12]
    Hq, Hkv, D = 4, 2, 8
    Tq, Tk = sum(lens_q), sum(lens_k)
    q, k, v = random_inputs((Tq, Hq, D), (Tk, Hkv, D), seed=9)
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    for causal in (False, True):
        o, lse = oracle.attention_varlen(q, k, v, cq, ck, scale=0.3, causal=causal)
        for s in range(len(lens_q)):
            qs = q[cq[s]:cq[s + 1]].permute(1, 0, 2)[None]
            ks = k[ck[s]:ck[s + 1]].permute(1, 0, 2)[None]
            vs = v[ck[s]:ck[s + 1]].permute(1, 0, 2)[None]
            od, ld = oracle.attention(qs, ks, vs, scale=0.3, causal=causal)
            assert np.array_equal(o[cq[s]:cq[s + 1]], od[0].transpose(1, 0, 2))
            assert np.array_equal(lse[:, cq[s]:cq[s + 1]], ld[0])
        # sampled rows agree with the full evaluation
        rows = np.array([0, 7, Tq + 3, 3 * Tq + Tq - 1, 2 * Tq + 20])
        os_, ls_ = oracle.attention_varlen(q, k, v, cq, ck, scale=0.3, causal=causal, rows=rows)
        h, t = rows // Tq, rows % Tq
        assert np.array_equal(os_, o[t, h])
        assert np.array_equal(ls_, lse[h, t])


def test_sampled_rows_match_full_evaluation():
    q, k, v = random_inputs((2, 4, 40, 8), (2, 2, 50, 8), seed=1)
    o, lse = oracle.attention(q, k, v, scale=0.4, causal=True)
    rows = np.array([0, 39, 40, 151, 2 * 4 * 40 - 1])
    os_, ls_ = oracle.attention(q, k, v, scale=0.4, causal=True, rows=rows)
    assert np.array_equal(os_, o.reshape(-1, 8)[rows])
    assert np.array_equal(ls_, lse.reshape(-1)[rows])


# ----------------------------------------------- tiling, order and partitions (recurrence)

def test_online_matches_definition_on_the_pages_case():
    # 5 queries that are the final positions of a 13-token cache, blocks 3 / 4
    rng = np.random.default_rng(7)
    q = rng.standard_normal((5, 16))
    k = rng.standard_normal((13, 16))
    v = rng.standard_normal((13, 8))
    ref, ref_lse = R.definition(q, k, v, causal=True, qpos=R.positions(5, 8))[2:]
    out, lse = R.online(q, k, v, causal=True, qpos=R.positions(5, 8), query_blocks=R.blocks(5, 3),
                        key_blocks=R.blocks(13, 4))
    assert np.max(np.abs(out - ref)) < 1e-10 and np.max(np.abs(lse - ref_lse)) < 1e-10
    # the C oracle (bottom-right alignment, Lq=5, Lk=13) is the same problem
    oc, lc = c_oracle_1head(q.astype(np.float32).tolist(), k.astype(np.float32).tolist(),
                            np.pad(v, ((0, 0), (0, 8))).astype(np.float32).tolist(),
                            scale=1 / 4.0, causal=True)
    rq, rl = R.definition(q.astype(np.float32), k.astype(np.float32),
                          v.astype(np.float32), causal=True, qpos=R.positions(5, 8))[2:]
    assert np.max(np.abs(oc[:, :8] - rq)) < 1e-12 and np.max(np.abs(lc - rl)) < 1e-12


@pytest.mark.parametrize("block_q", [1, 3, 32])
@pytest.mark.parametrize("block_k", [1, 4, 64, 128])
def test_tile_size_and_order_independence(block_q, block_k):
    rng = np.random.default_rng(block_q * 1000 + block_k)
    nq, nk = 37, 150
    q = rng.standard_normal((nq, 8)) * 20  # sharp softmax (scores x 20)
    k = rng.standard_normal((nk, 8))
    v = rng.standard_normal((nk, 8))
    qpos = R.positions(nq, nk - nq)
    ref, ref_lse = R.definition(q, k, v, causal=True, qpos=qpos)[2:]
    in_order = R.blocks(nk, block_k)
    shuffled = list(in_order)
    random.Random(block_q + block_k).shuffle(shuffled)
    for key_blocks in (in_order, shuffled):
        for tau in (None, 0.0, 8 * math.log(2.0)):
            out, lse = R.online(q, k, v, causal=True, qpos=qpos, query_blocks=R.blocks(nq, block_q),
                                key_blocks=key_blocks, tau=tau)
            assert np.max(np.abs(out - ref)) < 1e-10
            assert np.max(np.abs(lse - ref_lse)) < 1e-10


def test_fully_masked_rows_are_zero_with_minus_inf_lse():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((6, 8))
    k = rng.standard_normal((9, 8))
    v = rng.standard_normal((9, 8))
    # q_start = -2: the first two query rows precede every key
    out, lse = R.online(q, k, v, causal=True, qpos=R.positions(6, -2), query_blocks=R.blocks(6, 4),
                        key_blocks=R.blocks(9, 4))
    ref, ref_lse = R.definition(q, k, v, causal=True, qpos=R.positions(6, -2))[2:]
    assert np.all(out[:2] == 0) and np.all(lse[:2] == -np.inf)
    assert np.max(np.abs(out[2:] - ref[2:])) < 1e-10
    assert np.array_equal(ref_lse[:2], lse[:2])


def test_partition_merge_in_two_orders():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((7, 8))
    k = rng.standard_normal((30, 8))
    v = rng.standard_normal((30, 8))
    sc = 1 / math.sqrt(8)
    parts = [(0, 11), (11, 12), (12, 30)]
    st = [R.RowState.from_scores(R.score_matrix(q, k[a:b], sc), v[a:b]) for a, b in parts]
    ref, ref_lse = R.definition(q, k, v)[2:]
    for merged in (R.combine(R.combine(st[0], st[1]), st[2]),
                   R.combine(st[2], R.combine(st[1], st[0]))):
        m, l, u = merged.top, merged.mass, merged.acc
        assert np.max(np.abs(u / l[:, None] - ref)) < 1e-12
        assert np.max(np.abs(m + np.log(l) - ref_lse)) < 1e-12
    # the normalised-output form with natural-log normalisers
    outs = [R.from_normalised(*R.definition(q, k[a:b], v[a:b])[2:]) for a, b in parts]
    o, L = R.combine(outs[0], outs[1]).result()
    o, L = R.combine(R.from_normalised(o, L), outs[2]).result()
    assert np.max(np.abs(o - ref)) < 1e-12 and np.max(np.abs(L - ref_lse)) < 1e-12


def test_base2_lse_conversion():
    # L2 = log2 sum 2^{s2}, with s2 = s * log2(e); L = L2 * ln 2
    s = np.array([0.3, -1.2, 2.5, 0.0])
    s2 = s * math.log2(math.e)
    L2 = math.log2(np.sum(2.0 ** s2))
    _, lse = c_oracle_1head([[1.0]], [[float(x)] for x in s.astype(np.float32)], [[1.0]] * 4, scale=1.0)
    assert abs(L2 * math.log(2.0) - float(lse[0])) < 1e-6  # s rounded to fp32 in the oracle input
