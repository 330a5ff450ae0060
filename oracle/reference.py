"""Small fp64 numpy models of attention -- TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this module.  Nothing here is shared with the CUDA path.

Every model works on one (batch, head) slice: queries ``q [n, d]`` sitting at
integer token positions ``qpos [n]``, keys ``k [m, d]`` and values
``v [m, dv]`` at positions ``kpos [m]``.  Under causal masking query i may
read key j only when ``kpos[j] <= qpos[i]``; positions are absolute, so a
slice of the keys keeps its own positions (FlashAttention from Scratch,
sec. 5 "Run the math before writing a GPU kernel").

* :func:`definition` -- the score matrix S and the probability matrix P
  materialised, then O = P V and the natural-log normaliser per row
  (sec. 2 "Begin with one attention row"; sec. 4.4 for rows with no key).
* :class:`RowState` -- what a set of keys contributes to each query row,
  summarised as a reference exponent ``top``, the mass
  ``sum_j exp(s_j - top)`` and the accumulator ``sum_j exp(s_j - top) v_j``.
  Moving a summary to a larger reference multiplies both sums by
  ``exp(old - new)`` (sec. 4.1 "Maintain three quantities"), and summaries of
  two disjoint key sets add once they share a reference (sec. 4.3 "Merge
  independently computed partitions"): :func:`combine`.
* :func:`online` -- the streaming form: each query block starts from the
  empty summary and absorbs an explicit list of key blocks in the order the
  caller gives them.  With a threshold ``tau`` the reference only moves when
  a block's maximum passes it by more than ``tau`` (sec. 11.3 "Derive
  conditional rescaling correctly"); FlashAttention Cheat Sheet, sec. 5
  "Why online softmax is globally exact" is why every order and every
  blocking gives the same answer.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import NamedTuple, Optional, Sequence

import numpy as np

NEG_INF = -np.inf


def positions(count: int, first: int = 0) -> np.ndarray:
    """Token positions first, first + 1, ..., first + count - 1."""
    return np.arange(count, dtype=np.int64) + first


def blocks(count: int, size: int) -> list:
    """Consecutive (start, stop) index ranges of at most ``size`` entries."""
    assert size > 0
    return [(a, min(count, a + size)) for a in range(0, count, size)]


def allowed(qpos: np.ndarray, kpos: np.ndarray, causal: bool) -> np.ndarray:
    """Boolean [len(qpos), len(kpos)]: may query i read key j?"""
    qpos, kpos = np.asarray(qpos), np.asarray(kpos)
    if not causal:
        return np.ones((qpos.size, kpos.size), dtype=bool)
    return kpos[None, :] <= qpos[:, None]


def score_matrix(q, k, scale: float, qpos=None, kpos=None, causal: bool = False) -> np.ndarray:
    """scale * q k^T in fp64, with -inf where the pair is masked."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    qpos = positions(q.shape[0]) if qpos is None else qpos
    kpos = positions(k.shape[0]) if kpos is None else kpos
    raw = scale * (q @ k.T)
    return np.where(allowed(qpos, kpos, causal), raw, NEG_INF)


def exp_shifted(x, ref) -> np.ndarray:
    """exp(x - ref) elementwise (broadcast), with masked entries x = -inf
    contributing exactly 0.  Wherever x is finite, ref is too."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    shape = np.broadcast(x, ref).shape
    live = np.broadcast_to(np.isfinite(x), shape)
    out = np.zeros(shape)
    np.exp(np.broadcast_to(x, shape) - np.where(live, np.broadcast_to(ref, shape), 0.0),
           out=out, where=live)
    return out


def probabilities(s) -> np.ndarray:
    """Row softmax of a score matrix; a row with every entry masked is 0."""
    s = np.asarray(s, dtype=np.float64)
    w = exp_shifted(s, s.max(axis=1, keepdims=True))
    total = w.sum(axis=1, keepdims=True)
    return np.divide(w, total, out=np.zeros_like(w), where=total > 0)


class Attn(NamedTuple):
    s: np.ndarray    # [n, m] scores, -inf where masked
    p: np.ndarray    # [n, m] probabilities, rows sum to 1 (or are all 0)
    o: np.ndarray    # [n, dv]
    lse: np.ndarray  # [n] natural-log normaliser, -inf for a row with no key


def definition(q, k, v, scale: Optional[float] = None, causal: bool = False,
               qpos=None, kpos=None) -> Attn:
    """Attention with S and P materialised.  ``scale`` defaults to 1/sqrt(d)."""
    q = np.asarray(q, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[1])
    s = score_matrix(q, k, scale, qpos, kpos, causal)
    p = probabilities(s)
    top = s.max(axis=1)
    mass = exp_shifted(s, top[:, None]).sum(axis=1)
    lse = np.full(q.shape[0], NEG_INF)
    has_key = mass > 0
    lse[has_key] = top[has_key] + np.log(mass[has_key])
    return Attn(s, p, p @ v, lse)


@dataclass
class RowState:
    """Summary of the keys seen so far, per query row (see the module notes).
    An empty row has top = -inf, mass = 0 and a zero accumulator."""
    top: np.ndarray
    mass: np.ndarray
    acc: np.ndarray

    @classmethod
    def empty(cls, rows: int, dv: int) -> "RowState":
        return cls(np.full(rows, NEG_INF), np.zeros(rows), np.zeros((rows, dv)))

    @classmethod
    def from_scores(cls, s, v, top=None) -> "RowState":
        """Summary of one block of keys with scores ``s [n, m]`` and values
        ``v [m, dv]``, on the reference ``top`` (default: the row maxima)."""
        s = np.asarray(s, dtype=np.float64)
        top = s.max(axis=1) if top is None else np.asarray(top, dtype=np.float64)
        w = exp_shifted(s, top[:, None])
        return cls(top.copy(), w.sum(axis=1), w @ np.asarray(v, dtype=np.float64))

    def rebased(self, new_top) -> "RowState":
        """The same summary expressed on the reference ``new_top`` >= top."""
        factor = exp_shifted(self.top, new_top)
        return RowState(np.asarray(new_top, dtype=np.float64).copy(), self.mass * factor,
                        self.acc * factor[:, None])

    def copy(self) -> "RowState":
        return RowState(self.top.copy(), self.mass.copy(), self.acc.copy())

    def result(self):
        """(o, lse): o = acc / mass and lse = top + ln(mass); an empty row
        gives o = 0 and lse = -inf."""
        has_key = self.mass > 0
        o = np.zeros_like(self.acc)
        o[has_key] = self.acc[has_key] / self.mass[has_key, None]
        lse = np.full(self.mass.shape, NEG_INF)
        lse[has_key] = self.top[has_key] + np.log(self.mass[has_key])
        return o, lse


def combine(a: RowState, b: RowState) -> RowState:
    """Summary of the union of two disjoint key sets."""
    top = np.maximum(a.top, b.top)
    ra, rb = a.rebased(top), b.rebased(top)
    return RowState(top, ra.mass + rb.mass, ra.acc + rb.acc)


def from_normalised(o, lse) -> RowState:
    """A finished partial result read back as a summary: with reference
    lse the mass of a non-empty row is exactly 1 and its accumulator is o."""
    lse = np.asarray(lse, dtype=np.float64)
    mass = np.isfinite(lse).astype(np.float64)
    return RowState(lse.copy(), mass, np.asarray(o, dtype=np.float64) * mass[:, None])


def online(q, k, v, scale: Optional[float] = None, causal: bool = False, qpos=None, kpos=None,
           key_blocks: Optional[Sequence] = None, query_blocks: Optional[Sequence] = None,
           tau: Optional[float] = None, history: Optional[list] = None):
    """Streaming attention over explicit key blocks; returns (o, lse).

    ``key_blocks`` lists (start, stop) ranges of keys, visited in list order
    (default: one block of all keys); ``query_blocks`` splits the queries the
    same way.  ``tau`` (natural-log units) keeps a row's reference while the
    block maximum stays within ``tau`` of it; ``None`` always moves it to the
    running maximum.  ``history`` (a list) receives a copy of the first query
    block's summary after every key block.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[1])
    qpos = positions(q.shape[0]) if qpos is None else np.asarray(qpos)
    kpos = positions(k.shape[0]) if kpos is None else np.asarray(kpos)
    key_blocks = [(0, k.shape[0])] if key_blocks is None else list(key_blocks)
    query_blocks = [(0, q.shape[0])] if query_blocks is None else list(query_blocks)
    covered = sorted(j for a, b in key_blocks for j in range(a, b))
    assert covered == list(range(k.shape[0])), "key blocks must cover every key once"

    o = np.zeros((q.shape[0], v.shape[1]))
    lse = np.full(q.shape[0], NEG_INF)
    for n_qb, (r0, r1) in enumerate(query_blocks):
        state = RowState.empty(r1 - r0, v.shape[1])
        for a, b in key_blocks:
            s = score_matrix(q[r0:r1], k[a:b], scale, qpos[r0:r1], kpos[a:b], causal)
            block_top = s.max(axis=1)
            running = np.maximum(state.top, block_top)
            if tau is None:
                top = running
            else:
                stay = np.isfinite(state.top) & (block_top <= state.top + tau)
                top = np.where(stay, state.top, running)
            old, new = state.rebased(top), RowState.from_scores(s, v[a:b], top)
            state = RowState(top, old.mass + new.mass, old.acc + new.acc)
            if history is not None and n_qb == 0:
                history.append(state.copy())
        o[r0:r1], lse[r0:r1] = state.result()
    return o, lse
