"""fp64 CPU oracle for exact attention forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never imports it, and it imports nothing from the product.

* :func:`attention` -- the plain definition (materialised S and P, fp64) for
  dense ``[B, Hq, Lq, D]`` inputs, via the C routine in ``attention_ref.c``;
  ``rows`` restricts it to selected output rows so full-size problems can be
  checked on a sample.
* :func:`attention_varlen` -- the same for packed ``[T, H, D]`` batches with
  ``cu_seqlens`` prefix offsets: each sequence is an independent problem.
* :mod:`oracle.reference` -- small numpy models (definition and the
  online-softmax recurrence) used to pin the oracle to the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle_attention.so")
_SRC = os.path.join(_HERE, "attention_ref.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle in-tree with gcc (portable C, no ISA flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_attention_rows.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, i64p, i64p, i64p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_num_cpus.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_cpus() -> int:
    return int(_load().oracle_num_cpus())


def _as_f32(x) -> np.ndarray:
    """Exact fp32 copy of a bf16/fp32 torch tensor or array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _strides4(a: np.ndarray):
    """Element strides (b, h, i) of a [B, H, L, D] float32 array."""
    return (ctypes.c_int64 * 3)(*(s // 4 for s in a.strides[:3]))


def _run(qf, kf, vf, qs, ks, vs, B, Hq, Hkv, Lq, Lk, D, Dv, causal, scale, rows, nthreads):
    lib = _load()
    if rows is None:
        n = B * Hq * Lq
        rows_ptr = None
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows.size
        rows_ptr = rows.ctypes.data
    o = np.empty((n, Dv), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    if n == 0:
        return o, lse
    rc = lib.oracle_attention_rows(qf.ctypes.data, kf.ctypes.data, vf.ctypes.data, qs, ks, vs,
                                   B, Hq, Hkv, Lq, Lk, D, Dv, int(bool(causal)), float(scale),
                                   rows_ptr, n, o.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed with code {rc}")
    return o, lse


def attention(q, k, v, scale: float, causal: bool = False, rows=None, nthreads: int = 0):
    """Dense oracle.  q [B,Hq,Lq,D], k [B,Hkv,Lk,D], v [B,Hkv,Lk,Dv] (bf16 or
    fp32); Dv may differ from D.

    Returns (o, lse) in fp64: o [B,Hq,Lq,Dv] and lse [B,Hq,Lq] when ``rows`` is
    None, else o [n, Dv] and lse [n] for the flat row ids
    ``(b*Hq + h)*Lq + i`` in ``rows``.
    """
    qf, kf, vf = _as_f32(q), _as_f32(k), _as_f32(v)
    B, Hq, Lq, D = qf.shape
    _, Hkv, Lk, Dk = kf.shape
    Dv = vf.shape[3]
    if Dk != D or vf.shape[:3] != kf.shape[:3]:
        raise ValueError("shape mismatch between q, k and v")
    o, lse = _run(qf, kf, vf, _strides4(qf), _strides4(kf), _strides4(vf),
                  B, Hq, Hkv, Lq, Lk, D, Dv, causal, scale, rows, nthreads)
    if rows is None:
        return o.reshape(B, Hq, Lq, Dv), lse.reshape(B, Hq, Lq)
    return o, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool = False,
                     rows=None, nthreads: int = 0):
    """Packed oracle.  q [Tq,Hq,D], k [Tk,Hkv,D], v [Tk,Hkv,Dv]; sequence s spans tokens
    cu_seqlens[s]:cu_seqlens[s+1].  Causal masks are local to each sequence.

    Returns o [Tq,Hq,Dv] and lse [Hq,Tq] (fp64) when ``rows`` is None, else
    o [n,Dv] and lse [n] for flat ids ``h*Tq + t`` in ``rows``.
    """
    qf, kf, vf = _as_f32(q), _as_f32(k), _as_f32(v)
    Tq, Hq, D = qf.shape
    Hkv = kf.shape[1]
    Dv = vf.shape[2]
    cq = [int(x) for x in np.asarray(cu_seqlens_q).tolist()]
    ck = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
    if rows is None:
        o = np.zeros((Tq, Hq, Dv), dtype=np.float64)
        lse = np.full((Hq, Tq), -np.inf, dtype=np.float64)
    else:
        rows = np.asarray(rows, dtype=np.int64)
        o = np.zeros((rows.size, Dv), dtype=np.float64)
        lse = np.full((rows.size,), -np.inf, dtype=np.float64)
    for s in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[s], cq[s + 1], ck[s], ck[s + 1]
        Lq, Lk = q1 - q0, k1 - k0
        if Lq <= 0:
            continue
        if Lk <= 0:  # no keys at all: every row is empty (o = 0, lse = -inf)
            continue
        # element (b=0, h, i, d) of sequence s in the packed layout
        qs = (ctypes.c_int64 * 3)(0, qf.strides[1] // 4, qf.strides[0] // 4)
        ks = (ctypes.c_int64 * 3)(0, kf.strides[1] // 4, kf.strides[0] // 4)
        vs = (ctypes.c_int64 * 3)(0, vf.strides[1] // 4, vf.strides[0] // 4)
        qv, kv, vv = qf[q0:q1], kf[k0:k1], vf[k0:k1]
        if rows is None:
            os_, ls_ = _run(qv, kv, vv, qs, ks, vs, 1, Hq, Hkv, Lq, Lk, D, Dv, causal, scale,
                            None, nthreads)
            o[q0:q1] = os_.reshape(Hq, Lq, Dv).transpose(1, 0, 2)
            lse[:, q0:q1] = ls_.reshape(Hq, Lq)
        else:
            h = rows // Tq
            t = rows % Tq
            sel = np.nonzero((t >= q0) & (t < q1))[0]
            if sel.size == 0:
                continue
            local = h[sel] * Lq + (t[sel] - q0)
            os_, ls_ = _run(qv, kv, vv, qs, ks, vs, 1, Hq, Hkv, Lq, Lk, D, Dv, causal, scale,
                            local, nthreads)
            o[sel] = os_
            lse[sel] = ls_
    return o, lse
