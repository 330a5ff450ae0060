"""Exact attention forward on GB300 (sm_103a): Python binding of libfa_gb300.

The functions here only marshal arguments (tensor pointers, sizes, the
current CUDA stream) into the C ABI declared in ``include/fa_gb300.h``; every
step of the computation runs in the library's CUDA kernels.  There is no CPU
or eager-PyTorch fallback: if the library is missing or the device is not an
sm_103 GPU the call raises.

    o, lse = fa_fwd(q, k, v, causal=True)          # q [B,Hq,Lq,D], k/v [B,Hkv,Lk,D]
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max_q, max_k, causal=True)
    o, lse = fa_fwd_splitkv(q, k, v, causal=True)    # decode: (Hq/Hkv)*Lq <= 16, long Lk
    dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal=True)
    o, lse = fa_fwd_variant(q, k, v, window=(4095, 0), softcap=0.0, alibi_slopes=None)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = ["fa_fwd", "fa_fwd_varlen", "fa_fwd_hdim", "fa_fwd_varlen_hdim", "fa_fwd_varlen_noalloc", "fa_fwd_variant", "fa_fwd_varlen_variant",
           "fa_fwd_splitkv", "fp8_prepare", "fa_fwd_fp8", "fp8_sections", "splitkv_workspace", "fa_bwd",
           "bwd_workspace", "fa_bwd_varlen", "bwd_varlen_workspace", "fa_bwd_variant", "fa_bwd_varlen_variant", "fa_check", "fa_status_string", "fa_last_launch_count",
           "FAError", "library_path", "load_library", "EXPORTED_SYMBOLS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")
_lock = threading.Lock()
_lib = None

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
EXPORTED_SYMBOLS = ("fa_fwd", "fa_fwd_varlen", "fa_fwd_hdim", "fa_fwd_varlen_hdim", "fa_fwd_varlen_noalloc", "fa_fwd_variant", "fa_fwd_varlen_variant",
                    "fa_fwd_splitkv", "fa_fwd_splitkv_workspace", "fa_bwd", "fa_bwd_workspace", "fa_bwd_varlen",
                    "fa_bwd_varlen_workspace", "fa_bwd_variant", "fa_bwd_varlen_variant", "fa_fp8_workspace",
                    "fa_fp8_prepare", "fa_fwd_fp8", "fa_check", "fa_status_string", "fa_last_launch_count",
                    "fa_test_inject_fault")
SPLITKV_MAX_ROWS = 16  # (Hq / Hkv) * Lq limit of fa_fwd_splitkv
NOALLOC_MAX_SEQS = 16384  # FA_NOALLOC_MAX_SEQS in include/fa_gb300.h
VARLEN_SEQS_PER_LAUNCH = 1536  # FA_VARLEN_SEQS_PER_LAUNCH (64 for head dimensions (192, 128))


class _Variant(ctypes.Structure):
    # struct fa_variant in include/fa_gb300.h
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int), ("softcap", ctypes.c_float),
                ("alibi_slopes", ctypes.c_void_p)]


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libfa_gb300.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_fwd.restype = i
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
        lib.fa_fwd_varlen.restype = i
        lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, vp]
        lib.fa_fwd_hdim.restype = i
        lib.fa_fwd_hdim.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp]
        lib.fa_fwd_varlen_hdim.restype = i
        lib.fa_fwd_varlen_hdim.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, i, f, vp]
        lib.fa_fwd_varlen_noalloc.restype = i
        lib.fa_fwd_varlen_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, vp]
        lib.fa_fwd_splitkv.restype = i
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv_workspace.restype = i
        lib.fa_fwd_splitkv_workspace.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t),
                                                 ctypes.POINTER(ctypes.c_int)]
        vr = ctypes.POINTER(_Variant)
        lib.fa_fwd_variant.restype = i
        lib.fa_fwd_variant.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vr, f, vp]
        lib.fa_fwd_varlen_variant.restype = i
        lib.fa_fwd_varlen_variant.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vr, f, vp]
        lib.fa_fp8_workspace.restype = i
        lib.fa_fp8_workspace.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_fp8_prepare.restype = i
        lib.fa_fp8_prepare.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_fp8.restype = i
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, vp]
        lib.fa_bwd.restype = i
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
        lib.fa_bwd_workspace.restype = i
        lib.fa_bwd_workspace.argtypes = [i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_bwd_varlen.restype = i
        lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, vp,
                                      ctypes.c_size_t, vp]
        lib.fa_bwd_variant.restype = i
        lib.fa_bwd_variant.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vr, f, vp, ctypes.c_size_t,
                                       vp]
        lib.fa_bwd_varlen_variant.restype = i
        lib.fa_bwd_varlen_variant.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vr,
                                              f, vp, ctypes.c_size_t, vp]
        lib.fa_bwd_varlen_workspace.restype = i
        lib.fa_bwd_varlen_workspace.argtypes = [i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_check.restype = i
        lib.fa_check.argtypes = [vp]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_status_string.argtypes = [i]
        lib.fa_last_launch_count.restype = i
        lib.fa_last_launch_count.argtypes = []
        lib.fa_test_inject_fault.restype = None
        lib.fa_test_inject_fault.argtypes = [i]
        _lib = lib
        return lib


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_last_launch_count() -> int:
    return int(load_library().fa_last_launch_count())


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check_tensor(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int, on_device: bool = True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if on_device and t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
           softmax_scale: float | None = None, out: torch.Tensor | None = None,
           lse: torch.Tensor | None = None, stream=None):
    """Dense attention forward.  q [B,Hq,Lq,D], k/v [B,Hkv,Lk,D] bf16 CUDA.

    Returns (o [B,Hq,Lq,D] fp32, lse [B,Hq,Lq] fp32).  Asynchronous on the
    current (or given) stream.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, torch.bfloat16, 4)
    B, Hq, Lq, D = q.shape
    Bk, Hkv, Lk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    _check_tensor(out, "out", torch.float32, 4)
    if tuple(out.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Lq):
        raise ValueError("out/lse shape mismatch")
    _check_tensor(lse, "lse", torch.float32, 3)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                        B, Hq, Hkv, Lq, Lk, D, int(bool(causal)), float(softmax_scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd")
    return out, lse


def _check_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, out, lse):
    """Dtypes, ranks, layouts and shapes of a packed call (q [Tq,Hq,D], k and
    v [Tk,Hkv,D], offsets of equal length, out [Tq,Hq,D], lse [Hq,Tq]) first,
    then that every tensor lives on a CUDA device.  Returns (Tq, Hq, D, Tk, Hkv)."""
    named = [(q, "q", torch.bfloat16, 3), (k, "k", torch.bfloat16, 3), (v, "v", torch.bfloat16, 3),
             (cu_seqlens_q, "cu_seqlens_q", torch.int32, 1), (cu_seqlens_k, "cu_seqlens_k", torch.int32, 1),
             (out, "out", torch.float32, 3), (lse, "lse", torch.float32, 2)]
    for t, n, dt, nd in named:
        _check_tensor(t, n, dt, nd, on_device=False)
    Tq, Hq, D = q.shape
    Tk, Hkv, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Dk != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold num_seqs + 1 >= 2 offsets")
    if tuple(out.shape) != tuple(q.shape) or tuple(lse.shape) != (Hq, Tq):
        raise ValueError(f"out must be {tuple(q.shape)} and lse {(Hq, Tq)}, got {tuple(out.shape)} and "
                         f"{tuple(lse.shape)}")
    for t, n, _, _ in named:
        if t.device.type != "cuda":
            raise ValueError(f"{n} must be a CUDA tensor")
    return Tq, Hq, D, Tk, Hkv


def fa_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                  cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, causal: bool = False,
                  softmax_scale: float | None = None, out: torch.Tensor | None = None,
                  lse: torch.Tensor | None = None, stream=None):
    """Packed variable-length forward.  q [Tq,Hq,D], k/v [Tk,Hkv,D] bf16 CUDA,
    cu_seqlens_* int32 CUDA [num_seqs+1].  Returns (o [Tq,Hq,D] fp32, lse [Hq,Tq] fp32).
    Allocates nothing on the device beyond ``out``/``lse`` when they are not given."""
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    Tq, Hq, D, Tk, Hkv = _check_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, out, lse)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), cu_seqlens_q.numel() - 1,
                               Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, int(bool(causal)),
                               float(softmax_scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_varlen")
    return out, lse


def fa_fwd_hdim(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                softmax_scale: float | None = None, out: torch.Tensor | None = None,
                lse: torch.Tensor | None = None, stream=None):
    """Dense forward whose value head dimension Dv may differ from the
    query/key one D.  q [B,Hq,Lq,D], k [B,Hkv,Lk,D], v [B,Hkv,Lk,Dv] bf16 CUDA;
    (D, Dv) in {(64, 64), (128, 128), (192, 128)}.

    Returns (o [B,Hq,Lq,Dv] fp32, lse [B,Hq,Lq] fp32).  The default scale is
    1/sqrt(D).
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, torch.bfloat16, 4)
    B, Hq, Lq, D = q.shape
    Bk, Hkv, Lk, Dk = k.shape
    Dv = v.shape[3]
    if tuple(v.shape[:3]) != tuple(k.shape[:3]) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if out is None:
        out = torch.empty((B, Hq, Lq, Dv), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    _check_tensor(out, "out", torch.float32, 4)
    _check_tensor(lse, "lse", torch.float32, 3)
    if tuple(out.shape) != (B, Hq, Lq, Dv) or tuple(lse.shape) != (B, Hq, Lq):
        raise ValueError("out/lse shape mismatch")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_hdim(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                             B, Hq, Hkv, Lq, Lk, D, Dv, int(bool(causal)), float(softmax_scale),
                             _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_hdim")
    return out, lse


def fa_fwd_varlen_hdim(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                       cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, causal: bool = False,
                       softmax_scale: float | None = None, out: torch.Tensor | None = None,
                       lse: torch.Tensor | None = None, stream=None):
    """Packed forward with value head dimension Dv: q [Tq,Hq,D], k [Tk,Hkv,D],
    v [Tk,Hkv,Dv] bf16 CUDA.  Returns (o [Tq,Hq,Dv] fp32, lse [Hq,Tq] fp32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, torch.bfloat16, 3)
    _check_tensor(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check_tensor(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    Tq, Hq, D = q.shape
    Tk, Hkv, Dk = k.shape
    Dv = v.shape[2]
    if tuple(v.shape[:2]) != (Tk, Hkv) or Dk != D or cu_seqlens_q.numel() != cu_seqlens_k.numel():
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((Tq, Hq, Dv), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    _check_tensor(out, "out", torch.float32, 3)
    _check_tensor(lse, "lse", torch.float32, 2)
    if tuple(out.shape) != (Tq, Hq, Dv) or tuple(lse.shape) != (Hq, Tq):
        raise ValueError("out/lse shape mismatch")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_varlen_hdim(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                    cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), cu_seqlens_q.numel() - 1,
                                    Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, Dv,
                                    int(bool(causal)), float(softmax_scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_varlen_hdim")
    return out, lse


def fa_fwd_varlen_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                          cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, out: torch.Tensor,
                          lse: torch.Tensor, causal: bool = False, softmax_scale: float | None = None,
                          stream=None):
    """Packed forward for callers that cannot call cudaMalloc on the hot path
    (a process whose device memory all belongs to its own allocator, a server
    that must not allocate while serving): the caller provides ``out`` and
    ``lse``, and the whole batch's schedule (at most NOALLOC_MAX_SEQS
    sequences) goes into a fixed array inside the library, so one attention
    launch covers it.  Calls that can overlap on the GPU share that array and
    must be ordered.  Every shape is checked before the library is touched."""
    Tq, Hq, D, Tk, Hkv = _check_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, out, lse)
    if cu_seqlens_q.numel() - 1 > NOALLOC_MAX_SEQS:
        raise ValueError(f"at most {NOALLOC_MAX_SEQS} sequences")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_varlen_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                       cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), cu_seqlens_q.numel() - 1,
                                       Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, int(bool(causal)),
                                       float(softmax_scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_varlen_noalloc")
    return out, lse


def _variant(window, softcap, alibi_slopes, Hq: int, device):
    if alibi_slopes is not None:
        _check_tensor(alibi_slopes, "alibi_slopes", torch.float32, 1)
        if alibi_slopes.numel() != Hq or alibi_slopes.device != device:
            raise ValueError("alibi_slopes must be a float32 tensor of Hq elements on the inputs' device")
    wl, wr = window
    return _Variant(int(wl), int(wr), float(softcap), alibi_slopes.data_ptr() if alibi_slopes is not None else None)


def fa_fwd_variant(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window=(-1, -1), softcap: float = 0.0,
                   alibi_slopes: torch.Tensor | None = None, softmax_scale: float | None = None,
                   out: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """Dense forward with a key window (left, right) around each query's
    bottom-right-aligned position (-1 = unlimited), soft-capping of the
    scaled scores, or ALiBi slopes per query head.  D = 64 or 128."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, torch.bfloat16, 4)
    B, Hq, Lq, D = q.shape
    Bk, Hkv, Lk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError("shape mismatch")
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out is None else out
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor(out, "out", torch.float32, 4)
    _check_tensor(lse, "lse", torch.float32, 3)
    if tuple(out.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Lq):
        raise ValueError("out/lse shape mismatch")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    var = _variant(window, softcap, alibi_slopes, Hq, q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_variant(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq,
                                Hkv, Lq, Lk, D, ctypes.byref(var), float(softmax_scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_variant")
    return out, lse


def fa_fwd_varlen_variant(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                          cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, window=(-1, -1),
                          softcap: float = 0.0, alibi_slopes: torch.Tensor | None = None,
                          softmax_scale: float | None = None, out: torch.Tensor | None = None,
                          lse: torch.Tensor | None = None, stream=None):
    """Packed forward with a variant; windows and distances are per sequence."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, torch.bfloat16, 3)
    _check_tensor(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check_tensor(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out is None else out
    lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor(out, "out", torch.float32, 3)
    _check_tensor(lse, "lse", torch.float32, 2)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    var = _variant(window, softcap, alibi_slopes, Hq, q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_varlen_variant(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                       cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), cu_seqlens_q.numel() - 1,
                                       Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, ctypes.byref(var),
                                       float(softmax_scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_varlen_variant")
    return out, lse


def fp8_sections(B: int, Hq: int, Hkv: int, Lq: int, Lk: int) -> dict:
    """Byte offsets and shapes of the sections of a prepared FP8 buffer (the
    layout documented with fa_fp8_prepare in include/fa_gb300.h)."""
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    nq, nk = (Lq + 127) // 128, (Lk + 127) // 128
    lk_pad = nk * 128
    sec, off = {}, 0
    for name, nbytes, shape in (("qc", B * Hq * Lq * 128, (B, Hq, Lq, 128)), ("kc", B * Hkv * Lk * 128, (B, Hkv, Lk, 128)),
                                ("vt", B * Hkv * 128 * lk_pad, (B, Hkv, 128, lk_pad)), ("sq", B * Hq * nq * 4, (B, Hq, nq)),
                                ("sk", B * Hkv * nk * 4, (B, Hkv, nk)), ("sv", B * Hkv * 4, (B, Hkv)),
                                ("vmax", B * Hkv * 4, (B, Hkv))):
        sec[name] = (off, nbytes, shape)
        off = up(off + nbytes)
    sec["total"] = off
    return sec


def fp8_prepare(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, signs: torch.Tensor,
                prepared: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Rotate and quantise bf16 q [B,Hq,Lq,128], k/v [B,Hkv,Lk,128] for
    fa_fwd_fp8; signs: fp32 CUDA [128] of +-1.  Returns the prepared buffer
    (a CUDA uint8 tensor)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, torch.bfloat16, 4)
    _check_tensor(signs, "signs", torch.float32, 1)
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    lib = load_library()
    n = ctypes.c_size_t(0)
    st = lib.fa_fp8_workspace(B, Hq, Hkv, Lq, Lk, D, ctypes.byref(n))
    if st != FA_OK:
        raise FAError(st, "fa_fp8_workspace")
    if prepared is None or prepared.numel() < n.value:
        prepared = torch.empty(n.value, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = lib.fa_fp8_prepare(q.data_ptr(), k.data_ptr(), v.data_ptr(), signs.data_ptr(), B, Hq, Hkv, Lq, Lk, D,
                                prepared.data_ptr(), prepared.numel(), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fp8_prepare")
    return prepared


def fa_fwd_fp8(prepared: torch.Tensor, B: int, Hq: int, Hkv: int, Lq: int, Lk: int, causal: bool = False,
               softmax_scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
               D: int = 128, stream=None):
    """Attention of a buffer made by fp8_prepare.  Returns (o fp32 [B,Hq,Lq,D], lse fp32 [B,Hq,Lq])."""
    out = torch.empty((B, Hq, Lq, D), dtype=torch.float32, device=prepared.device) if out is None else out
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=prepared.device) if lse is None else lse
    _check_tensor(out, "out", torch.float32, 4)
    _check_tensor(lse, "lse", torch.float32, 3)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(prepared.device):
        st = lib.fa_fwd_fp8(prepared.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Lq, Lk, D,
                            int(bool(causal)), float(softmax_scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    return out, lse


def splitkv_workspace(B: int, Hq: int, Hkv: int, Lq: int, Lk: int, D: int, num_splits: int = 0) -> tuple[int, int]:
    """(workspace bytes, partitions) fa_fwd_splitkv uses for this shape on the current device."""
    nbytes, used = ctypes.c_size_t(0), ctypes.c_int(0)
    st = load_library().fa_fwd_splitkv_workspace(B, Hq, Hkv, Lq, Lk, D, int(num_splits), ctypes.byref(nbytes),
                                                 ctypes.byref(used))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_splitkv_workspace")
    return int(nbytes.value), int(used.value)


def fa_fwd_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                   softmax_scale: float | None = None, num_splits: int = 0, out: torch.Tensor | None = None,
                   lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """Split-KV (decode) forward.  q [B,Hq,Lq,D], k/v [B,Hkv,Lk,D] bf16 CUDA with
    (Hq/Hkv)*Lq <= 16.  ``num_splits`` <= 0 lets the library choose.  The
    partial-result workspace is taken from ``workspace`` (a CUDA uint8 tensor)
    or allocated here through PyTorch.  Returns (o fp32, lse fp32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, torch.bfloat16, 4)
    B, Hq, Lq, D = q.shape
    Bk, Hkv, Lk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    _check_tensor(out, "out", torch.float32, 4)
    _check_tensor(lse, "lse", torch.float32, 3)
    if tuple(out.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Lq):
        raise ValueError("out/lse shape mismatch")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q.device):
        nbytes, _ = splitkv_workspace(B, Hq, Hkv, Lq, Lk, D, num_splits)
        if nbytes and (workspace is None or workspace.numel() * workspace.element_size() < nbytes):
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if (nbytes and workspace is not None) else None
        ws_len = workspace.numel() * workspace.element_size() if ws_ptr else 0
        st = lib.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                B, Hq, Hkv, Lq, Lk, D, int(bool(causal)), float(softmax_scale), int(num_splits),
                                ws_ptr, ws_len, _stream_handle(stream))
        if ws_ptr and isinstance(stream, torch.cuda.Stream):
            workspace.record_stream(stream)  # keep the block out of reuse until that stream is done
    if st != FA_OK:
        raise FAError(st, "fa_fwd_splitkv")
    return out, lse


def bwd_workspace(B: int, Hq: int, Lq: int) -> int:
    """Workspace bytes fa_bwd needs."""
    nbytes = ctypes.c_size_t(0)
    st = load_library().fa_bwd_workspace(B, Hq, Lq, ctypes.byref(nbytes))
    if st != FA_OK:
        raise FAError(st, "fa_bwd_workspace")
    return int(nbytes.value)


def fa_bwd_variant(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
                   dout: torch.Tensor, window=(-1, -1), softcap: float = 0.0,
                   alibi_slopes: torch.Tensor | None = None, softmax_scale: float | None = None,
                   dq: torch.Tensor | None = None, dk: torch.Tensor | None = None, dv: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, stream=None):
    """Backward of fa_fwd_variant for key windows, soft-capping and ALiBi
    (D = 64 or 128); o and lse from fa_fwd_variant with the same variant."""
    var = _variant(window, softcap, alibi_slopes, q.shape[1], q.device)
    return fa_bwd(q, k, v, o, lse, dout, False, softmax_scale, dq, dk, dv, workspace, stream, variant=var)


def fa_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
           dout: torch.Tensor, causal: bool = False, softmax_scale: float | None = None,
           dq: torch.Tensor | None = None, dk: torch.Tensor | None = None, dv: torch.Tensor | None = None,
           workspace: torch.Tensor | None = None, stream=None, variant=None):
    """Backward of fa_fwd.  q/dout [B,Hq,Lq,D], k/v [B,Hkv,Lk,D] bf16; o fp32
    [B,Hq,Lq,D] and lse fp32 [B,Hq,Lq] from fa_fwd.  Returns (dq, dk, dv) fp32."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _check_tensor(t, n, torch.bfloat16, 4)
    _check_tensor(o, "o", torch.float32, 4)
    _check_tensor(lse, "lse", torch.float32, 3)
    B, Hq, Lq, D = q.shape
    Bk, Hkv, Lk, Dk = k.shape
    if (tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D or tuple(dout.shape) != tuple(q.shape)
            or tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Lq)):
        raise ValueError("shape mismatch")
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device) if dv is None else dv
    for t, n, shp in ((dq, "dq", q.shape), (dk, "dk", k.shape), (dv, "dv", k.shape)):
        _check_tensor(t, n, torch.float32, 4)
        if tuple(t.shape) != tuple(shp):
            raise ValueError(f"{n} shape mismatch")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q.device):
        nbytes = bwd_workspace(B, Hq, Lq)
        if workspace is None or workspace.numel() * workspace.element_size() < nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Lq, Lk, D)
        tail = (float(softmax_scale), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                _stream_handle(stream))
        if variant is None:
            st, name = lib.fa_bwd(*args, int(bool(causal)), *tail), "fa_bwd"
        else:
            st, name = lib.fa_bwd_variant(*args, ctypes.byref(variant), *tail), "fa_bwd_variant"
        if isinstance(stream, torch.cuda.Stream):
            workspace.record_stream(stream)
    if st != FA_OK:
        raise FAError(st, name)
    return dq, dk, dv


def bwd_varlen_workspace(num_seqs: int, total_q: int, Hq: int) -> int:
    """Workspace bytes fa_bwd_varlen needs."""
    nbytes = ctypes.c_size_t(0)
    st = load_library().fa_bwd_varlen_workspace(num_seqs, total_q, Hq, ctypes.byref(nbytes))
    if st != FA_OK:
        raise FAError(st, "fa_bwd_varlen_workspace")
    return int(nbytes.value)


def fa_bwd_varlen_variant(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
                          dout: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                          max_seqlen_q: int, max_seqlen_k: int, window=(-1, -1), softcap: float = 0.0,
                          alibi_slopes: torch.Tensor | None = None, softmax_scale: float | None = None,
                          dq: torch.Tensor | None = None, dk: torch.Tensor | None = None,
                          dv: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """Backward of fa_fwd_varlen_variant for key windows, soft-capping and
    ALiBi (D = 64 or 128)."""
    var = _variant(window, softcap, alibi_slopes, q.shape[1], q.device)
    return fa_bwd_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, False,
                         softmax_scale, dq, dk, dv, workspace, stream, variant=var)


def fa_bwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
                  dout: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, max_seqlen_q: int,
                  max_seqlen_k: int, causal: bool = False, softmax_scale: float | None = None,
                  dq: torch.Tensor | None = None, dk: torch.Tensor | None = None, dv: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, stream=None, variant=None):
    """Backward of fa_fwd_varlen.  q/dout [Tq,Hq,D], k/v [Tk,Hkv,D] bf16; o fp32
    [Tq,Hq,D] and lse fp32 [Hq,Tq] from fa_fwd_varlen; cu_seqlens_* int32 CUDA.
    Returns (dq, dk, dv) fp32 in the layouts of q, k and v."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _check_tensor(t, n, torch.bfloat16, 3)
    _check_tensor(o, "o", torch.float32, 3)
    _check_tensor(lse, "lse", torch.float32, 2)
    _check_tensor(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check_tensor(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    Tq, Hq, D = q.shape
    Tk, Hkv, Dk = k.shape
    if (tuple(v.shape) != tuple(k.shape) or Dk != D or tuple(dout.shape) != tuple(q.shape)
            or tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != (Hq, Tq)
            or cu_seqlens_q.numel() != cu_seqlens_k.numel()):
        raise ValueError("shape mismatch")
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device) if dv is None else dv
    for t, n, shp in ((dq, "dq", q.shape), (dk, "dk", k.shape), (dv, "dv", k.shape)):
        _check_tensor(t, n, torch.float32, 3)
        if tuple(t.shape) != tuple(shp):
            raise ValueError(f"{n} shape mismatch")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    n_seqs = cu_seqlens_q.numel() - 1
    lib = load_library()
    with torch.cuda.device(q.device):
        nbytes = bwd_varlen_workspace(n_seqs, Tq, Hq)
        if workspace is None or workspace.numel() * workspace.element_size() < nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                n_seqs, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D)
        tail = (float(softmax_scale), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                _stream_handle(stream))
        if variant is None:
            st, name = lib.fa_bwd_varlen(*args, int(bool(causal)), *tail), "fa_bwd_varlen"
        else:
            st, name = lib.fa_bwd_varlen_variant(*args, ctypes.byref(variant), *tail), "fa_bwd_varlen_variant"
        if isinstance(stream, torch.cuda.Stream):
            workspace.record_stream(stream)
    if st != FA_OK:
        raise FAError(st, name)
    return dq, dk, dv


def fa_check(stream=None) -> int:
    """Synchronise the stream and raise if a kernel latched an error."""
    st = load_library().fa_check(_stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_check")
    return st
