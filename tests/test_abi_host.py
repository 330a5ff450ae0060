"""C ABI checks that need no GPU: the library loads, exports every function
include/fa_gb300.h declares, and rejects bad arguments before touching the
device."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import exact_attention_07_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_07_gb300 import _build
    _build.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert set(declared_functions()) == set(fa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, f"{name} not exported"
        assert hasattr(lib, name)


def test_status_strings(lib):
    for code in range(5):
        assert fa.fa_status_string(code)
    assert fa.fa_status_string(99) == "unknown status"


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, B=1, Hq=2, Hkv=1, Lq=8, Lk=8, D=64, causal=0, scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, D, causal, scale, None)


def test_dense_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, q=None) == INV
    assert _fwd(lib, lse=None) == INV
    assert _fwd(lib, B=0) == INV
    assert _fwd(lib, Lq=-1) == INV
    assert _fwd(lib, Lk=0) == INV
    assert _fwd(lib, Hq=3, Hkv=2) == INV             # Hq % Hkv != 0
    assert _fwd(lib, scale=0.0) == INV
    assert _fwd(lib, scale=float("nan")) == INV
    assert _fwd(lib, scale=float("inf")) == INV
    assert _fwd(lib, q=24) == INV                    # not 16-byte aligned
    assert _fwd(lib, D=96) == UNS
    assert _fwd(lib, D=256) == UNS
    assert lib.fa_last_launch_count() == 0


def test_varlen_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED

    def call(cu_q=32, cu_k=32, n=2, tq=10, tk=10, mq=8, mk=8, Hq=2, Hkv=2, D=128, scale=0.1):
        return lib.fa_fwd_varlen(16, 16, 16, 16, 16, cu_q, cu_k, n, tq, tk, mq, mk, Hq, Hkv, D, 1, scale, None)

    assert call(cu_q=None) == INV
    assert call(n=0) == INV
    assert call(tq=0) == INV
    assert call(mk=0) == INV
    assert call(Hq=4, Hkv=3) == INV
    assert call(cu_k=34) == INV                      # int32 offsets must be 4-byte aligned
    assert call(scale=-1.0) == INV
    assert call(D=80) == UNS


def test_noalloc_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED

    def call(q=16, cu_q=32, n=2, tq=10, tk=10, Hq=2, Hkv=2, D=128):
        return lib.fa_fwd_varlen_noalloc(q, 16, 16, 16, 16, cu_q, 32, n, tq, tk, 8, 8, Hq, Hkv, D, 1,
                                         ctypes.c_float(0.1), None)

    assert call(q=None) == INV
    assert call(cu_q=None) == INV
    assert call(n=0) == INV
    assert call(Hq=4, Hkv=3) == INV
    assert call(D=80) == UNS
    assert call(D=192) == UNS  # (192, 128) needs fa_fwd_varlen_hdim
    n = fa.NOALLOC_MAX_SEQS + 1
    assert call(n=n, tq=n, tk=n) == INV  # beyond the fixed array, rejected before any device work
    assert lib.fa_last_launch_count() == 0


def _packed_cpu(Tq=10, Tk=12, Hq=2, Hkv=1, D=64, n=2):
    bf, f32 = torch.bfloat16, torch.float32
    return dict(q=torch.zeros(Tq, Hq, D, dtype=bf), k=torch.zeros(Tk, Hkv, D, dtype=bf),
                v=torch.zeros(Tk, Hkv, D, dtype=bf), cu_seqlens_q=torch.zeros(n + 1, dtype=torch.int32),
                cu_seqlens_k=torch.zeros(n + 1, dtype=torch.int32), out=torch.zeros(Tq, Hq, D, dtype=f32),
                lse=torch.zeros(Hq, Tq, dtype=f32))


@pytest.mark.parametrize("entry", ["fa_fwd_varlen", "fa_fwd_varlen_noalloc"])
def test_packed_wrappers_check_every_shape_before_the_device(entry):
    """A wrong-shaped buffer is rejected with ValueError before the library is
    touched (CPU tensors: the shape checks come before the device check)."""
    fn = getattr(fa, entry)

    def call(**over):
        a = _packed_cpu()
        a.update(over)
        return fn(a["q"], a["k"], a["v"], a["cu_seqlens_q"], a["cu_seqlens_k"], 8, 8, out=a["out"], lse=a["lse"])

    f32, bf = torch.float32, torch.bfloat16
    with pytest.raises(ValueError, match="out must be"):
        call(out=torch.zeros(9, 2, 64, dtype=f32))              # undersized O
    with pytest.raises(ValueError, match="out must be"):
        call(lse=torch.zeros(2, 9, dtype=f32))                  # undersized LSE
    with pytest.raises(ValueError, match="shape mismatch"):
        call(v=torch.zeros(11, 1, 64, dtype=bf))                # V shorter than K
    with pytest.raises(ValueError, match="shape mismatch"):
        call(k=torch.zeros(12, 1, 128, dtype=bf), v=torch.zeros(12, 1, 128, dtype=bf))  # Dk != D
    with pytest.raises(ValueError, match="offsets"):
        call(cu_seqlens_k=torch.zeros(2, dtype=torch.int32))    # fewer key offsets
    with pytest.raises(ValueError, match="CUDA tensor"):
        call()                                                  # right shapes, host memory


def test_splitkv_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED

    def call(q=16, o=16, B=2, Hq=8, Hkv=2, Lq=1, Lk=100, D=128, scale=0.1, splits=0):
        return lib.fa_fwd_splitkv(q, 16, 16, o, 16, B, Hq, Hkv, Lq, Lk, D, 0, scale, splits, None, 0, None)

    assert call(q=None) == INV
    assert call(o=None) == INV
    assert call(B=0) == INV
    assert call(Lk=0) == INV
    assert call(Lq=-3) == INV
    assert call(Hq=6, Hkv=4) == INV
    assert call(scale=float("nan")) == INV
    assert call(o=40) == INV                         # misaligned output
    assert call(D=96) == UNS
    assert call(Hq=32, Hkv=1) == UNS                 # 32 query rows per KV head
    assert call(Hq=8, Hkv=2, Lq=5) == UNS            # 4 heads x 5 rows = 20 > 16
    n = ctypes.c_size_t(0)
    assert lib.fa_fwd_splitkv_workspace(2, 8, 2, 1, 100, 128, 0, None, None) == INV
    assert lib.fa_fwd_splitkv_workspace(2, 64, 2, 1, 100, 128, 0, ctypes.byref(n), None) == UNS
    assert lib.fa_fwd_splitkv_workspace(2, 8, 2, 1, 100, 80, 0, ctypes.byref(n), None) == UNS
    assert lib.fa_last_launch_count() == 0


def test_bwd_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED

    def call(q=16, dq=16, ws=16, B=1, Hq=2, Hkv=1, Lq=64, Lk=64, D=128, scale=0.1, wsb=1 << 20):
        return lib.fa_bwd(q, 16, 16, 16, 16, 16, dq, 16, 16, B, Hq, Hkv, Lq, Lk, D, 1, scale, ws, wsb, None)

    assert call(q=None) == INV
    assert call(dq=None) == INV
    assert call(ws=None) == INV
    assert call(B=0) == INV
    assert call(Lk=-1) == INV
    assert call(Hq=3, Hkv=2) == INV
    assert call(scale=0.0) == INV
    assert call(dq=20) == INV                        # misaligned
    assert call(wsb=100) == INV                      # workspace too small
    assert call(D=96) == UNS
    assert call(D=256) == UNS
    n = ctypes.c_size_t(0)
    assert lib.fa_bwd_workspace(2, 3, 130, ctypes.byref(n)) == fa.FA_OK
    assert n.value == 2 * 4 * 2 * 3 * 256            # delta and lse2, rows padded to 128
    assert lib.fa_bwd_workspace(2, 3, 0, ctypes.byref(n)) == INV


def test_variant_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED
    from exact_attention_07_gb300 import _Variant

    def call(var, D=128):
        return lib.fa_fwd_variant(16, 16, 16, 16, 16, 1, 2, 1, 64, 64, D, var, 0.1, None)

    assert call(None) == INV
    assert call(ctypes.byref(_Variant(-1, 0, float("nan"), None))) == INV
    assert call(ctypes.byref(_Variant(-1, 0, -1.0, None))) == INV
    assert call(ctypes.byref(_Variant(-1, 0, 0.0, 18))) == INV        # misaligned slopes
    assert call(ctypes.byref(_Variant(-1, 0, 0.0, None)), D=96) == UNS   # head dimensions 64 and 128 only
    assert lib.fa_fwd_varlen_variant(16, 16, 16, 16, 16, 32, 32, 1, 10, 10, 8, 8, 2, 2, 128, None, 0.1,
                                     None) == INV


def test_fp8_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED
    n = ctypes.c_size_t(0)
    assert lib.fa_fp8_workspace(1, 2, 1, 300, 200, 128, ctypes.byref(n)) == fa.FA_OK
    sec = fa.fp8_sections(1, 2, 1, 300, 200)
    assert n.value == sec["total"]
    assert sec["vt"][2] == (1, 1, 128, 256)                       # keys padded to a multiple of 128
    assert lib.fa_fp8_workspace(1, 2, 1, 300, 200, 64, ctypes.byref(n)) == UNS
    assert lib.fa_fp8_workspace(1, 3, 2, 300, 200, 128, ctypes.byref(n)) == INV
    assert lib.fa_fp8_prepare(16, 16, 16, 16, 1, 2, 1, 64, 64, 128, 16, 10, None) == INV   # buffer too small
    assert lib.fa_fp8_prepare(16, 16, 16, 18, 1, 2, 1, 64, 64, 128, 16, 1 << 20, None) == INV  # signs misaligned
    assert lib.fa_fwd_fp8(None, 16, 16, 1, 2, 1, 64, 64, 128, 0, 0.1, None) == INV
    assert lib.fa_fwd_fp8(16, 16, 16, 1, 2, 1, 64, 64, 128, 0, -0.1, None) == INV


def test_hdim_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED

    def call(D=192, Dv=128, v=16, B=1, scale=0.1):
        return lib.fa_fwd_hdim(16, 16, v, 16, 16, B, 2, 1, 64, 64, D, Dv, 1, scale, None)

    assert call(v=None) == INV
    assert call(Dv=0) == INV
    assert call(B=0) == INV
    assert call(scale=float("inf")) == INV
    for D, Dv in ((192, 192), (128, 64), (64, 128), (256, 128), (192, 64), (160, 128)):
        assert call(D=D, Dv=Dv) == UNS, (D, Dv)

    def vcall(D=192, Dv=128, n=2):
        return lib.fa_fwd_varlen_hdim(16, 16, 16, 16, 16, 32, 32, n, 10, 10, 8, 8, 2, 2, D, Dv, 1, 0.1, None)

    assert vcall(n=0) == INV
    assert vcall(Dv=-1) == INV
    assert vcall(D=128, Dv=192) == UNS
    assert lib.fa_last_launch_count() == 0


def test_bwd_varlen_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED

    def call(cu_q=32, dq=16, ws=16, n=2, tq=10, tk=10, mq=8, mk=8, Hq=2, Hkv=1, D=128, scale=0.1, wsb=1 << 20):
        return lib.fa_bwd_varlen(16, 16, 16, 16, 16, 16, dq, 16, 16, cu_q, 32, n, tq, tk, mq, mk, Hq, Hkv, D, 1,
                                 scale, ws, wsb, None)

    assert call(cu_q=None) == INV
    assert call(dq=None) == INV
    assert call(ws=None) == INV
    assert call(n=0) == INV
    assert call(tk=0) == INV
    assert call(Hq=3, Hkv=2) == INV
    assert call(cu_q=34) == INV                      # int32 offsets must be 4-byte aligned
    assert call(wsb=64) == INV                       # workspace too small
    assert call(D=80) == UNS
    n = ctypes.c_size_t(0)
    assert lib.fa_bwd_varlen_workspace(3, 1000, 4, ctypes.byref(n)) == fa.FA_OK
    rows = (1000 + 127) // 128 * 128 + 128 * 3       # each sequence padded to 128 rows
    assert n.value >= 2 * 4 * rows * 4 + 4 * (4 * 3 + 3)
    assert lib.fa_bwd_varlen_workspace(0, 1000, 4, ctypes.byref(n)) == INV
    assert lib.fa_last_launch_count() == 0


def test_bwd_variant_argument_validation(lib):
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED
    from exact_attention_07_gb300 import _Variant

    def call(var, D=128):
        return lib.fa_bwd_variant(16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 2, 1, 64, 64, D, var, 0.1, 16, 1 << 20, None)

    assert call(None) == INV
    assert call(ctypes.byref(_Variant(-1, 0, float("nan"), None))) == INV
    assert call(ctypes.byref(_Variant(-1, 0, 0.0, 18))) == INV        # misaligned slopes
    assert call(ctypes.byref(_Variant(-1, 0, 0.0, None)), D=96) == UNS   # head dimensions 64 and 128 only
    assert lib.fa_bwd_varlen_variant(16, 16, 16, 16, 16, 16, 16, 16, 16, 32, 32, 1, 10, 10, 8, 8, 2, 2, 128, None,
                                     0.1, 16, 1 << 20, None) == INV
    assert lib.fa_last_launch_count() == 0
