"""In-tree build of the CUDA library ``libfa_gb300.so`` (sm_103a only).

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library next to this file's package.  No CMake, no torch extension
machinery: the library exports a plain C ABI (include/fa_gb300.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa_gb300.so")
SOURCES = ["fa_api.cu", "fa_fwd_d64.cu", "fa_fwd_d128.cu", "fa_decode.cu", "fa_decode_tc.cu", "fa_bwd.cu", "fa_fwd_var.cu", "fa_fwd_fp8.cu", "fa_fp8.cu", "fa_fwd_d192.cu", "fa_bwd_var.cu", "fa_fwd_var64.cu", "fa_bwd_var64.cu"]
HEADERS = ["fa_fwd_kernel.cuh", "ptx_sm103.cuh", "fa_params.h", "fa_launch.h", "fa_decode.h", "fa_bwd.h", "fa_fp8.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")


def common_flags() -> list[str]:
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                   "-I", os.path.join(ROOT, "include")]


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *common_flags(), "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile (if stale) and link libfa_gb300.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "fa_gb300.h"),
                                                                  __file__]
    if not force and not verbose_ptxas and not _stale(LIB, deps):
        return LIB
    logs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = []
        for obj, log in ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES):
            objs.append(obj)
            logs.append(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{cuda_lib_dir()}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose_ptxas:
        print("\n".join(logs))
    return LIB


if __name__ == "__main__":
    import sys
    build(force=True, verbose_ptxas="-v" in sys.argv)
    print(LIB)
