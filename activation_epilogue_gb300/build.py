"""Build ``libgemmepi.so`` in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel (``-gencode
arch=compute_103a,code=sm_103a -lineinfo -O3``), with the CUDA runtime linked statically,
so the library needs only the NVIDIA driver at run time; ``-Xptxas -v`` register and
shared-memory reports are kept in ``_build/ptxas.log``.

    python -m activation_epilogue_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgemmepi.so")
SOURCES = ["api.cu", "host_exec.cu", "ffn_api.cu", "layernorm_api.cu", "gemm_pair.cu",
           "gemm_pair_fp8.cu",
           "gemm_rowtile.cu", "gemm_swapped.cu", "gemm_fwd_bias.cu", "gemm_fwd_relu.cu",
           "gemm_fwd_gelu.cu", "gemm_fwd_relu_aux.cu", "gemm_fwd_residual.cu",
           "gemm_smallm.cu", "ffn_onchip.cu", "elementwise.cu", "layernorm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "gemm_epi.h"))
    return [f for f in files if os.path.isfile(f)]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps() + [__file__])


def _compile(nvcc: str, src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s), SOURCES))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as fh:
        for src, (_, log) in zip(SOURCES, results):
            fh.write(f"==== {src}\n{log}\n")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
