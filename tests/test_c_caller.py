"""The C ABI from a plain C11 program (tests/c_caller.c): the header compiles as C with
warnings as errors and every call the program makes links against libgemmepi.so (CPU);
on a GPU the program runs RELU_AUX_BIAS plans for the swapped, row-tile and CTA-pair
kernels and checks D and the mask bit for bit against integer arithmetic, then runs the FFN
block in each of its modes (and without allocation) against its own double-precision sum."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_caller.c")


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    return None


def _compile(tmp_path):
    from activation_epilogue_gb300 import build
    lib = build.build()
    cuda = _cuda_home()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cuda is None or cc is None:
        pytest.skip("no C compiler or CUDA runtime headers")
    libdir = os.path.dirname(lib)
    cudalib = os.path.join(cuda, "lib64")
    exe = str(tmp_path / "c_caller")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), SRC, "-L", libdir, "-lgemmepi", "-L", cudalib,
           "-lcudart", "-lm", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_caller_compiles_and_links(tmp_path):
    _compile(tmp_path)


@pytest.mark.gpu
def test_c_caller_runs(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok"), r.stdout
    # the three kernels the shapes are meant to reach
    for variant in ("variant=small-m", "variant=swapped", "variant=row-tile", "variant=row-pair"):
        assert variant in r.stdout, r.stdout
    # the FFN block's modes
    for mode in ("ffn one launch:", "ffn two launches:", "ffn one launch, H on chip", "ffn noalloc"):
        assert mode in r.stdout, r.stdout
