"""CPU oracle for the fused GEMM + bias/activation epilogue.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package; the library (``activation_epilogue_gb300``) never does.
It shares no code with the CUDA path.

The arithmetic lives in ``gemm_epi_oracle.c`` (plain C, double precision, OpenMP over
rows); this module compiles it with gcc on first use and wraps it with numpy arrays.
What each function computes, and the page passage it follows, is stated in the C file:

* "Fusing bias into cuBLASLt matmul with nvmath-python for PyTorch inference"
  (blog.hotdry.top, 2025-09-22): the BIAS / RELU_BIAS / RELU_AUX_BIAS epilogs, the bias
  shapes (m,1) and (1,n), and the code example's A[m,k] . B[k,n] + bias.
* "Operator fusion in model inference, from LayerNorm to residual connections"
  (wmrh.cn/news/429806), section 1 flowchart and section 3: the FFN chain
  matmul -> bias -> GELU -> matmul -> bias, and the residual add.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_epi_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# A prebuilt oracle library to load instead (used by the mutation test, which builds copies
# of the oracle with planted mistakes and checks that the pins catch each one).
_LIB_OVERRIDE = os.environ.get("GEMM_EPI_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

DTYPES = {"f16": 0, "bf16": 1}
EPILOGS = {"BIAS": 0, "RELU_BIAS": 1, "GELU_BIAS": 2, "RELU_AUX_BIAS": 3,
           "BIAS_RESIDUAL": 4, "NONE": 5, "TANH_BIAS": 6, "GELU_AUX_BIAS": 7}
BWD_KINDS = {"DRELU_BGRAD": 0, "DGELU_BGRAD": 1}
BIAS_LAYOUTS = {"M1": 0, "1N": 1}


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, OpenMP, no fast-math)."""
    with _lock:
        stale = (not os.path.exists(_LIB)
                 or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
                   "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if _LIB_OVERRIDE:
        lib = ctypes.CDLL(_LIB_OVERRIDE)
    else:
        build()
        lib = ctypes.CDLL(_LIB)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_decode_f16.restype = ctypes.c_double
    lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_bf16.restype = ctypes.c_double
    lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_encode_f16.restype = ctypes.c_uint16
    lib.oracle_encode_f16.argtypes = [ctypes.c_double]
    lib.oracle_encode_bf16.restype = ctypes.c_uint16
    lib.oracle_encode_bf16.argtypes = [ctypes.c_double]
    lib.oracle_gelu.restype = ctypes.c_double
    lib.oracle_gelu.argtypes = [ctypes.c_double]
    lib.oracle_encode_array.restype = None
    lib.oracle_encode_array.argtypes = [i32, vp, i64, vp]
    lib.oracle_decode_array.restype = None
    lib.oracle_decode_array.argtypes = [i32, vp, i64, vp]
    lib.oracle_gemm_epi.restype = i32
    lib.oracle_gemm_epi.argtypes = [i64, i64, i64, i32, i32, i32, vp, vp, vp, vp,
                                    vp, i64, vp, i64, vp, vp]
    lib.oracle_aux_pack.restype = None
    lib.oracle_aux_pack.argtypes = [vp, i64, i64, vp]
    lib.oracle_ffn.restype = i32
    lib.oracle_ffn.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.oracle_gelu_grad.restype = ctypes.c_double
    lib.oracle_gelu_grad.argtypes = [ctypes.c_double]
    lib.oracle_gemm_bwd.restype = i32
    lib.oracle_gemm_bwd.argtypes = [i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.oracle_num_threads.restype = i32
    lib.oracle_num_threads.argtypes = []
    f64 = ctypes.c_double
    lib.oracle_decode_e4m3.restype = f64
    lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_gemm_epi_fp8.restype = i32
    lib.oracle_gemm_epi_fp8.argtypes = [i64, i64, i64, i32, i32, vp, vp, f64, f64, vp, vp, vp,
                                        vp]
    lib.oracle_layernorm.restype = i32
    lib.oracle_layernorm.argtypes = [i64, i64, i32, vp, vp, vp, vp, f64, vp, vp]
    lib.oracle_ln_gemm_gelu.restype = i32
    lib.oracle_ln_gemm_gelu.argtypes = [i64, i64, i64, i32, vp, vp, vp, f64, vp, vp, vp]
    lib.oracle_ln_ffn.restype = i32
    lib.oracle_ln_ffn.argtypes = [i64, i64, i64, i32, vp, vp, vp, f64, vp, vp, vp, vp, vp, vp,
                                  vp, vp]
    _lib = lib
    return lib


def _bits(x) -> np.ndarray:
    """16-bit payload of a numpy uint16/float16 array or a CPU torch 16-bit tensor."""
    if hasattr(x, "detach"):                       # a torch tensor
        import torch
        x = x.detach().contiguous().cpu().view(torch.int16).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype.itemsize != 2:
        raise TypeError(f"expected 16-bit elements, got {x.dtype}")
    return x.view(np.uint16)


def _ptr(a) -> int | None:
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def decode(dtype: str, bits) -> np.ndarray:
    b = _bits(bits)
    out = np.empty(b.shape, np.float64)
    _load().oracle_decode_array(DTYPES[dtype], _ptr(b), b.size, _ptr(out))
    return out


def encode(dtype: str, x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_encode_array(DTYPES[dtype], _ptr(x), x.size, _ptr(out))
    return out


def gelu(x: float) -> float:
    return float(_load().oracle_gelu(float(x)))


def gemm_epi(A, B, bias, *, dtype: str, epilog: str, bias_layout: str = "1N",
             residual=None, rows=None, cols=None, want_pre: bool = False):
    """D (and optionally pre) in double for the selected rows x cols of the m x n output.

    A: m x k, B: k x n, bias: m or n elements (or None for NONE), residual: m x n.  All are
    16-bit arrays (numpy uint16/float16 or CPU torch tensors) of ``dtype``.
    """
    A16, B16 = _bits(A), _bits(B)
    m, k = A16.shape
    k2, n = B16.shape
    if k2 != k:
        raise ValueError("inner dimensions differ")
    bias16 = None if bias is None else _bits(bias).reshape(-1)
    res16 = None if residual is None else _bits(residual)
    rows = np.arange(m, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cols = np.arange(n, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    D = np.empty((rows.size, cols.size), np.float64)
    pre = np.empty_like(D) if want_pre else None
    rc = _load().oracle_gemm_epi(m, n, k, DTYPES[dtype], EPILOGS[epilog],
                                 BIAS_LAYOUTS[bias_layout], _ptr(A16), _ptr(B16),
                                 _ptr(bias16), _ptr(res16), _ptr(rows), rows.size,
                                 _ptr(cols), cols.size, _ptr(pre), _ptr(D))
    if rc != 0:
        raise ValueError("oracle_gemm_epi: bad arguments or out of memory")
    return (D, pre) if want_pre else D


def aux_pack(pre: np.ndarray) -> np.ndarray:
    """uint32[rows][ceil(n/32)] mask words from full rows of pre (rows x n)."""
    pre = np.ascontiguousarray(pre, np.float64)
    r, n = pre.shape
    words = np.empty((r, (n + 31) // 32), np.uint32)
    _load().oracle_aux_pack(_ptr(pre), r, n, _ptr(words))
    return words


def ffn(X, W1, b1, W2, b2, R, *, dtype: str = "bf16"):
    """(H_bits, H_exact, Y): the stored hidden activation, its unrounded value, the output."""
    X16, W116, b116 = _bits(X), _bits(W1), _bits(b1).reshape(-1)
    W216, b216, R16 = _bits(W2), _bits(b2).reshape(-1), _bits(R)
    t, d = X16.shape
    f = W116.shape[1]
    H = np.empty((t, f), np.uint16)
    Hx = np.empty((t, f), np.float64)
    Y = np.empty((t, d), np.float64)
    rc = _load().oracle_ffn(t, d, f, DTYPES[dtype], _ptr(X16), _ptr(W116), _ptr(b116),
                            _ptr(W216), _ptr(b216), _ptr(R16), _ptr(H), _ptr(Hx), _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_ffn: bad arguments or out of memory")
    return H, Hx, Y


def gelu_grad(x: float) -> float:
    return float(_load().oracle_gelu_grad(float(x)))


def gemm_bwd(A, B, *, dtype: str, kind: str, bias_layout: str = "1N", mask=None, pre=None):
    """(D, dbias) in double for the backward epilogues DRELU_BGRAD (mask: uint32 words
    [m][ceil(n/32)]) and DGELU_BGRAD (pre: the stored 16-bit pre-activation, m x n)."""
    A16, B16 = _bits(A), _bits(B)
    m, k = A16.shape
    n = B16.shape[1]
    mk = None
    if mask is not None:
        mk = np.ascontiguousarray(mask).view(np.uint32).reshape(m, (n + 31) // 32)
    pr = None if pre is None else _bits(pre)
    D = np.empty((m, n), np.float64)
    dbias = np.empty(m if bias_layout == "M1" else n, np.float64)
    rc = _load().oracle_gemm_bwd(m, n, k, DTYPES[dtype], BWD_KINDS[kind],
                                 BIAS_LAYOUTS[bias_layout], _ptr(A16), _ptr(B16), _ptr(mk),
                                 _ptr(pr), _ptr(D), _ptr(dbias))
    if rc != 0:
        raise ValueError("oracle_gemm_bwd: bad arguments or out of memory")
    return D, dbias


def layernorm(X, gamma, beta, *, eps: float, dtype: str, residual=None):
    """(Y, stats) in double: LayerNorm of the rows of X (t x d) times gamma plus beta (plus
    the residual), and per row (mean, 1 / sqrt(var + eps))."""
    X16 = _bits(X)
    t, d = X16.shape
    g16, b16 = _bits(gamma).reshape(-1), _bits(beta).reshape(-1)
    r16 = None if residual is None else _bits(residual)
    Y = np.empty((t, d), np.float64)
    stats = np.empty((t, 2), np.float64)
    rc = _load().oracle_layernorm(t, d, DTYPES[dtype], _ptr(X16), _ptr(r16), _ptr(g16),
                                  _ptr(b16), float(eps), _ptr(Y), _ptr(stats))
    if rc != 0:
        raise ValueError("oracle_layernorm: bad arguments")
    return Y, stats


def ln_gemm_gelu(A, gamma, beta, W, b, *, eps: float, dtype: str):
    """D = GELU(LayerNorm(A) . W + b) in double (LayerNorm(A) not rounded)."""
    A16, W16 = _bits(A), _bits(W)
    m, k = A16.shape
    n = W16.shape[1]
    D = np.empty((m, n), np.float64)
    rc = _load().oracle_ln_gemm_gelu(m, n, k, DTYPES[dtype], _ptr(A16),
                                     _ptr(_bits(gamma).reshape(-1)),
                                     _ptr(_bits(beta).reshape(-1)), float(eps), _ptr(W16),
                                     _ptr(_bits(b).reshape(-1)), _ptr(D))
    if rc != 0:
        raise ValueError("oracle_ln_gemm_gelu: bad arguments or out of memory")
    return D


def ln_ffn(X, gamma, beta, W1, b1, W2, b2, R, *, eps: float, dtype: str = "bf16"):
    """(H_bits, H_exact, Y) of the pre-LayerNorm FFN block."""
    X16, W116, W216 = _bits(X), _bits(W1), _bits(W2)
    t, d = X16.shape
    f = W116.shape[1]
    H = np.empty((t, f), np.uint16)
    Hx = np.empty((t, f), np.float64)
    Y = np.empty((t, d), np.float64)
    rc = _load().oracle_ln_ffn(t, d, f, DTYPES[dtype], _ptr(X16), _ptr(_bits(gamma).reshape(-1)),
                               _ptr(_bits(beta).reshape(-1)), float(eps), _ptr(W116),
                               _ptr(_bits(b1).reshape(-1)), _ptr(W216),
                               _ptr(_bits(b2).reshape(-1)), _ptr(_bits(R)), _ptr(H), _ptr(Hx),
                               _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_ln_ffn: bad arguments or out of memory")
    return H, Hx, Y


def _bytes8(x) -> np.ndarray:
    """8-bit payload of a numpy uint8 array or a CPU torch 8-bit tensor (e.g. float8_e4m3fn)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().contiguous().cpu().view(torch.uint8).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype.itemsize != 1:
        raise TypeError(f"expected 8-bit elements, got {x.dtype}")
    return x.view(np.uint8)


def decode_e4m3(bits) -> np.ndarray:
    b = _bytes8(bits)
    lib = _load()
    return np.array([lib.oracle_decode_e4m3(int(v)) for v in b.reshape(-1)],
                    np.float64).reshape(b.shape)


def gemm_epi_fp8(A, Bt, bias, *, scale_a: float, scale_b: float, epilog: str,
                 bias_layout: str = "1N", residual=None, want_pre: bool = False):
    """D (and pre) in double for E4M3 A (m x k) and Bt (n x k), bf16 bias / residual."""
    A8, B8 = _bytes8(A), _bytes8(Bt)
    m, k = A8.shape
    n, k2 = B8.shape
    if k2 != k:
        raise ValueError("inner dimensions differ")
    b16 = None if bias is None else _bits(bias).reshape(-1)
    r16 = None if residual is None else _bits(residual)
    D = np.empty((m, n), np.float64)
    pre = np.empty_like(D) if want_pre else None
    rc = _load().oracle_gemm_epi_fp8(m, n, k, EPILOGS[epilog], BIAS_LAYOUTS[bias_layout],
                                     _ptr(A8), _ptr(B8), float(scale_a), float(scale_b),
                                     _ptr(b16), _ptr(r16), _ptr(pre), _ptr(D))
    if rc != 0:
        raise ValueError("oracle_gemm_epi_fp8: bad arguments or out of memory")
    return (D, pre) if want_pre else D
