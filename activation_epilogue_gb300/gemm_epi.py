"""Python binding of the C ABI in ``include/gemm_epi.h`` (ctypes; argument marshalling only).

Every function has the C name and forwards to ``libgemmepi.so``; the tensors are PyTorch
CUDA tensors, used only as device memory, and the stream is the current torch stream
unless one is given.  All the computation happens in the library's kernels: if the
library is missing or cannot be loaded, the calls raise instead of computing anything
another way.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgemmepi.so")

DTYPE = {"f16": 0, "bf16": 1, "e4m3": 2}
EPILOG = {"BIAS": 0, "RELU_BIAS": 1, "GELU_BIAS": 2, "RELU_AUX_BIAS": 3, "BIAS_RESIDUAL": 4,
          "NONE": 5, "TANH_BIAS": 6, "GELU_AUX_BIAS": 7, "DRELU_BGRAD": 8, "DGELU_BGRAD": 9,
          "LN_GELU_BIAS": 10}
BACKWARD = ("DRELU_BGRAD", "DGELU_BGRAD")
BIAS_LAYOUT = {"M1": 0, "1N": 1}
OPTION = {"VARIANT": 0, "TILE_N": 1, "SPLIT_K": 2, "GRID": 3, "GROUP_M": 4,
          "WAIT_LIMIT_US": 5, "DEBUG_STALL": 6, "PREFETCH": 7, "PDL": 8, "SPLIT_MODE": 9,
          "TILE_M": 10, "TILE_ORDER": 11, "B_READY": 12}
STATUS = {0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED_SHAPE", 3: "ERR_MISALIGNED",
          4: "ERR_NO_DEVICE", 5: "ERR_ARCH", 6: "ERR_ALLOC", 7: "ERR_LAUNCH",
          8: "ERR_DEVICE_TIMEOUT", 9: "ERR_SCRATCH_LIMIT"}

# Every symbol include/gemm_epi.h declares.
EXPORTS = ["gemm_epi_plan", "gemm_epi_plan_set_option", "gemm_epi_execute",
           "gemm_epi_execute_ex", "gemm_epi_execute_unfused", "gemm_epi_free",
           "gemm_epi_sync_status", "gemm_epi_status_string", "gemm_epi_plan_describe",
           "gemm_epi_aux_words_per_row", "gemm_epi_ffn_plan", "gemm_epi_ffn_execute",
           "gemm_epi_ffn_hidden", "gemm_epi_ffn_sync_status", "gemm_epi_ffn_free",
           "gemm_epi_ffn_execute_noalloc", "gemm_epi_execute_operands",
           "gemm_epi_execute_operands_unfused", "gemm_epi_ffn_set_option",
           "gemm_epi_ffn_plan_describe", "gemm_epi_layernorm", "gemm_epi_layernorm_stats",
           "gemm_epi_layernorm_fold", "gemm_epi_ffn_plan_layernorm",
           "gemm_epi_ffn_execute_layernorm", "gemm_epi_execute_host"]
FFN_OPTION = {"LAUNCHES": 0, "SPLIT2": 1, "TILE_ORDER": 2, "B_READY": 3}

# Largest t * f the allocation-free FFN call accepts (its static scratch holds H).
FFN_NOALLOC_MAX_HIDDEN = 16 * 1024 * 1024

_lib = None
_lock = threading.Lock()


class Operands(ctypes.Structure):
    """gemm_epi_operands: every operand of one call (NULL where the epilog uses none)."""
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("D", ctypes.c_void_p), ("aux", ctypes.c_void_p),
                ("aux_in", ctypes.c_void_p), ("dbias", ctypes.c_void_p),
                ("ln_stats", ctypes.c_void_p), ("ln_colsum", ctypes.c_void_p),
                ("ln_bias", ctypes.c_void_p), ("scale_a", ctypes.c_void_p),
                ("scale_b", ctypes.c_void_p)]


class GemmEpiError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {status_string(status)}")


def load_library(path: str | None = None):
    """Load libgemmepi.so (raises OSError if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        lib = ctypes.CDLL(path or LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.gemm_epi_plan.restype = i32
        lib.gemm_epi_plan.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32, i32, i32]
        lib.gemm_epi_plan_set_option.restype = i32
        lib.gemm_epi_plan_set_option.argtypes = [vp, i32, i64]
        lib.gemm_epi_execute.restype = i32
        lib.gemm_epi_execute.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        lib.gemm_epi_execute_ex.restype = i32
        lib.gemm_epi_execute_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        lib.gemm_epi_execute_unfused.restype = i32
        lib.gemm_epi_execute_unfused.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.gemm_epi_free.restype = i32
        lib.gemm_epi_free.argtypes = [vp]
        lib.gemm_epi_sync_status.restype = i32
        lib.gemm_epi_sync_status.argtypes = [vp, vp]
        lib.gemm_epi_status_string.restype = ctypes.c_char_p
        lib.gemm_epi_status_string.argtypes = [i32]
        lib.gemm_epi_plan_describe.restype = ctypes.c_char_p
        lib.gemm_epi_plan_describe.argtypes = [vp]
        lib.gemm_epi_aux_words_per_row.restype = i64
        lib.gemm_epi_aux_words_per_row.argtypes = [i64]
        lib.gemm_epi_ffn_plan.restype = i32
        lib.gemm_epi_ffn_plan.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32]
        lib.gemm_epi_ffn_execute.restype = i32
        lib.gemm_epi_ffn_execute.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.gemm_epi_ffn_hidden.restype = vp
        lib.gemm_epi_ffn_hidden.argtypes = [vp]
        lib.gemm_epi_ffn_sync_status.restype = i32
        lib.gemm_epi_ffn_sync_status.argtypes = [vp, vp]
        lib.gemm_epi_ffn_free.restype = i32
        lib.gemm_epi_ffn_free.argtypes = [vp]
        lib.gemm_epi_ffn_execute_noalloc.restype = i32
        lib.gemm_epi_ffn_execute_noalloc.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, vp,
                                                     vp, vp]
        lib.gemm_epi_ffn_set_option.restype = i32
        lib.gemm_epi_ffn_set_option.argtypes = [vp, i32, i64]
        lib.gemm_epi_ffn_plan_describe.restype = ctypes.c_char_p
        lib.gemm_epi_ffn_plan_describe.argtypes = [vp]
        f32 = ctypes.c_float
        lib.gemm_epi_layernorm.restype = i32
        lib.gemm_epi_layernorm.argtypes = [i64, i64, i32, vp, vp, vp, vp, f32, vp, vp]
        lib.gemm_epi_layernorm_stats.restype = i32
        lib.gemm_epi_layernorm_stats.argtypes = [i64, i64, i32, vp, f32, vp, vp]
        lib.gemm_epi_layernorm_fold.restype = i32
        lib.gemm_epi_layernorm_fold.argtypes = [i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.gemm_epi_ffn_plan_layernorm.restype = i32
        lib.gemm_epi_ffn_plan_layernorm.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32]
        lib.gemm_epi_ffn_execute_layernorm.restype = i32
        lib.gemm_epi_ffn_execute_layernorm.argtypes = [vp, vp, f32, vp, vp, vp, vp, vp, vp, vp,
                                                       vp]
        lib.gemm_epi_execute_host.restype = i32
        lib.gemm_epi_execute_host.argtypes = [vp, ctypes.POINTER(Operands), vp]
        lib.gemm_epi_execute_operands.restype = i32
        lib.gemm_epi_execute_operands.argtypes = [vp, ctypes.POINTER(Operands), vp]
        lib.gemm_epi_execute_operands_unfused.restype = i32
        lib.gemm_epi_execute_operands_unfused.argtypes = [vp, ctypes.POINTER(Operands), vp, vp]
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().gemm_epi_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise GemmEpiError(status, what)


def _ptr(t):
    """Device address of a tensor (None -> NULL); raw integers pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous (row-major)")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- the C functions, by name -------------------------------------------------------------

def gemm_epi_plan(m: int, n: int, k: int, dtype: str, epilog: str, bias_layout: str = "1N"):
    h = ctypes.c_void_p()
    _check(load_library().gemm_epi_plan(ctypes.byref(h), m, n, k, DTYPE[dtype], EPILOG[epilog],
                                        BIAS_LAYOUT[bias_layout]), "gemm_epi_plan")
    return h.value


def gemm_epi_plan_set_option(plan, option: str, value: int):
    _check(load_library().gemm_epi_plan_set_option(plan, OPTION[option], int(value)),
           f"gemm_epi_plan_set_option({option}={value})")


def gemm_epi_execute(plan, A, B, bias, D, aux=None, stream=None):
    _check(load_library().gemm_epi_execute(plan, _ptr(A), _ptr(B), _ptr(bias), _ptr(D),
                                           _ptr(aux), _stream(stream)), "gemm_epi_execute")


def gemm_epi_execute_ex(plan, A, B, bias, residual, D, aux=None, stream=None):
    _check(load_library().gemm_epi_execute_ex(plan, _ptr(A), _ptr(B), _ptr(bias),
                                              _ptr(residual), _ptr(D), _ptr(aux),
                                              _stream(stream)), "gemm_epi_execute_ex")


def gemm_epi_execute_unfused(plan, A, B, bias, residual, pre, D, aux=None, stream=None):
    _check(load_library().gemm_epi_execute_unfused(plan, _ptr(A), _ptr(B), _ptr(bias),
                                                   _ptr(residual), _ptr(pre), _ptr(D),
                                                   _ptr(aux), _stream(stream)),
           "gemm_epi_execute_unfused")


def _operands(A, B, bias, residual, D, aux, aux_in, dbias, ln=None, scales=None) -> Operands:
    ln_stats, ln_colsum, ln_bias = ln if ln is not None else (None, None, None)
    scale_a, scale_b = scales if scales is not None else (None, None)
    return Operands(_ptr(A), _ptr(B), _ptr(bias), _ptr(residual), _ptr(D), _ptr(aux),
                    _ptr(aux_in), _ptr(dbias), _ptr(ln_stats), _ptr(ln_colsum), _ptr(ln_bias),
                    _ptr(scale_a), _ptr(scale_b))


def gemm_epi_execute_operands(plan, A, B, D, bias=None, residual=None, aux=None, aux_in=None,
                              dbias=None, stream=None, ln=None, scales=None):
    """ln: (stats, colsum, bias_folded) for the LN_GELU_BIAS epilog; scales: (scale_a,
    scale_b) device fp32 scalars for E4M3 plans (B is then given transposed, n x k)."""
    ops = _operands(A, B, bias, residual, D, aux, aux_in, dbias, ln, scales)
    _check(load_library().gemm_epi_execute_operands(plan, ctypes.byref(ops), _stream(stream)),
           "gemm_epi_execute_operands")


def gemm_epi_execute_host(plan, A, B, D, bias=None, residual=None, aux=None, stream=None):
    """The fused call on host tensors (CPU, contiguous, preferably pinned): copies in, GEMM and
    copies out pipelined in row chunks by the library; ordered on `stream`."""
    ops = _operands(A, B, bias, residual, D, aux, None, None)
    _check(load_library().gemm_epi_execute_host(plan, ctypes.byref(ops), _stream(stream)),
           "gemm_epi_execute_host")


def gemm_epi_execute_operands_unfused(plan, A, B, D, pre, bias=None, residual=None, aux=None,
                                      aux_in=None, dbias=None, stream=None, ln=None,
                                      scales=None):
    ops = _operands(A, B, bias, residual, D, aux, aux_in, dbias, ln, scales)
    _check(load_library().gemm_epi_execute_operands_unfused(plan, ctypes.byref(ops), _ptr(pre),
                                                            _stream(stream)),
           "gemm_epi_execute_operands_unfused")


def gemm_epi_layernorm(t: int, d: int, dtype: str, X, residual, gamma, beta, eps: float, Y,
                       stream=None):
    _check(load_library().gemm_epi_layernorm(t, d, DTYPE[dtype], _ptr(X), _ptr(residual),
                                             _ptr(gamma), _ptr(beta), float(eps), _ptr(Y),
                                             _stream(stream)), "gemm_epi_layernorm")


def gemm_epi_layernorm_stats(t: int, d: int, dtype: str, X, eps: float, stats, stream=None):
    _check(load_library().gemm_epi_layernorm_stats(t, d, DTYPE[dtype], _ptr(X), float(eps),
                                                   _ptr(stats), _stream(stream)),
           "gemm_epi_layernorm_stats")


def gemm_epi_layernorm_fold(d: int, f: int, dtype: str, gamma, beta, W, b, W_folded, colsum,
                            bias_folded, stream=None):
    _check(load_library().gemm_epi_layernorm_fold(d, f, DTYPE[dtype], _ptr(gamma), _ptr(beta),
                                                  _ptr(W), _ptr(b), _ptr(W_folded),
                                                  _ptr(colsum), _ptr(bias_folded),
                                                  _stream(stream)), "gemm_epi_layernorm_fold")


def gemm_epi_ffn_plan_layernorm(t: int, d: int, f: int, dtype: str = "bf16"):
    h = ctypes.c_void_p()
    _check(load_library().gemm_epi_ffn_plan_layernorm(ctypes.byref(h), t, d, f, DTYPE[dtype]),
           "gemm_epi_ffn_plan_layernorm")
    return h.value


def gemm_epi_ffn_execute_layernorm(plan, X, eps: float, W1_folded, colsum, b1_folded, W2, b2, R,
                                   Y, stream=None):
    _check(load_library().gemm_epi_ffn_execute_layernorm(plan, _ptr(X), float(eps),
                                                         _ptr(W1_folded), _ptr(colsum),
                                                         _ptr(b1_folded), _ptr(W2), _ptr(b2),
                                                         _ptr(R), _ptr(Y), _stream(stream)),
           "gemm_epi_ffn_execute_layernorm")


def gemm_epi_free(plan):
    _check(load_library().gemm_epi_free(plan), "gemm_epi_free")


def gemm_epi_sync_status(plan, stream=None) -> int:
    """Returns the status code (0, or 8 = a device-side wait ran out)."""
    return int(load_library().gemm_epi_sync_status(plan, _stream(stream)))


def gemm_epi_status_string(status: int) -> str:
    return status_string(status)


def gemm_epi_plan_describe(plan) -> str:
    return load_library().gemm_epi_plan_describe(plan).decode()


def gemm_epi_aux_words_per_row(n: int) -> int:
    return int(load_library().gemm_epi_aux_words_per_row(n))


def gemm_epi_ffn_plan(t: int, d: int, f: int, dtype: str = "bf16"):
    h = ctypes.c_void_p()
    _check(load_library().gemm_epi_ffn_plan(ctypes.byref(h), t, d, f, DTYPE[dtype]),
           "gemm_epi_ffn_plan")
    return h.value


def gemm_epi_ffn_execute(plan, X, W1, b1, W2, b2, R, Y, stream=None):
    _check(load_library().gemm_epi_ffn_execute(plan, _ptr(X), _ptr(W1), _ptr(b1), _ptr(W2),
                                               _ptr(b2), _ptr(R), _ptr(Y), _stream(stream)),
           "gemm_epi_ffn_execute")


def gemm_epi_ffn_set_option(plan, option: str, value: int):
    _check(load_library().gemm_epi_ffn_set_option(plan, FFN_OPTION[option], int(value)),
           f"gemm_epi_ffn_set_option({option}={value})")


def gemm_epi_ffn_plan_describe(plan) -> str:
    return load_library().gemm_epi_ffn_plan_describe(plan).decode()


def gemm_epi_ffn_hidden(plan) -> int:
    return load_library().gemm_epi_ffn_hidden(plan) or 0


def gemm_epi_ffn_sync_status(plan, stream=None) -> int:
    return int(load_library().gemm_epi_ffn_sync_status(plan, _stream(stream)))


def gemm_epi_ffn_free(plan):
    _check(load_library().gemm_epi_ffn_free(plan), "gemm_epi_ffn_free")


def gemm_epi_ffn_execute_noalloc(t: int, d: int, f: int, dtype: str, X, W1, b1, W2, b2, R, Y,
                                 stream=None):
    """The FFN block without allocating: for callers that must not allocate device memory.
    H lives in the library's static scratch, so calls on one device must not overlap."""
    _check(load_library().gemm_epi_ffn_execute_noalloc(t, d, f, DTYPE[dtype], _ptr(X), _ptr(W1),
                                                       _ptr(b1), _ptr(W2), _ptr(b2), _ptr(R),
                                                       _ptr(Y), _stream(stream)),
           "gemm_epi_ffn_execute_noalloc")


class FfnPlan:
    """The FFN block Y = GELU(X.W1 + b1).W2 + b2 + R as one plan (two fused launches)."""

    def __init__(self, t, d, f, dtype="bf16", layernorm=False, **options):
        self.t, self.d, self.f, self.dtype = t, d, f, dtype
        self.handle = (gemm_epi_ffn_plan_layernorm(t, d, f, dtype) if layernorm
                       else gemm_epi_ffn_plan(t, d, f, dtype))
        for key, value in options.items():
            gemm_epi_ffn_set_option(self.handle, key.upper(), value)

    def describe(self) -> str:
        return gemm_epi_ffn_plan_describe(self.handle)

    def execute(self, X, W1, b1, W2, b2, R, Y, stream=None):
        gemm_epi_ffn_execute(self.handle, X, W1, b1, W2, b2, R, Y, stream)

    def execute_layernorm(self, X, eps, W1_folded, colsum, b1_folded, W2, b2, R, Y,
                          stream=None):
        gemm_epi_ffn_execute_layernorm(self.handle, X, eps, W1_folded, colsum, b1_folded, W2,
                                       b2, R, Y, stream)

    def hidden(self):
        """The plan's H buffer as a torch tensor view (t x f) on the current device."""
        import torch
        ptr = gemm_epi_ffn_hidden(self.handle)
        if not ptr:
            return None
        return _tensor_from_ptr(ptr, (self.t, self.f), self.dtype)

    def sync_status(self, stream=None) -> int:
        return gemm_epi_ffn_sync_status(self.handle, stream)

    def free(self):
        if self.handle:
            gemm_epi_ffn_free(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def _tensor_from_ptr(ptr: int, shape, dtype: str):
    """A torch tensor that aliases library-owned device memory (read-only use)."""
    import torch
    td = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    n = 1
    for s in shape:
        n *= s

    class _Holder:
        __cuda_array_interface__ = {"shape": (n,), "typestr": "<i2", "data": (ptr, False),
                                    "version": 3}
    return torch.as_tensor(_Holder(), device="cuda").view(td).view(*shape)


# ---- a small owner object around a plan ---------------------------------------------------

class Plan:
    """A plan with its free() tied to the object (context manager or explicit free())."""

    def __init__(self, m, n, k, dtype="bf16", epilog="BIAS", bias_layout="1N", **options):
        self.m, self.n, self.k = m, n, k
        self.dtype, self.epilog, self.bias_layout = dtype, epilog, bias_layout
        self.handle = gemm_epi_plan(m, n, k, dtype, epilog, bias_layout)
        for key, value in options.items():
            gemm_epi_plan_set_option(self.handle, key.upper(), value)

    def set_option(self, option: str, value: int):
        gemm_epi_plan_set_option(self.handle, option.upper(), value)

    def describe(self) -> str:
        return gemm_epi_plan_describe(self.handle)

    def execute(self, A, B, bias, D, aux=None, residual=None, stream=None, aux_in=None,
                dbias=None, ln=None, scales=None):
        gemm_epi_execute_operands(self.handle, A, B, D, bias=bias, residual=residual, aux=aux,
                                  aux_in=aux_in, dbias=dbias, stream=stream, ln=ln,
                                  scales=scales)

    def execute_host(self, A, B, bias, D, aux=None, residual=None, stream=None):
        gemm_epi_execute_host(self.handle, A, B, D, bias=bias, residual=residual, aux=aux,
                              stream=stream)

    def execute_unfused(self, A, B, bias, pre, D, aux=None, residual=None, stream=None,
                        aux_in=None, dbias=None, ln=None, scales=None):
        gemm_epi_execute_operands_unfused(self.handle, A, B, D, pre, bias=bias, residual=residual,
                                          aux=aux, aux_in=aux_in, dbias=dbias, stream=stream,
                                          ln=ln, scales=scales)

    def sync_status(self, stream=None) -> int:
        return gemm_epi_sync_status(self.handle, stream)

    def free(self):
        if self.handle:
            gemm_epi_free(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass
