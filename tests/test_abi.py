"""The C ABI library, without a GPU: it loads, exports every declared symbol, and its
argument checks reject bad plans before touching a device."""
import os
import re

import pytest

from activation_epilogue_gb300 import build as libbuild
from activation_epilogue_gb300 import gemm_epi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return gemm_epi.load_library()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^[A-Za-z_][\w ]*?\**\s*\b(gemm_epi_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert sorted(gemm_epi.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def _header_enums():
    text = open(os.path.join(ROOT, "include", "gemm_epi.h")).read()
    return {name: int(v) for name, v in re.findall(r"\b(GEMM_EPI_\w+)\s*=\s*(\d+)", text)}


def test_binding_tables_match_the_header():
    """Every enum value the binding passes through the C ABI is the header's, and every
    option the header declares has a binding name."""
    h = _header_enums()
    assert {f"GEMM_EPI_{k.upper()}": v for k, v in gemm_epi.DTYPE.items()} == \
        {k: v for k, v in h.items() if k in ("GEMM_EPI_F16", "GEMM_EPI_BF16", "GEMM_EPI_E4M3")}
    for name, v in gemm_epi.EPILOG.items():
        assert h[f"GEMM_EPI_{name}"] == v, name
    for name, v in gemm_epi.BIAS_LAYOUT.items():
        assert h[f"GEMM_EPI_BIAS_{name}"] == v, name
    for v, name in gemm_epi.STATUS.items():
        assert h[f"GEMM_EPI_{name}"] == v, name
    opts = {k[len("GEMM_EPI_OPT_"):]: v for k, v in h.items() if k.startswith("GEMM_EPI_OPT_")}
    assert opts == gemm_epi.OPTION
    ffn = {k[len("GEMM_EPI_FFN_OPT_"):]: v for k, v in h.items()
           if k.startswith("GEMM_EPI_FFN_OPT_")}
    assert ffn == gemm_epi.FFN_OPTION


def test_status_strings(lib):
    for code, name in gemm_epi.STATUS.items():
        assert name in gemm_epi.status_string(code)
    assert "UNKNOWN" in gemm_epi.status_string(99)


def test_aux_words_per_row(lib):
    assert [gemm_epi.gemm_epi_aux_words_per_row(n) for n in (0, 1, 31, 32, 33, 4096)] == \
        [0, 1, 1, 1, 2, 128]


@pytest.mark.parametrize("args,code", [
    ((-1, 8, 8), 2), ((8, 12, 8), 2), ((8, 8, 12), 2), ((8, 8, -8), 2), ((2 ** 31, 8, 8), 2),
])
def test_bad_shapes_rejected_before_device(lib, args, code):
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.gemm_epi_plan(*args, "bf16", "BIAS", "1N")
    assert e.value.status == code


def test_bad_enums_rejected(lib):
    import ctypes
    h = ctypes.c_void_p()
    assert lib.gemm_epi_plan(ctypes.byref(h), 8, 8, 8, 7, 0, 0) == 1
    assert lib.gemm_epi_plan(ctypes.byref(h), 8, 8, 8, 0, 11, 0) == 1
    assert lib.gemm_epi_plan(ctypes.byref(h), 8, 8, 8, 0, -1, 0) == 1
    assert lib.gemm_epi_plan(ctypes.byref(h), 8, 8, 8, 0, 0, 5) == 1
    assert lib.gemm_epi_plan(None, 8, 8, 8, 0, 0, 0) == 1
    assert h.value is None


def test_null_handles_are_safe(lib):
    import ctypes
    assert lib.gemm_epi_free(None) == 0
    assert lib.gemm_epi_execute(None, None, None, None, None, None, None) == 1
    ops = gemm_epi.Operands()
    assert lib.gemm_epi_execute_operands(None, ctypes.byref(ops), None) == 1
    assert lib.gemm_epi_execute_operands_unfused(None, ctypes.byref(ops), None, None) == 1
    assert lib.gemm_epi_sync_status(None, None) == 1
    assert lib.gemm_epi_plan_set_option(None, 0, 0) == 1
    assert lib.gemm_epi_plan_describe(None) == b""


def test_no_device_reported_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.gemm_epi_plan(64, 64, 64, "bf16", "BIAS", "1N")
    assert e.value.status == 4
