"""The allocation-free FFN call.

Some callers cannot allocate device memory: a serving runtime that owns all device memory
through its own pool and forbids cudaMalloc after start-up, or code running where an
allocation would stall or fail.  gemm_epi_ffn_execute_noalloc serves them by keeping the
FFN's hidden activation in a static device array of the library instead of a plan-owned
allocation.  These tests call it through the C ABI and compare its output with the planned
FFN call (gemm_epi_ffn_plan + gemm_epi_ffn_execute) on the same inputs, on two calls in a
row, within the bf16 tolerance every parity test uses.  The file is named so that pytest
collects it last.
"""
import ctypes

import pytest
import torch

from activation_epilogue_gb300 import gemm_epi
from parity_helpers import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _inputs(t, d, f, seed):
    g = torch.Generator().manual_seed(seed)

    def r(*s, sc=1.0):
        return (torch.randn(*s, generator=g) * sc).to(torch.bfloat16).cuda()
    return dict(X=r(t, d), W1=r(d, f, sc=0.05), b1=r(f, sc=0.05), W2=r(f, d, sc=0.05),
                b2=r(d, sc=0.05), R=r(t, d))


def _noalloc(lib, t, d, f, x, Y):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.gemm_epi_ffn_execute_noalloc(t, d, f, 1, x["X"].data_ptr(), x["W1"].data_ptr(),
                                            x["b1"].data_ptr(), x["W2"].data_ptr(),
                                            x["b2"].data_ptr(), x["R"].data_ptr(),
                                            Y.data_ptr(), ctypes.c_void_p(stream))


@pytest.mark.parametrize("t,d,f", [(4096, 1024, 4096), (300, 136, 264)])
def test_noalloc_ffn_matches_planned_ffn_twice(t, d, f):
    lib = gemm_epi.load_library()
    x = _inputs(t, d, f, seed=t + f)
    ref = torch.empty((t, d), dtype=torch.bfloat16, device="cuda")
    with gemm_epi.FfnPlan(t, d, f) as plan:
        plan.execute(x["X"], x["W1"], x["b1"], x["W2"], x["b2"], x["R"], ref)
        assert plan.sync_status() == 0
    want = ref.double().cpu().numpy()
    for call in range(2):
        Y = torch.full((t, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, t, d, f, x, Y) == 0, f"call {call}"
        torch.cuda.synchronize()
        err = rel_err(Y, want)
        assert err <= TOL["bf16"], f"call {call}: rel err {err:.3e}"


def test_noalloc_ffn_rejects_hidden_beyond_scratch():
    lib = gemm_epi.load_library()
    x = _inputs(8, 8, 8, seed=1)
    Y = torch.empty((8, 8), dtype=torch.bfloat16, device="cuda")
    t, f = 4097, 4096                      # t * f one row over the 16 Mi-element limit
    assert t * f > gemm_epi.FFN_NOALLOC_MAX_HIDDEN
    status = _noalloc(lib, t, 8, f, x, Y)
    assert status == 9                     # GEMM_EPI_ERR_SCRATCH_LIMIT
    assert "scratch" in gemm_epi.status_string(status)
