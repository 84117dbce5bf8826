"""The allocation-free FFN call.

Some callers cannot allocate device memory: a serving runtime that owns all device memory
through its own pool and forbids cudaMalloc after start-up, or code running where an
allocation would stall or fail.  gemm_epi_ffn_execute_noalloc serves them by keeping the
FFN's hidden activation (and its launches' status words and tile counters) in a static
device array of the library instead of plan-owned allocations.  These tests call it
through the C ABI and compare its output with the planned FFN call (gemm_epi_ffn_plan +
gemm_epi_ffn_execute) on the same inputs, on two calls in a row, and with the CPU oracle,
within the tolerance every parity test uses; they also check that a call leaves the
device's free memory unchanged.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi
from parity_helpers import TOL, rel_err

pytestmark = pytest.mark.gpu

TD = {"bf16": torch.bfloat16, "f16": torch.float16}
DTYPE_CODE = {"f16": 0, "bf16": 1}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _inputs(t, d, f, seed, dtype="bf16"):
    g = torch.Generator().manual_seed(seed)

    def r(*s, sc=1.0):
        return (torch.randn(*s, generator=g) * sc).to(TD[dtype]).cuda()
    return dict(X=r(t, d), W1=r(d, f, sc=0.05), b1=r(f, sc=0.05), W2=r(f, d, sc=0.05),
                b2=r(d, sc=0.05), R=r(t, d))


def _noalloc(lib, t, d, f, x, Y, dtype="bf16"):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.gemm_epi_ffn_execute_noalloc(t, d, f, DTYPE_CODE[dtype], x["X"].data_ptr(),
                                            x["W1"].data_ptr(), x["b1"].data_ptr(),
                                            x["W2"].data_ptr(), x["b2"].data_ptr(),
                                            x["R"].data_ptr(), Y.data_ptr(),
                                            ctypes.c_void_p(stream))


# (t, d, f, dtype): the block workload (CTA-pair kernels), row tiles, the small-m kernel
CASES = [(4096, 1024, 4096, "bf16"), (300, 136, 264, "bf16"), (300, 136, 264, "f16"),
         (64, 256, 512, "bf16")]


@pytest.mark.parametrize("t,d,f,dtype", CASES)
def test_noalloc_ffn_matches_planned_ffn_twice(t, d, f, dtype):
    lib = gemm_epi.load_library()
    x = _inputs(t, d, f, seed=t + f, dtype=dtype)
    ref = torch.empty((t, d), dtype=TD[dtype], device="cuda")
    with gemm_epi.FfnPlan(t, d, f, dtype) as plan:
        plan.execute(x["X"], x["W1"], x["b1"], x["W2"], x["b2"], x["R"], ref)
        assert plan.sync_status() == 0
    want = ref.double().cpu().numpy()
    for call in range(2):
        Y = torch.full((t, d), float("nan"), dtype=TD[dtype], device="cuda")
        assert _noalloc(lib, t, d, f, x, Y, dtype) == 0, f"call {call}"
        torch.cuda.synchronize()
        err = rel_err(Y, want)
        assert err <= TOL[dtype], f"call {call}: rel err {err:.3e}"


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_noalloc_ffn_against_the_oracle(dtype):
    # Y against the oracle's chain; then, with W2 the identity on the first d rows and b2 = R
    # = 0, Y is H's first d columns exactly (one product per element), checked against
    # GELU(X.W1 + b1) itself
    lib = gemm_epi.load_library()
    t, d, f = 300, 136, 264
    x = _inputs(t, d, f, seed=17, dtype=dtype)
    cpu = {k: v.cpu() for k, v in x.items()}
    _, H_exact, Y_ref = oracle.ffn(**cpu, dtype=dtype)
    for call in range(2):
        Y = torch.full((t, d), float("nan"), dtype=TD[dtype], device="cuda")
        assert _noalloc(lib, t, d, f, x, Y, dtype) == 0
        torch.cuda.synchronize()
        assert rel_err(Y, Y_ref) <= TOL[dtype], f"call {call}"
    eye = torch.zeros((f, d), dtype=TD[dtype])
    eye[:d, :d] = torch.eye(d, dtype=TD[dtype])
    xi = dict(x, W2=eye.cuda(), b2=torch.zeros(d, dtype=TD[dtype]).cuda(),
              R=torch.zeros((t, d), dtype=TD[dtype]).cuda())
    Y = torch.full((t, d), float("nan"), dtype=TD[dtype], device="cuda")
    assert _noalloc(lib, t, d, f, xi, Y, dtype) == 0
    torch.cuda.synchronize()
    assert rel_err(Y, H_exact[:, :d]) <= TOL[dtype]
    H_bits, _, Y_h = oracle.ffn(**{k: v.cpu() for k, v in xi.items()}, dtype=dtype)
    assert np.array_equal(Y_h, oracle.decode(dtype, H_bits)[:, :d])  # (the reduction itself)


def test_noalloc_ffn_allocates_no_device_memory():
    lib = gemm_epi.load_library()
    t, d, f = 4096, 1024, 4096
    x = _inputs(t, d, f, seed=5)
    Y = torch.empty((t, d), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, t, d, f, x, Y) == 0        # first call: address look-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc(lib, t, d, f, x, Y) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_ffn_rejects_hidden_beyond_scratch():
    lib = gemm_epi.load_library()
    x = _inputs(8, 8, 8, seed=1)
    Y = torch.empty((8, 8), dtype=torch.bfloat16, device="cuda")
    t, f = 4097, 4096                      # t * f one row over the 16 Mi-element limit
    assert t * f > gemm_epi.FFN_NOALLOC_MAX_HIDDEN
    status = _noalloc(lib, t, 8, f, x, Y)
    assert status == 9                     # GEMM_EPI_ERR_SCRATCH_LIMIT
    assert "scratch" in gemm_epi.status_string(status)
