"""The fused call on HOST buffers (gemm_epi_execute_host): chunked, pipelined copies and
GEMMs, checked against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi, workloads
from parity_helpers import AUX_BAND, TD, TOL, aux_bad_bits, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _host(t, pinned=True):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=pinned)
    h.copy_(t)
    return h


def _run_host(p, m, n, k, dtype, epilog, layout, pinned=True, plan=None, options=None):
    A, B = _host(p["A"], pinned), _host(p["B"], pinned)
    bias = _host(p["bias"], pinned) if epilog != "NONE" else None
    R = _host(p["R"], pinned) if epilog == "BIAS_RESIDUAL" else None
    D = torch.full((m, n), float("nan"), dtype=TD[dtype], pin_memory=pinned)
    aux = None
    if epilog == "RELU_AUX_BIAS":
        aux = torch.full((m, (n + 31) // 32), -1, dtype=torch.int32, pin_memory=pinned)
    elif epilog == "GELU_AUX_BIAS":
        aux = torch.full((m, n), float("nan"), dtype=TD[dtype], pin_memory=pinned)
    own = plan is None
    if own:
        plan = gemm_epi.Plan(m, n, k, dtype, epilog, layout, **(options or {}))
    try:
        plan.execute_host(A, B, bias, D, aux=aux, residual=R)
        torch.cuda.current_stream().synchronize()
        assert plan.sync_status() == 0
    finally:
        if own:
            plan.free()
    return D, aux


@pytest.mark.parametrize("m", [300, 5000, 9000])
@pytest.mark.parametrize("epilog,layout", [("BIAS", "M1"), ("RELU_AUX_BIAS", "1N"),
                                           ("BIAS_RESIDUAL", "1N"), ("GELU_AUX_BIAS", "M1"),
                                           ("TANH_BIAS", "1N"), ("NONE", "1N")])
def test_execute_host_parity(m, epilog, layout):
    n, k = 264, 136
    p = workloads.random_problem(m, n, k, dtype="bf16", bias_layout=layout, residual=True,
                                 seed=m + len(epilog))
    D, aux = _run_host(p, m, n, k, "bf16", epilog, layout)
    want, pre = oracle.gemm_epi(p["A"], p["B"], None if epilog == "NONE" else p["bias"],
                                dtype="bf16", epilog=epilog, bias_layout=layout,
                                residual=p["R"] if epilog == "BIAS_RESIDUAL" else None,
                                want_pre=True)
    assert rel_err(D, want) <= TOL["bf16"]
    if epilog == "RELU_AUX_BIAS":
        assert aux_bad_bits(aux.numpy().view(np.uint32), pre, AUX_BAND) == 0
    if epilog == "GELU_AUX_BIAS":
        assert rel_err(aux, pre) <= TOL["bf16"]


def test_execute_host_pageable_memory_and_reuse():
    m, n, k = 3000, 520, 200
    p = workloads.random_problem(m, n, k, dtype="f16", seed=3)
    want = oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="f16", epilog="GELU_BIAS")
    with gemm_epi.Plan(m, n, k, "f16", "GELU_BIAS", "1N") as plan:
        for pinned in (False, True, True):
            D, _ = _run_host(p, m, n, k, "f16", "GELU_BIAS", "1N", pinned=pinned, plan=plan)
            assert rel_err(D, want) <= TOL["f16"]
        plan.set_option("TILE_N", 128)          # the chunk plans are rebuilt
        D, _ = _run_host(p, m, n, k, "f16", "GELU_BIAS", "1N", plan=plan)
        assert rel_err(D, want) <= TOL["f16"]


def test_execute_host_rules():
    h = torch.zeros((64, 64), dtype=torch.bfloat16, pin_memory=True)
    with gemm_epi.Plan(64, 64, 64, "bf16", "DRELU_BGRAD", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.execute_host(h, h, None, h)
        assert e.value.status == 1
    with gemm_epi.Plan(64, 64, 64, "bf16", "BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:        # bias missing
            plan.execute_host(h, h, None, h)
        assert e.value.status == 1
    with gemm_epi.Plan(0, 64, 64, "bf16", "BIAS", "1N") as plan:  # empty: nothing to do
        plan.execute_host(None, None, None, None)


def test_execute_host_large_chunks_pair_kernel():
    # 20 chunks of 1024 rows x 8192 columns, so every one of the three device slots is
    # reused several times: each chunk plan runs the CTA-pair kernel (128 tiles: the static
    # order; the plan itself, on device buffers, 2560 tiles and the dynamic order); rows on
    # and around chunk edges checked by the oracle, and the whole result against the same
    # plan on device buffers
    m, n, k = 20480, 8192, 64
    p = workloads.random_problem(m, n, k, dtype="bf16", bias_layout="1N", residual=False,
                                 seed=2048)
    with gemm_epi.Plan(m, n, k, "bf16", "RELU_AUX_BIAS", "1N") as plan:
        assert "variant=row-pair " in plan.describe() and "order=dynamic" in plan.describe()
        D, aux = _run_host(p, m, n, k, "bf16", "RELU_AUX_BIAS", "1N", plan=plan)
        dev = torch.device("cuda")
        Dd = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        auxd = torch.empty((m, n // 32), dtype=torch.int32, device=dev)
        plan.execute(p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev), Dd, aux=auxd)
        assert plan.sync_status() == 0
    assert torch.equal(D, Dd.cpu())
    assert torch.equal(aux, auxd.cpu())
    rows = [0, 1, 1023, 1024, 1025, 2047, 2048, 3071, 3072, 10239, 10240, 20478, 20479]
    want, pre = oracle.gemm_epi(p["A"][rows], p["B"], p["bias"], dtype="bf16",
                                epilog="RELU_AUX_BIAS", bias_layout="1N", want_pre=True)
    assert rel_err(D[rows], want) <= TOL["bf16"]
    words = aux[rows].numpy().view(np.uint32)
    assert aux_bad_bits(words, pre, AUX_BAND) == 0


@pytest.mark.parametrize("m,n,k,dtype,epilog,layout", [
    (4096, 8192, 2048, "bf16", "RELU_BIAS", "1N"),    # 2 panels of 4096 over 3 chunks
    (4096, 8200, 2048, "f16", "GELU_BIAS", "M1"),     # panels of 4352 and 3848 columns
    (3072, 8192, 2048, "bf16", "NONE", "1N"),         # exactly 3 chunks, all in panels
    (3300, 12288, 2048, "bf16", "TANH_BIAS", "1N"),   # 2 full chunks in panels, a shorter one after
    (8192, 16384, 2048, "bf16", "BIAS", "1N"),        # 2 panels of 8192, then 5 more chunks
])
def test_execute_host_column_panels(m, n, k, dtype, epilog, layout, pinned=True):
    # B of 32 MiB or more: the first chunks' columns of D are computed panel by panel of B
    # while B is still coming in; the whole result must equal the same plan on device
    # buffers bit for bit (the same K order per element), and rows on chunk edges the oracle
    p = workloads.random_problem(m, n, k, dtype=dtype, bias_layout=layout, residual=False,
                                 seed=m + n)
    with gemm_epi.Plan(m, n, k, dtype, epilog, layout) as plan:
        D, _ = _run_host(p, m, n, k, dtype, epilog, layout, plan=plan, pinned=pinned)
        dev = torch.device("cuda")
        Dd = torch.empty((m, n), dtype=TD[dtype], device=dev)
        bias = p["bias"].to(dev) if epilog != "NONE" else None
        plan.execute(p["A"].to(dev), p["B"].to(dev), bias, Dd)
        assert plan.sync_status() == 0
    assert torch.equal(D, Dd.cpu())
    chunks = max(1, min(32, m // 1024))       # the pipeline's rows per chunk
    chunk = min(m, -(-(-(-m // chunks)) // 128) * 128)
    rows = sorted(r for r in {0, 1, chunk - 1, chunk, 2 * chunk - 1, 2 * chunk, 3 * chunk, m - 1}
                  if r < m)
    want = oracle.gemm_epi(p["A"][rows], p["B"], None if epilog == "NONE" else
                           (p["bias"][rows] if layout == "M1" else p["bias"]),
                           dtype=dtype, epilog=epilog, bias_layout=layout)
    assert rel_err(D[rows], want) <= TOL[dtype]


@pytest.mark.parametrize("m,n,k,dtype,epilog,layout", [
    (4096, 8192, 2048, "bf16", "RELU_BIAS", "1N"),
    (3300, 12288, 2048, "f16", "GELU_BIAS", "M1"),
])
def test_execute_host_column_panels_pageable(m, n, k, dtype, epilog, layout):
    # the same with pageable host buffers (the 2-D copies of B's panels and D's columns are
    # staged by the driver)
    test_execute_host_column_panels(m, n, k, dtype, epilog, layout, pinned=False)


def test_execute_host_chunks_with_automatic_split():
    # chunk plans of 1024 x 512 x 2048 take K slices through a cluster and L2 by themselves
    # (each chunk plan owns its workspace); bias along the rows, offset per chunk
    m, n, k = 2048, 512, 2048
    p = workloads.random_problem(m, n, k, dtype="f16", bias_layout="M1", residual=False, seed=77)
    with gemm_epi.Plan(m, n, k, "f16", "BIAS", "M1") as plan:
        D, _ = _run_host(p, m, n, k, "f16", "BIAS", "M1", plan=plan)
        dev = torch.device("cuda")
        Dd = torch.empty((m, n), dtype=torch.float16, device=dev)
        plan.execute(p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev), Dd)
        assert plan.sync_status() == 0
    rows = [0, 1, 1023, 1024, 1025, 2047]
    want = oracle.gemm_epi(p["A"][rows], p["B"], p["bias"][rows], dtype="f16", epilog="BIAS",
                           bias_layout="M1")
    assert rel_err(D[rows], want) <= TOL["f16"]
    assert rel_err(Dd.cpu()[rows], want) <= TOL["f16"]
