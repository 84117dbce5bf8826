"""GPU parity of the E4M3 (FP8) path with per-tensor scales: D = epi(sa * sb * (A.B) + bias),
A m x k and B transposed (n x k) in E4M3, bias / residual / D in bfloat16, against the CPU
oracle."""
import numpy as np
import pytest
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi, workloads
from parity_helpers import AUX_BAND, TOL, aux_bad_bits, rel_err

pytestmark = pytest.mark.gpu

EPILOGS = ["BIAS", "RELU_BIAS", "GELU_BIAS", "RELU_AUX_BIAS", "BIAS_RESIDUAL", "NONE"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _run(p, m, n, k, epilog, layout, unfused=False, options=None):
    dev = torch.device("cuda")
    A, Bt = p["A"].to(dev), p["Bt"].to(dev)
    sa = torch.tensor([p["scale_a"]], dtype=torch.float32, device=dev)
    sb = torch.tensor([p["scale_b"]], dtype=torch.float32, device=dev)
    bias = p["bias"].to(dev) if epilog != "NONE" else None
    R = p["R"].to(dev) if epilog == "BIAS_RESIDUAL" else None
    D = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=dev)
    aux = (torch.full((m, (n + 31) // 32), -1, dtype=torch.int32, device=dev)
           if epilog == "RELU_AUX_BIAS" else None)
    with gemm_epi.Plan(m, n, k, "e4m3", epilog, layout, **(options or {})) as plan:
        if unfused:
            pre = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            plan.execute_unfused(A, Bt, bias, pre, D, aux=aux, residual=R, scales=(sa, sb))
        else:
            plan.execute(A, Bt, bias, D, aux=aux, residual=R, scales=(sa, sb))
        assert plan.sync_status() == 0
        desc = plan.describe()
    words = None if aux is None else aux.cpu().numpy().view(np.uint32)
    return D.cpu(), words, desc


def _check(p, m, n, k, epilog, layout, unfused=False, options=None):
    D, words, desc = _run(p, m, n, k, epilog, layout, unfused, options)
    want, pre = oracle.gemm_epi_fp8(p["A"], p["Bt"], p["bias"] if epilog != "NONE" else None,
                                    scale_a=p["scale_a"], scale_b=p["scale_b"], epilog=epilog,
                                    bias_layout=layout, residual=p.get("R"), want_pre=True)
    err = rel_err(D, want)
    slack = 0.0
    if unfused:
        # the unfused GEMM rounds sa sb A.B to bf16 before the epilogue pass
        pre0 = oracle.gemm_epi_fp8(p["A"], p["Bt"], None, scale_a=p["scale_a"],
                                   scale_b=p["scale_b"], epilog="NONE")
        slack = 2.0 ** -8 * np.abs(pre0)
    got = D.double().numpy()
    assert np.all(np.abs(got - want) <= TOL["bf16"] * (np.abs(want) + 1) + slack), \
        f"rel err {err:.3e} ({desc})"
    if words is not None:
        band = AUX_BAND + (2 * slack if unfused else 0.0)
        assert aux_bad_bits(words, pre, band) == 0, desc
    return D, want, desc


@pytest.mark.parametrize("epilog", EPILOGS)
@pytest.mark.parametrize("shape", [(300, 520, 208), (600, 264, 1040), (16, 264, 128), (1, 8, 16)])
def test_fp8_parity(epilog, shape):
    m, n, k = shape
    layout = "M1" if (len(epilog) + m) % 2 else "1N"
    p = workloads.random_fp8_problem(m, n, k, bias_layout=layout, seed=m + n + k + len(epilog),
                                     residual=True)
    _, _, desc = _check(p, m, n, k, epilog, layout)
    assert "dtype=e4m3" in desc and "variant=row-pair" in desc


@pytest.mark.parametrize("epilog", EPILOGS)
@pytest.mark.parametrize("shape", [(1000, 520, 208), (600, 264, 1040), (300, 776, 400)])
def test_fp8_static_tile_order(epilog, shape):
    # the pair kernel with the static tile order (the automatic one is the dynamic order)
    m, n, k = shape
    layout = "M1" if (len(epilog) + m) % 3 == 0 else "1N"
    p = workloads.random_fp8_problem(m, n, k, bias_layout=layout, seed=m + n + k + 7 * len(epilog),
                                     residual=True)
    _, _, desc = _check(p, m, n, k, epilog, layout, options={"TILE_ORDER": 1})
    assert "dtype=e4m3" in desc and "order=static" in desc


@pytest.mark.parametrize("order", [1, 2])
def test_fp8_walk(order):
    m, n, k = 2304, 1000, 512          # 9 row tiles, 4 column tiles, few pairs walking
    p = workloads.random_fp8_problem(m, n, k, bias_layout="1N", seed=2304, residual=True)
    _check(p, m, n, k, "RELU_AUX_BIAS", "1N", options={"GRID": 8, "TILE_ORDER": order})


@pytest.mark.parametrize("m,n,order", [(65536, 16384, "dynamic"), (4096, 4096, "static"),
                                       (1024, 1024, "static")])
def test_fp8_plan_is_a_pair_plan(m, n, order):
    # the tile counter from eight waves of tiles over the pairs up
    with gemm_epi.Plan(m, n, 8192, "e4m3", "RELU_BIAS", "1N") as plan:
        d = plan.describe()
        assert "variant=row-pair " in d and f"order={order}" in d, d


@pytest.mark.parametrize("bn", [224, 256])
@pytest.mark.parametrize("epilog", ["RELU_AUX_BIAS", "GELU_BIAS", "BIAS_RESIDUAL"])
@pytest.mark.parametrize("shape", [(600, 520, 272), (300, 1000, 400), (520, 232, 1040)])
def test_fp8_tile_widths(epilog, shape, bn):
    # 256 x 224 tiles: each CTA's half of B is 112 rows, loaded in 128-row boxes (the 16 extra
    # rows belong to the next tile or lie past the edge); n = 520, 1000, 232 leave ragged
    # last column tiles at both widths
    m, n, k = shape
    layout = "M1" if (m + bn) % 3 == 0 else "1N"
    p = workloads.random_fp8_problem(m, n, k, bias_layout=layout, seed=m + n + k + bn,
                                     residual=True)
    _, _, desc = _check(p, m, n, k, epilog, layout, options={"TILE_N": bn})
    assert f"tile=256x{bn} " in desc, desc


def test_fp8_integer_bit_exact_224():
    m, n, k = 520, 1000, 64
    g = torch.Generator().manual_seed(224)
    p = {"A": torch.randint(-4, 5, (m, k), generator=g).float().to(torch.float8_e4m3fn),
         "Bt": torch.randint(-4, 5, (n, k), generator=g).float().to(torch.float8_e4m3fn),
         "scale_a": 1.0, "scale_b": 1.0,
         "bias": torch.randint(-8, 9, (n,), generator=g).to(torch.bfloat16)}
    D, _, desc = _run(p, m, n, k, "RELU_BIAS", "1N", options={"TILE_N": 224})
    assert "tile=256x224 " in desc
    want = oracle.gemm_epi_fp8(p["A"], p["Bt"], p["bias"], scale_a=1.0, scale_b=1.0,
                               epilog="RELU_BIAS")
    assert np.array_equal(D.double().numpy(), want), desc


@pytest.mark.parametrize("m,n,bn", [(4096, 4096, 224), (65536, 16384, 256), (2048, 2048, 256)])
def test_fp8_tile_width_choice(m, n, bn):
    # the width with fewer waves of tiles over the pairs (224 on a tie): 4096 x 4096 is
    # 304 tiles of 224 (4 waves) against 256 of 256 (3.4, paid as 4); 2048 x 2048 is 64
    # tiles of 256 (one wave) against 80 of 224 (two)
    with gemm_epi.Plan(m, n, 8192, "e4m3", "RELU_BIAS", "1N") as plan:
        assert f"tile=256x{bn} " in plan.describe(), plan.describe()


@pytest.mark.parametrize("epilog", ["RELU_AUX_BIAS", "BIAS_RESIDUAL", "GELU_BIAS"])
def test_fp8_unfused(epilog):
    m, n, k = 300, 264, 208
    p = workloads.random_fp8_problem(m, n, k, seed=77, residual=True)
    _check(p, m, n, k, epilog, "1N", unfused=True)


def test_fp8_integer_bit_exact():
    # integers in {-4..4} are exact in E4M3; with k = 64 and unit scales every sum is an
    # exact integer below 2^10, exact in bfloat16 too
    m, n, k = 520, 264, 64
    g = torch.Generator().manual_seed(5)
    p = {"A": torch.randint(-4, 5, (m, k), generator=g).float().to(torch.float8_e4m3fn),
         "Bt": torch.randint(-4, 5, (n, k), generator=g).float().to(torch.float8_e4m3fn),
         "scale_a": 1.0, "scale_b": 1.0,
         "bias": torch.randint(-8, 9, (n,), generator=g).to(torch.bfloat16)}
    D, _, desc = _run(p, m, n, k, "RELU_BIAS", "1N")
    want = oracle.gemm_epi_fp8(p["A"], p["Bt"], p["bias"], scale_a=1.0, scale_b=1.0,
                               epilog="RELU_BIAS")
    assert np.array_equal(D.double().numpy(), want), desc


def test_fp8_only_the_product_of_the_scales_matters():
    m, n, k = 256, 256, 256
    p = workloads.random_fp8_problem(m, n, k, seed=9)
    p1 = dict(p, scale_a=0.5, scale_b=4.0)
    p2 = dict(p, scale_a=2.0, scale_b=1.0)
    D1, _, _ = _run(p1, m, n, k, "BIAS", "1N")
    D2, _, _ = _run(p2, m, n, k, "BIAS", "1N")
    assert torch.equal(D1, D2)


def test_fp8_full_2048():
    m = n = k = 2048
    p = workloads.random_fp8_problem(m, n, k, seed=2048, residual=True)
    _check(p, m, n, k, "GELU_BIAS", "1N")


def test_fp8_rules():
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.Plan(64, 64, 64, "e4m3", "GELU_AUX_BIAS", "1N")
    assert e.value.status == 1
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.Plan(64, 64, 24, "e4m3", "BIAS", "1N")
    assert e.value.status == 2
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.Plan(64, 64, 64, "e4m3", "BIAS", "1N", VARIANT=1)
    assert e.value.status == 1
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.Plan(64, 64, 64, "e4m3", "BIAS", "1N", TILE_N=128)
    assert e.value.status == 1
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.FfnPlan(64, 64, 64, "e4m3")
    assert e.value.status == 1
    dev = torch.device("cuda")
    A = torch.zeros((64, 64), dtype=torch.uint8, device=dev)
    D = torch.empty((64, 64), dtype=torch.bfloat16, device=dev)
    b = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    s = torch.ones(1, dtype=torch.float32, device=dev)
    with gemm_epi.Plan(64, 64, 64, "e4m3", "BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:     # scales missing
            plan.execute(A, A, b, D)
        assert e.value.status == 1
        plan.execute(A, A, b, D, scales=(s, s))
        assert plan.sync_status() == 0
        assert torch.equal(D.cpu(), torch.zeros(64, 64, dtype=torch.bfloat16))


@pytest.mark.parametrize("i", range(16))
def test_fp8_random_cases(i):
    # seeded random shapes (k a multiple of 16), epilogs, layouts, both tile orders
    import random
    r = random.Random(7000 + i)
    m, n, k = r.randint(1, 900), 8 * r.randint(1, 100), 16 * r.randint(1, 40)
    epilog = r.choice(EPILOGS)
    layout = r.choice(["M1", "1N"])
    opts = {"VARIANT": 3, "TILE_ORDER": r.choice([1, 2])}
    if r.random() < 0.3:
        opts["GRID"] = r.choice([4, 8])
    if r.random() < 0.5:
        opts["TILE_N"] = r.choice([224, 256])
    p = workloads.random_fp8_problem(m, n, k, bias_layout=layout, seed=r.randint(0, 10 ** 6),
                                     residual=True)
    _check(p, m, n, k, epilog, layout, options=opts)
