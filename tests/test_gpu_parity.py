"""GPU parity: the fused kernels through the C ABI against the CPU oracle, element by element,
at sizes that span several tiles and ragged tails in M, N and K."""
import numpy as np
import pytest
import torch

from activation_epilogue_gb300 import gemm_epi, workloads
from parity_helpers import TD, TOL, check, rel_err, run

pytestmark = pytest.mark.gpu

EPILOGS = ["BIAS", "RELU_BIAS", "GELU_BIAS", "RELU_AUX_BIAS", "BIAS_RESIDUAL", "NONE", "TANH_BIAS",
           "GELU_AUX_BIAS"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _inputs(m, n, k, dtype, layout, seed, kind="normal"):
    return workloads.random_problem(m, n, k, dtype=dtype, bias_layout=layout, residual=True,
                                    seed=seed, kind=kind)


# ---- row-tile kernel: every N tile width, epilog, dtype and both bias layouts --------------

@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("epilog", EPILOGS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rowtile_parity(bn, epilog, dtype):
    m, n, k = 300, 520, 200            # 3 ragged M tiles, ragged N tiles, 4 K blocks (last 8)
    layout = "M1" if (bn // 64 + EPILOGS.index(epilog)) % 2 else "1N"
    p = _inputs(m, n, k, dtype, layout, seed=bn + 7 * EPILOGS.index(epilog))
    check(p, m, n, k, dtype, epilog, layout, options={"VARIANT": 1, "TILE_N": bn})


@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_rowtile_both_layouts_relu_aux(layout):
    m, n, k = 384, 264, 136
    p = _inputs(m, n, k, "bf16", layout, seed=5)
    check(p, m, n, k, "bf16", "RELU_AUX_BIAS", layout, options={"VARIANT": 1, "TILE_N": 128})


# ---- swapped small-m kernel -----------------------------------------------------------------

@pytest.mark.parametrize("m", [1, 16, 20, 64, 100, 256])
@pytest.mark.parametrize("epilog", EPILOGS)
def test_swapped_parity(m, epilog):
    n, k = 520, 200
    layout = "M1" if (m + EPILOGS.index(epilog)) % 2 else "1N"
    p = _inputs(m, n, k, "bf16", layout, seed=1000 + m)
    check(p, m, n, k, "bf16", epilog, layout, options={"VARIANT": 2})


def test_swapped_f16():
    m, n, k = 48, 392, 264
    p = _inputs(m, n, k, "f16", "1N", seed=77)
    check(p, m, n, k, "f16", "GELU_BIAS", "1N", options={"VARIANT": 2})


# ---- small-m kernel: K split over a cluster, partial sums added in the leader CTA ---------

@pytest.mark.parametrize("m", [1, 7, 16, 20, 33, 64])
@pytest.mark.parametrize("epilog", EPILOGS)
def test_smallm_parity(m, epilog):
    n, k = 392, 1000                   # ragged column tile, 16 K blocks (last one 40 deep)
    layout = "M1" if (m + EPILOGS.index(epilog)) % 2 else "1N"
    dtype = "f16" if (m + EPILOGS.index(epilog)) % 3 == 0 else "bf16"
    p = _inputs(m, n, k, dtype, layout, seed=2000 + m + 31 * EPILOGS.index(epilog))
    _, _, _, _, desc = check(p, m, n, k, dtype, epilog, layout, options={"VARIANT": 5})
    assert "variant=small-m" in desc, desc


@pytest.mark.parametrize("split,effective", [(2, 2), (3, 2), (4, 4), (5, 4), (6, 4), (7, 4),
                                             (8, 8)])
def test_smallm_every_split(split, effective):
    # 16 K blocks (the last one 40 deep) in slices of 8, 4 or 2 blocks; each rank owns
    # 32 / split rows of D (a multiple of 4), so other splits are lowered to the next one
    m, n, k = 24, 776, 1000
    p = _inputs(m, n, k, "bf16", "1N", seed=2100 + split)
    _, _, _, _, desc = check(p, m, n, k, "bf16", "GELU_BIAS", "1N",
                             options={"VARIANT": 5, "SPLIT_K": split})
    assert f"split_k={effective}(cluster)" in desc, desc


@pytest.mark.parametrize("bn", [16, 32, 64])
def test_smallm_row_tile_widths(bn):
    m, n, k = 12, 264, 200
    p = _inputs(m, n, k, "bf16", "M1", seed=2200 + bn)
    _, _, _, _, desc = check(p, m, n, k, "bf16", "RELU_AUX_BIAS", "M1",
                             options={"VARIANT": 5, "TILE_N": bn})
    assert f"tile=128x{bn} " in desc, desc


@pytest.mark.parametrize("epilog", ["BIAS", "RELU_BIAS", "RELU_AUX_BIAS", "BIAS_RESIDUAL", "NONE"])
def test_smallm_integer_bit_exact(epilog):
    m, n, k = 40, 520, 512             # 8 K blocks over a cluster: exact fp32 partial sums
    p = _inputs(m, n, k, "bf16", "1N", seed=2300, kind="int")
    check(p, m, n, k, "bf16", epilog, "1N", options={"VARIANT": 5}, exact=True)


@pytest.mark.parametrize("t", [16, 64])
def test_smallm_workload_shape_deterministic(t):
    # the GELU workload shape: repeated calls give the same bits (the partial sums are added
    # in slice order, whichever CTA stores first)
    m, n, k = t, 3072, 768
    p = _inputs(m, n, k, "bf16", "1N", seed=3000 + t)
    dev = torch.device("cuda")
    A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
    outs = []
    with gemm_epi.Plan(m, n, k, "bf16", "GELU_BIAS", "1N") as plan:
        assert "variant=small-m" in plan.describe()
        for _ in range(3):
            D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            plan.execute(A, B, bias, D)
            outs.append(D.cpu())
        assert plan.sync_status() == 0
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    from parity_helpers import oracle_ref
    want, _ = oracle_ref(p, "bf16", "GELU_BIAS", "1N")
    assert rel_err(outs[0], want) <= TOL["bf16"]


def test_smallm_option_rules():
    with gemm_epi.Plan(16, 264, 136, "bf16", "DRELU_BGRAD", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("VARIANT", 5)     # no backward epilogue in the small-m kernel
        assert e.value.status == 1
    with gemm_epi.Plan(100, 264, 136, "bf16", "BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("VARIANT", 5)     # m > 64
        assert e.value.status == 1
    with gemm_epi.Plan(16, 264, 136, "bf16", "BIAS", "1N", variant=5) as plan:
        plan.set_option("SPLIT_K", 4)         # 3 K blocks, 16 rows: lowered to 2 slices
        assert "variant=small-m" in plan.describe() and "split_k=2(cluster)" in plan.describe()
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("TILE_N", 8)
        assert e.value.status == 1
        assert "split_k=2(cluster)" in plan.describe()  # previous configuration kept
    with gemm_epi.Plan(16, 264, 1024, "bf16", "BIAS", "1N", variant=5) as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("SPLIT_K", 1)     # one 1024-deep slab per CTA does not fit
        assert e.value.status == 1
    with gemm_epi.Plan(16, 264, 16384, "bf16", "BIAS", "1N") as plan:
        # K slabs of 2048 do not fit in shared memory: not the small-m kernel; over 256 K
        # blocks, row tiles with K split over a cluster (the swapped kernel would stream
        # each 128-column panel of B through one of 3 SMs)
        d = plan.describe()
        assert "variant=row-tile" in d and "(cluster+L2)" in d, d
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("VARIANT", 5)
        assert e.value.status == 1


def test_smallm_timeout_path():
    # a launch whose copies never arrive runs out the wait limit and reports it; the next
    # launch of the same plan is correct
    m, n, k = 16, 520, 512
    p = _inputs(m, n, k, "bf16", "1N", seed=2400)
    dev = torch.device("cuda")
    A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
    D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "BIAS", "1N", variant=5) as plan:
        assert "split_k=" in plan.describe() and "split_k=1 " not in plan.describe()
        plan.set_option("WAIT_LIMIT_US", 20000)
        plan.set_option("DEBUG_STALL", 1)
        plan.execute(A, B, bias, D)
        assert plan.sync_status() == 8
        plan.set_option("DEBUG_STALL", 0)
        plan.execute(A, B, bias, D)
        assert plan.sync_status() == 0
    from parity_helpers import oracle_ref
    want, _ = oracle_ref(p, "bf16", "BIAS", "1N")
    assert rel_err(D, want) <= TOL["bf16"]


# ---- integer inputs: every correct result is bit-exact ------------------------------------

@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("epilog", ["BIAS", "RELU_BIAS", "RELU_AUX_BIAS", "BIAS_RESIDUAL", "NONE"])
def test_integer_inputs_bit_exact(variant, epilog):
    m, n, k = (200 if variant == 1 else 40), 136, 64
    p = _inputs(m, n, k, "bf16", "1N", seed=3, kind="int")
    check(p, m, n, k, "bf16", epilog, "1N", options={"VARIANT": variant}, exact=True)
    # the unfused baseline rounds A.B to bf16 first; with |A.B| <= 256 that is exact too
    check(p, m, n, k, "bf16", epilog, "1N", options={"VARIANT": variant}, exact=True,
          unfused=True)


# ---- unfused baseline -----------------------------------------------------------------------

@pytest.mark.parametrize("epilog", EPILOGS)
def test_unfused_parity(epilog):
    m, n, k = 300, 264, 136
    p = _inputs(m, n, k, "bf16", "1N", seed=21)
    check(p, m, n, k, "bf16", epilog, "1N", unfused=True)


# ---- persistence: few CTAs walking many tiles (accumulator and ring phases wrap) ----------

@pytest.mark.parametrize("grid,group_m", [(1, 1), (3, 2), (7, 16)])
def test_persistent_tile_walk(grid, group_m):
    m, n, k = 640, 512, 520            # 5 x 4 tiles of 128 x 128, 9 K blocks
    p = _inputs(m, n, k, "bf16", "1N", seed=grid)
    check(p, m, n, k, "bf16", "RELU_AUX_BIAS", "1N",
          options={"VARIANT": 1, "TILE_N": 128, "GRID": grid, "GROUP_M": group_m})


# ---- edge cases ---------------------------------------------------------------------------

@pytest.mark.parametrize("m,n,k", [(1, 8, 8), (5, 8, 8), (129, 8, 8), (257, 40, 8), (300, 33 * 8, 72)])
@pytest.mark.parametrize("epilog", ["RELU_AUX_BIAS", "GELU_BIAS", "BIAS_RESIDUAL"])
def test_small_and_ragged(m, n, k, epilog):
    p = _inputs(m, n, k, "bf16", "M1", seed=m + n + k)
    check(p, m, n, k, "bf16", epilog, "M1")


@pytest.mark.parametrize("epilog", ["BIAS", "RELU_AUX_BIAS", "GELU_BIAS", "BIAS_RESIDUAL",
                                    "GELU_AUX_BIAS"])
@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_k_zero_is_activation_of_bias(epilog, layout):
    m, n = 70, 72
    p = _inputs(m, n, 0, "bf16", layout, seed=4)
    check(p, m, n, 0, "bf16", epilog, layout)


def test_empty_problem_launches_nothing():
    dev = torch.device("cuda")
    for m, n in [(0, 64), (64, 0)]:
        D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        with gemm_epi.Plan(m, n, 64, "bf16", "BIAS", "1N") as plan:
            A = torch.empty((m, 64), dtype=torch.bfloat16, device=dev)
            B = torch.empty((64, n), dtype=torch.bfloat16, device=dev)
            b = torch.empty((max(n, 1),), dtype=torch.bfloat16, device=dev)
            plan.execute(A, B, b, D)
            assert plan.sync_status() == 0
            assert "empty" in plan.describe()


def test_residual_in_place():
    m, n, k = 260, 264, 128
    p = _inputs(m, n, k, "bf16", "1N", seed=9)
    dev = torch.device("cuda")
    A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
    R = p["R"].to(dev)
    with gemm_epi.Plan(m, n, k, "bf16", "BIAS_RESIDUAL", "1N") as plan:
        plan.execute(A, B, bias, R, residual=R)       # D is the residual buffer
        assert plan.sync_status() == 0
    from parity_helpers import oracle_ref
    want, _ = oracle_ref(p, "bf16", "BIAS_RESIDUAL", "1N")
    assert rel_err(R, want) <= TOL["bf16"]


# ---- closed forms on the GPU ----------------------------------------------------------------

@pytest.mark.parametrize("variant", [1, 2])
def test_zero_A_gives_exact_broadcast_bias(variant):
    m, n, k = (200 if variant == 1 else 24), 136, 64
    p = _inputs(m, n, k, "f16", "M1", seed=11)
    p["A"] = torch.zeros_like(p["A"])
    D, _, _ = run(p, m, n, k, "f16", "BIAS", "M1", options={"VARIANT": variant})
    want = p["bias"][:, None].expand(m, n)
    assert torch.equal(D, want)


def test_identity_B_gives_A_plus_bias():
    m, n = 192, 128
    p = _inputs(m, n, n, "bf16", "1N", seed=12)
    p["B"] = torch.eye(n, dtype=torch.bfloat16)
    check(p, m, n, n, "bf16", "BIAS", "1N")


def test_gelu_textbook_points_through_the_kernel():
    # A = I (m = k), B holds chosen x values, bias = 0, so pre = x and D = GELU(x).
    xs = torch.tensor([-3.0, -2.0, -1.5, -1.0, -0.5, 0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0],
                      dtype=torch.float64)
    m = k = 16
    n = 16
    Bx = torch.zeros(k, n, dtype=torch.float64)
    Bx[: len(xs), 0] = xs
    inputs = {"A": torch.eye(m, dtype=torch.float16), "B": Bx.to(torch.float16),
              "bias": torch.zeros(n, dtype=torch.float16)}
    D, _, _ = run(inputs, m, n, k, "f16", "GELU_BIAS", "1N")
    from scipy.special import ndtr
    want = xs.numpy() * ndtr(xs.numpy())
    got = D[: len(xs), 0].double().numpy()
    # binary16 rounding of the output: 2^-11 relative, plus fp32 erf error
    assert np.max(np.abs(got - want) / (np.abs(want) + 1)) < 1.2e-3


def test_gelu_accuracy_on_a_dense_grid():
    """16384 pre-activations in [-12, 12] through the fused kernel (A = I, bias = 0, f16):
    the kernel's GELU is within 3.1e-5 * max(1, |x|) of x * Phi(x), plus the f16 rounding
    of the output."""
    from scipy.special import ndtr
    m = k = 16
    n = 1024
    xs = torch.linspace(-12.0, 12.0, m * n, dtype=torch.float64).to(torch.float16)
    inputs = {"A": torch.eye(m, dtype=torch.float16), "B": xs.reshape(k, n),
              "bias": torch.zeros(n, dtype=torch.float16)}
    for variant in (1, 3):
        D, _, desc = run(inputs, m, n, k, "f16", "GELU_BIAS", "1N",
                         options={"VARIANT": variant} if variant != 1 else None)
        x = xs.double().numpy().reshape(k, n)
        want = x * ndtr(x)
        got = D.double().numpy()
        bound = 3.1e-5 * np.maximum(1.0, np.abs(x)) + 2.0 ** -11 * np.abs(want) + 6e-8
        bad = np.abs(got - want) > bound
        assert not bad.any(), (desc, x[bad][:5], got[bad][:5], want[bad][:5])


# ---- the timeout path -----------------------------------------------------------------------

def test_device_wait_limit_reports_timeout_and_context_survives():
    m, n, k = 256, 256, 128
    p = _inputs(m, n, k, "bf16", "1N", seed=13)
    dev = torch.device("cuda")
    A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
    D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "BIAS", "1N", variant=1) as plan:
        plan.set_option("WAIT_LIMIT_US", 20000)      # 20 ms
        plan.set_option("DEBUG_STALL", 1)
        plan.execute(A, B, bias, D)
        assert plan.sync_status() == 8             # GEMM_EPI_ERR_DEVICE_TIMEOUT
        assert plan.sync_status() == 0             # reading clears it
        plan.set_option("DEBUG_STALL", 0)
    # the context is still usable
    check(p, m, n, k, "bf16", "BIAS", "1N")


# ---- host-side validation with a device -----------------------------------------------------

def test_execute_argument_errors():
    dev = torch.device("cuda")
    m, n, k = 64, 64, 64
    A = torch.zeros((m, k), dtype=torch.bfloat16, device=dev)
    B = torch.zeros((k, n), dtype=torch.bfloat16, device=dev)
    b = torch.zeros((n,), dtype=torch.bfloat16, device=dev)
    D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    aux = torch.empty((m, 2), dtype=torch.int32, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "RELU_AUX_BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.execute(A, B, b, D)                               # aux missing
        assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.execute(A, B, None, D, aux=aux)                   # bias missing
        assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.execute(A.data_ptr() + 2, B, b, D, aux=aux)       # misaligned A
        assert e.value.status == 3
    with gemm_epi.Plan(m, n, k, "bf16", "BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.execute(A, B, b, D, aux=aux)                      # aux not allowed
        assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("TILE_N", 96)
        assert e.value.status == 1
    with gemm_epi.Plan(300, n, k, "bf16", "BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError):
            plan.set_option("VARIANT", 2)                          # swapped needs m <= 256
        assert "row-tile" in plan.describe()                       # previous config kept


# ---- the FFN entry points -------------------------------------------------------------------

@pytest.mark.parametrize("launches", [0, 1, 2])
@pytest.mark.parametrize("t,d,f", [(300, 136, 264), (16, 256, 520), (1, 8, 8), (520, 264, 776)])
def test_ffn_plan_parity(t, d, f, launches):
    import oracle
    g = torch.Generator().manual_seed(t + d + f)

    def r(*s, sc=1.0):
        return (torch.randn(*s, generator=g) * sc).to(torch.bfloat16)
    cpu = dict(X=r(t, d), W1=r(d, f, sc=0.1), b1=r(f, sc=0.1), W2=r(f, d, sc=0.1),
               b2=r(d, sc=0.1), R=r(t, d))
    dev = torch.device("cuda")
    gi = {k: v.to(dev) for k, v in cpu.items()}
    Y = torch.empty((t, d), dtype=torch.bfloat16, device=dev)
    with gemm_epi.FfnPlan(t, d, f, launches=launches) as plan:
        if launches:
            assert plan.describe().startswith("one launch" if launches == 1 else "two launches")
        plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
        assert plan.sync_status() == 0
        H = plan.hidden().cpu()
        # twice in a row: the second call must give the same result
        Y1 = Y.clone()
        plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
        assert plan.sync_status() == 0
        assert torch.equal(Y, Y1)
    H_ref, H_exact, Y_ref = oracle.ffn(**cpu)
    assert rel_err(H, H_exact) <= TOL["bf16"]
    assert rel_err(Y, Y_ref) <= TOL["bf16"]
    Y2 = oracle.gemm_epi(H, cpu["W2"], cpu["b2"], dtype="bf16", epilog="BIAS_RESIDUAL",
                         residual=cpu["R"])
    assert rel_err(Y, Y2) <= TOL["bf16"]


@pytest.mark.parametrize("launches", [1, 2])
def test_ffn_in_place_on_residual(launches):
    t, d, f = 200, 128, 256
    g = torch.Generator().manual_seed(5)
    dev = torch.device("cuda")

    def r(*s, sc=1.0):
        return (torch.randn(*s, generator=g) * sc).to(torch.bfloat16)
    cpu = dict(X=r(t, d), W1=r(d, f, sc=0.1), b1=r(f, sc=0.1), W2=r(f, d, sc=0.1),
               b2=r(d, sc=0.1), R=r(t, d))
    gi = {k: v.to(dev) for k, v in cpu.items()}
    with gemm_epi.FfnPlan(t, d, f, launches=launches) as plan:
        plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], gi["R"])
        assert plan.sync_status() == 0
    import oracle
    _, _, Y_ref = oracle.ffn(**cpu)
    assert rel_err(gi["R"], Y_ref) <= TOL["bf16"]


def test_ffn_one_launch_many_row_blocks_few_pairs():
    """Few CTA pairs walking many GEMM-1 and GEMM-2 tiles: GEMM-2 tiles wait on row blocks
    that other pairs (and the same pair, earlier) finish; also repeated calls reuse the
    zeroed counters."""
    import oracle
    t, d, f = 1300, 520, 1032
    g = torch.Generator().manual_seed(44)

    def r(*s, sc=1.0):
        return (torch.randn(*s, generator=g) * sc).to(torch.bfloat16)
    cpu = dict(X=r(t, d, sc=0.5), W1=r(d, f, sc=0.05), b1=r(f, sc=0.1), W2=r(f, d, sc=0.05),
               b2=r(d, sc=0.1), R=r(t, d))
    dev = torch.device("cuda")
    gi = {k: v.to(dev) for k, v in cpu.items()}
    Y = torch.empty((t, d), dtype=torch.bfloat16, device=dev)
    with gemm_epi.FfnPlan(t, d, f, launches=1) as plan:
        for _ in range(3):
            plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
        assert plan.sync_status() == 0
        H = plan.hidden().cpu()
    H_ref, H_exact, Y_ref = oracle.ffn(**cpu)
    assert rel_err(H, H_exact) <= TOL["bf16"]
    assert rel_err(Y, Y_ref) <= TOL["bf16"]


def test_ffn_option_rules():
    with gemm_epi.FfnPlan(300, 136, 264) as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            gemm_epi.gemm_epi_ffn_set_option(plan.handle, "LAUNCHES", 4)
        assert e.value.status == 1
        assert "in 1 K slice of" in plan.describe() or plan.describe().startswith("two")
        for bad in (3, 5, 8, -1):
            with pytest.raises(gemm_epi.GemmEpiError) as e:
                gemm_epi.gemm_epi_ffn_set_option(plan.handle, "SPLIT2", bad)
            assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            gemm_epi.gemm_epi_ffn_set_option(plan.handle, "TILE_ORDER", 3)
        assert e.value.status == 1
        gemm_epi.gemm_epi_ffn_set_option(plan.handle, "LAUNCHES", 2)
        assert plan.describe().startswith("two launches")


@pytest.mark.parametrize("t,d,f", [(300, 256, 512), (130, 512, 256), (1, 256, 256),
                                   (520, 1024, 768)])
def test_ffn_onchip_parity(t, d, f):
    """H kept on chip (LAUNCHES = 3): Y against the oracle's chain (which rounds H to bf16 as
    the kernel does); ragged token counts; repeated calls give the same bits."""
    import oracle
    cpu = _ffn_inputs(t, d, f, 11 * t + d + f)
    dev = torch.device("cuda")
    gi = {k: v.to(dev) for k, v in cpu.items()}
    Y = torch.full((t, d), float("nan"), dtype=torch.bfloat16, device=dev)
    with gemm_epi.FfnPlan(t, d, f, launches=3) as plan:
        assert plan.describe().startswith("one launch, H on chip"), plan.describe()
        plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
        assert plan.sync_status() == 0
        Y1 = Y.clone()
        plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
        assert plan.sync_status() == 0
        assert torch.equal(Y, Y1)
    _, _, Y_ref = oracle.ffn(**cpu)
    assert rel_err(Y, Y_ref) <= TOL["bf16"]


@pytest.mark.parametrize("launches", [1, 2, 3])
def test_ffn_f16_modes(launches):
    """The FFN plan on binary16 operands (H stored in binary16) in each mode: one launch, two
    launches, H on chip."""
    import oracle
    t, d, f = 300, 256, 512
    g = torch.Generator().manual_seed(1616 + launches)

    def r(*sh, sc=1.0):
        return (torch.randn(*sh, generator=g) * sc).to(torch.float16)
    cpu = dict(X=r(t, d, sc=0.5), W1=r(d, f, sc=0.05), b1=r(f, sc=0.1), W2=r(f, d, sc=0.05),
               b2=r(d, sc=0.1), R=r(t, d))
    dev = torch.device("cuda")
    gi = {k: v.to(dev) for k, v in cpu.items()}
    Y = torch.empty((t, d), dtype=torch.float16, device=dev)
    with gemm_epi.FfnPlan(t, d, f, "f16", launches=launches) as plan:
        plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
        assert plan.sync_status() == 0
        H = plan.hidden().cpu()
    H_ref, H_exact, Y_ref = oracle.ffn(**cpu, dtype="f16")
    if launches != 3:
        assert rel_err(H, H_exact) <= TOL["f16"]
    assert rel_err(Y, Y_ref) <= TOL["f16"]


def test_ffn_onchip_rules():
    with gemm_epi.FfnPlan(300, 136, 264) as plan:          # d, f not multiples of 256
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            gemm_epi.gemm_epi_ffn_set_option(plan.handle, "LAUNCHES", 3)
        assert e.value.status == 2
        assert not plan.describe().startswith("one launch, H on chip")
    with gemm_epi.FfnPlan(256, 256, 256, layernorm=True) as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            gemm_epi.gemm_epi_ffn_set_option(plan.handle, "LAUNCHES", 3)
        assert e.value.status == 1
    with gemm_epi.FfnPlan(256, 256, 256) as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            gemm_epi.gemm_epi_ffn_set_option(plan.handle, "LAUNCHES", 4)
        assert e.value.status == 1


def _ffn_inputs(t, d, f, seed):
    g = torch.Generator().manual_seed(seed)

    def r(*s, sc=1.0):
        return (torch.randn(*s, generator=g) * sc).to(torch.bfloat16)
    return dict(X=r(t, d, sc=0.5), W1=r(d, f, sc=0.05), b1=r(f, sc=0.1), W2=r(f, d, sc=0.05),
                b2=r(d, sc=0.1), R=r(t, d))


# (t, d, f, requested K slices of GEMM 2, slices the shape gives): f = 1032 has 17 K blocks
# of H (slices of 12 or 8 blocks: 2 or 3 slices, the last one ragged); f = 776 has 13
# (4 slices of 4, the last of 1 block: GEMM-1 tile 3 holds only 8 columns of H)
FFN_SPLIT_CASES = [(300, 136, 1032, 2, 2), (300, 136, 1032, 4, 3), (520, 264, 776, 4, 4),
                   (1300, 520, 1032, 4, 3), (16, 256, 2048, 4, 4), (600, 1024, 4096, 2, 2)]


@pytest.mark.parametrize("order", [1, 2])
@pytest.mark.parametrize("t,d,f,split2,slices", FFN_SPLIT_CASES)
def test_ffn_one_launch_split2_parity(t, d, f, split2, slices, order):
    """One launch with GEMM 2 split along K: each slice a unit of its own, the partial sums
    added by the slice that finishes last, in slice order.  Against the oracle; repeated
    calls give the same bits (the counts are back at zero and the sum order is fixed)."""
    import oracle
    cpu = _ffn_inputs(t, d, f, t + 7 * d + f)
    dev = torch.device("cuda")
    gi = {k: v.to(dev) for k, v in cpu.items()}
    Y = torch.empty((t, d), dtype=torch.bfloat16, device=dev)
    with gemm_epi.FfnPlan(t, d, f, launches=1, split2=split2, tile_order=order) as plan:
        desc = plan.describe()
        assert desc.startswith("one launch")
        assert f"in {slices} K slices" in desc, desc
        assert ("order=dynamic" if order == 2 else "order=static") in desc
        outs = []
        for _ in range(3):
            plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
            assert plan.sync_status() == 0
            outs.append(Y.clone())
        H = plan.hidden().cpu()
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    H_ref, H_exact, Y_ref = oracle.ffn(**cpu)
    assert rel_err(H, H_exact) <= TOL["bf16"]
    assert rel_err(Y, Y_ref) <= TOL["bf16"]
    Y2 = oracle.gemm_epi(H, cpu["W2"], cpu["b2"], dtype="bf16", epilog="BIAS_RESIDUAL",
                         residual=cpu["R"])
    assert rel_err(Y, Y2) <= TOL["bf16"]


def test_ffn_split2_order_independent():
    """The same K slices in the static and the dynamic order give the same bits: which pair
    runs a slice, and which slice finishes last, does not change the sum."""
    t, d, f = 1300, 520, 1032
    cpu = _ffn_inputs(t, d, f, 99)
    dev = torch.device("cuda")
    gi = {k: v.to(dev) for k, v in cpu.items()}
    outs = []
    for order in (1, 2):
        Y = torch.empty((t, d), dtype=torch.bfloat16, device=dev)
        with gemm_epi.FfnPlan(t, d, f, launches=1, split2=4, tile_order=order) as plan:
            plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
            assert plan.sync_status() == 0
        outs.append(Y)
    assert torch.equal(outs[0], outs[1])


# ---- split-K: partial sums through device memory (mode 2), across a cluster (mode 1), or
# across a cluster through an L2 workspace (mode 3) ------------------------------------------

SPLIT_WHERE = {1: "(cluster)", 2: "(device memory)", 3: "(cluster+L2)"}

SPLIT_CASES = [(1, 1, 64, 2), (1, 1, 128, 3), (1, 1, 256, 4), (1, 1, 64, 4),
               (1, 2, 0, 2), (1, 2, 0, 3), (1, 2, 0, 4),
               (3, 1, 64, 2), (3, 1, 128, 3), (3, 1, 256, 4), (3, 1, 128, 4),
               (3, 2, 0, 2), (3, 2, 0, 4),
               (2, 1, 64, 2), (2, 1, 128, 3), (2, 1, 256, 4), (2, 1, 64, 8),
               (2, 2, 0, 2), (2, 2, 0, 6), (2, 2, 0, 8), (2, 2, 16, 5)]


@pytest.mark.parametrize("mode,variant,bn,split", SPLIT_CASES)
@pytest.mark.parametrize("epilog", ["BIAS", "GELU_BIAS", "RELU_AUX_BIAS", "BIAS_RESIDUAL"])
def test_split_k_parity(mode, variant, bn, split, epilog):
    m, n, k = (300 if variant == 1 else 40), 520, 1000    # 16 K blocks, the last one 40 deep
    layout = "M1" if (split + len(epilog)) % 2 else "1N"
    p = _inputs(m, n, k, "bf16", layout, seed=split * 10 + variant + 100 * mode)
    opts = {"VARIANT": variant, "SPLIT_K": split, "SPLIT_MODE": mode}
    if bn:
        opts["TILE_N"] = bn
    _, _, _, _, desc = check(p, m, n, k, "bf16", epilog, layout, options=opts)
    kpb = -(-16 // split)                       # K blocks per slice; no slice is left empty
    assert f"split_k={-(-16 // kpb)}{SPLIT_WHERE[mode]}" in desc


@pytest.mark.parametrize("mode,variant,split", [(1, 1, 4), (1, 2, 3), (2, 1, 4), (2, 2, 6),
                                                (3, 1, 4), (3, 1, 2), (3, 2, 3)])
def test_split_k_integer_bit_exact(mode, variant, split):
    m, n, k = (256 if variant == 1 else 16), 264, 512
    p = _inputs(m, n, k, "bf16", "1N", seed=31, kind="int")
    check(p, m, n, k, "bf16", "RELU_AUX_BIAS", "1N", options={"VARIANT": variant,
                                                             "SPLIT_K": split,
                                                             "SPLIT_MODE": mode}, exact=True)


def test_split_k_device_memory_repeats_and_is_deterministic():
    # The per-tile counts return to zero after every launch, so a plan can be executed again
    # (with other inputs); the slices are added in slice order, so results repeat bit for bit.
    from parity_helpers import oracle_ref
    m, n, k = 24, 776, 1544
    dev = torch.device("cuda")
    with gemm_epi.Plan(m, n, k, "bf16", "GELU_BIAS", "1N", variant=2) as plan:
        plan.set_option("SPLIT_K", 7)
        plan.set_option("SPLIT_MODE", 2)
        assert "split_k=7(device memory)" in plan.describe()
        for seed in (1, 2):
            p = _inputs(m, n, k, "bf16", "1N", seed=500 + seed)
            A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
            outs = []
            for _ in range(4):
                D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                plan.execute(A, B, bias, D)
                outs.append(D)
            assert plan.sync_status() == 0
            for D in outs[1:]:
                assert torch.equal(D, outs[0])
            want, _ = oracle_ref(p, "bf16", "GELU_BIAS", "1N")
            assert rel_err(outs[0], want) <= TOL["bf16"]


@pytest.mark.parametrize("variant,bn,m", [(1, 128, 300), (2, 0, 24)])
def test_split_k_cluster_l2_repeats_and_is_deterministic(variant, bn, m):
    # Cluster slices whose partial sums pass through the workspace: the owner adds its own
    # and the peers' sums in rank order, so repeated launches (each a programmatic dependent
    # of the one before, rewriting the workspace) give the same bits.
    from parity_helpers import oracle_ref
    n, k = 776, 1544
    dev = torch.device("cuda")
    with gemm_epi.Plan(m, n, k, "bf16", "GELU_BIAS", "1N", variant=variant) as plan:
        if bn:
            plan.set_option("TILE_N", bn)
        plan.set_option("SPLIT_K", 4)
        plan.set_option("SPLIT_MODE", 3)
        assert "split_k=4(cluster+L2)" in plan.describe()
        for seed in (1, 2):
            p = _inputs(m, n, k, "bf16", "1N", seed=700 + seed)
            A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
            outs = []
            for _ in range(4):
                D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                plan.execute(A, B, bias, D)
                outs.append(D)
            assert plan.sync_status() == 0
            for D in outs[1:]:
                assert torch.equal(D, outs[0])
            want, _ = oracle_ref(p, "bf16", "GELU_BIAS", "1N")
            assert rel_err(outs[0], want) <= TOL["bf16"]


def test_split_k_device_memory_after_timeout():
    # A launch that gives up on a wait still counts every CTA, so the next launch is right.
    from parity_helpers import oracle_ref
    m, n, k = 32, 520, 1000
    p = _inputs(m, n, k, "bf16", "1N", seed=61)
    dev = torch.device("cuda")
    A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
    D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "BIAS", "1N", variant=2) as plan:
        plan.set_option("SPLIT_K", 4)
        plan.set_option("SPLIT_MODE", 2)
        plan.set_option("WAIT_LIMIT_US", 20000)
        plan.set_option("DEBUG_STALL", 1)
        plan.execute(A, B, bias, D)
        assert plan.sync_status() == 8
        plan.set_option("DEBUG_STALL", 0)
        plan.execute(A, B, bias, D)
        assert plan.sync_status() == 0
    want, _ = oracle_ref(p, "bf16", "BIAS", "1N")
    assert rel_err(D, want) <= TOL["bf16"]


def test_split_option_rules():
    with gemm_epi.Plan(40, 520, 1000, "bf16", "BIAS", "1N", variant=2) as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("SPLIT_K", 9)
        assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("SPLIT_MODE", 4)
        assert e.value.status == 1
        for mode in (1, 3):
            plan.set_option("SPLIT_MODE", mode)
            with pytest.raises(gemm_epi.GemmEpiError) as e:
                plan.set_option("SPLIT_K", 5)        # a cluster holds at most 4 slices
            assert e.value.status == 1
        plan.set_option("SPLIT_MODE", 2)
        plan.set_option("SPLIT_K", 5)
        assert "split_k=4(device memory)" in plan.describe()   # 16 K blocks: 4 x 4


# ---- swapped kernel with tiles narrower than m (several tiles along the rows of D) --------

@pytest.mark.parametrize("m,bn", [(40, 16), (100, 32), (256, 64), (200, 16)])
@pytest.mark.parametrize("epilog", ["GELU_BIAS", "RELU_AUX_BIAS", "BIAS_RESIDUAL", "GELU_AUX_BIAS"])
def test_swapped_narrow_tiles(m, bn, epilog):
    n, k = 392, 328
    layout = "M1" if (m + len(epilog)) % 2 else "1N"
    p = _inputs(m, n, k, "bf16", layout, seed=900 + m + bn)
    _, _, _, _, desc = check(p, m, n, k, "bf16", epilog, layout,
                             options={"VARIANT": 2, "TILE_N": bn, "TILE_M": 128})
    assert f"tile=128x{bn}" in desc


@pytest.mark.parametrize("m", [1, 16, 64, 100, 256])
def test_small_m_tile_width_choice(m):
    # the swapped kernel takes the narrowest power-of-two tile (>= 16 rows) whose tiles all
    # get their own SM
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 3072
    full = 16
    while full < m:
        full *= 2
    want = full
    for bn in (16, 32, 64, 128):
        if bn < full and (n // 128) * -(-m // bn) <= sms:
            want = bn
            break
    with gemm_epi.Plan(m, n, 768, "bf16", "GELU_BIAS", "1N", variant=2) as plan:
        assert f"tile=128x{want}" in plan.describe(), plan.describe()


# ---- swapped kernel with 64 columns of D per tile (64-row MMAs) -----------------------------

M64_EPILOGS = ["BIAS", "RELU_BIAS", "GELU_BIAS", "NONE", "TANH_BIAS", "BIAS_RESIDUAL",
               "GELU_AUX_BIAS"]


@pytest.mark.parametrize("m,n,k,bn", [(1, 264, 136, 16), (16, 200, 72, 16), (40, 392, 200, 16),
                                      (100, 136, 328, 32), (256, 520, 200, 64),
                                      (20, 3072, 768, 16)])
@pytest.mark.parametrize("epilog", M64_EPILOGS)
def test_swapped_m64_parity(m, n, k, bn, epilog):
    # ragged n (the last tile's later lane quarters hold no columns), both bias layouts,
    # both dtypes
    layout = "M1" if (m + len(epilog)) % 2 else "1N"
    dtype = "f16" if (m + k) % 3 == 0 else "bf16"
    p = _inputs(m, n, k, dtype, layout, seed=1300 + m + n)
    _, _, _, _, desc = check(p, m, n, k, dtype, epilog, layout,
                             options={"VARIANT": 2, "TILE_N": bn, "TILE_M": 64})
    assert f"tile=64x{bn}" in desc, desc


@pytest.mark.parametrize("epilog", ["BIAS", "RELU_BIAS", "NONE", "BIAS_RESIDUAL"])
def test_swapped_m64_integer_bit_exact(epilog):
    m, n, k = 24, 328, 136
    p = _inputs(m, n, k, "bf16", "1N", seed=1400, kind="int")
    check(p, m, n, k, "bf16", epilog, "1N", options={"VARIANT": 2, "TILE_M": 64}, exact=True)


def test_swapped_m64_only_on_request():
    with gemm_epi.Plan(16, 3072, 768, "bf16", "GELU_BIAS", "1N", variant=2) as plan:
        assert "variant=swapped tile=128x16" in plan.describe(), plan.describe()
        plan.set_option("TILE_M", 64)
        assert "variant=swapped tile=64x16" in plan.describe(), plan.describe()
        plan.set_option("TILE_M", 0)
        assert "variant=swapped tile=128x16" in plan.describe(), plan.describe()


def test_swapped_m64_option_rules():
    with gemm_epi.Plan(16, 264, 136, "bf16", "RELU_AUX_BIAS", "1N", variant=2) as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("TILE_M", 64)
        assert e.value.status == 1
        assert "tile=128x" in plan.describe()          # previous configuration kept
    with gemm_epi.Plan(16, 264, 136, "bf16", "GELU_BIAS", "1N", variant=2) as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("TILE_M", 32)
        assert e.value.status == 1
        plan.set_option("SPLIT_K", 2)                  # a K split keeps 128-column tiles
        assert "tile=128x" in plan.describe() and "split_k=2" in plan.describe()
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("TILE_M", 64)
        assert e.value.status == 1


def test_row_tiles_over_long_k_split_in_a_cluster():
    # 64 row tiles of 128 x 64 on 152 SMs over 32 K blocks: the model's choice, 32 tiles of
    # 128 x 128 in 4 K slices through a cluster, the partial sums through L2
    with gemm_epi.Plan(1024, 512, 2048, "f16", "BIAS", "M1") as plan:
        d = plan.describe()
        assert "variant=row-tile" in d and "tile=128x128" in d and "split_k=4(cluster+L2)" in d, d
        plan.set_option("SPLIT_MODE", 1)               # the same slices over DSMEM
        assert "tile=128x128" in plan.describe() and "split_k=4(cluster) " in plan.describe()
        plan.set_option("SPLIT_MODE", 0)
        plan.set_option("TILE_N", 64)                  # a fixed width: the slices for it
        assert "tile=128x64" in plan.describe() and "split_k=2(cluster+L2)" in plan.describe()
    with gemm_epi.Plan(1024, 512, 512, "f16", "BIAS", "M1") as plan:   # 8 K blocks: no split
        assert "split_k=1 " in plan.describe()
    p = _inputs(1024, 512, 2048, "f16", "M1", seed=1001)
    check(p, 1024, 512, 2048, "f16", "BIAS", "M1")
    check(p, 1024, 512, 2048, "f16", "BIAS", "M1", options={"SPLIT_MODE": 1})


@pytest.mark.parametrize("m,n,k,variant", [(256, 1024, 8192, "row-tile"), (64, 3072, 8192, "row-tile"),
                                           (256, 3072, 768, "swapped"), (100, 3072, 768, "swapped"),
                                           (200, 512, 256, "swapped"), (256, 3072, 1536, "swapped"),
                                           (256, 4096, 4096, "row-tile")])
def test_small_m_long_k_plan_choice(m, n, k, variant):
    # m <= 256 beyond the small-m kernel: the swapped kernel, unless K is long enough that
    # row tiles with K split over a cluster are well ahead in the model
    p = _inputs(m, n, k, "bf16", "1N", seed=3100 + m)
    _, _, _, _, desc = check(p, m, n, k, "bf16", "BIAS", "1N")
    assert f"variant={variant}" in desc, desc
    if variant == "row-tile":
        assert "(cluster+L2)" in desc, desc


def test_auto_split_clusters_all_resident():
    # 48 tiles of 128 x 128 in clusters of 3 do not all fit on the GPU at once (a GPC's SMs
    # are not a multiple of 3), so the automatic choice never takes them
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for m, n, k in [(256, 3072, 1536), (256, 3072, 768), (384, 2048, 3072)]:
        with gemm_epi.Plan(m, n, k, "bf16", "GELU_BIAS", "1N") as plan:
            fields = dict(kv.split("=", 1) for kv in plan.describe().split() if "=" in kv)
        split = int(fields["split_k"].split("(")[0])
        if split > 1:
            assert int(fields["grid"]) <= sms and split != 3, fields


@pytest.mark.parametrize("m,epilog,variant", [
    (16, "GELU_BIAS", "small-m"), (64, "GELU_BIAS", "small-m"), (1, "RELU_AUX_BIAS", "small-m"),
    (256, "GELU_BIAS", "swapped"), (16, "DRELU_BGRAD", "swapped"), (100, "BIAS", "swapped")])
def test_small_m_plan_choice(m, epilog, variant):
    # m <= 64 with a forward epilog: the small-m kernel, K split over a cluster so that its
    # 24 column tiles x the slices occupy most SMs, every cluster resident at once; larger m
    # and the backward epilogs: the swapped kernel, unsplit (a split through the swapped
    # kernel's ring measured slower)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with gemm_epi.Plan(m, 3072, 768, "bf16", epilog, "1N") as plan:
        desc = plan.describe()
    fields = dict(kv.split("=") for kv in desc.split() if "=" in kv)
    assert fields["variant"] == variant, desc
    if variant == "swapped":
        assert fields["split_k"] == "1", desc
    else:
        split = int(fields["split_k"].split("(")[0])
        assert split >= 2 and fields["split_k"].endswith("(cluster)"), desc
        assert int(fields["grid"]) == 24 * split <= sms, desc


@pytest.mark.parametrize("variant", [1, 2])
def test_l2_prefetch_option_keeps_results(variant):
    m, n, k = (384 if variant == 1 else 64), 520, 1000
    p = _inputs(m, n, k, "bf16", "1N", seed=41)
    check(p, m, n, k, "bf16", "RELU_AUX_BIAS", "1N",
          options={"VARIANT": variant, "PREFETCH": 4, "SPLIT_K": 1})


@pytest.mark.parametrize("variant", [1, 2])
def test_programmatic_launch_sees_preceding_writes(variant):
    # The fused kernel starts as a programmatic dependent of the stream's previous work;
    # its reads must still see what that work wrote.  Torch kernels rewrite A and the bias
    # just before the call, and a second call consumes the first call's output.
    m, n, k = (256 if variant == 1 else 48), 264, 264
    p = _inputs(m, n, k, "bf16", "1N", seed=51)
    q = _inputs(m, n, k, "bf16", "1N", seed=52)
    dev = torch.device("cuda")
    A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
    B2 = q["B"][:n, :].contiguous().to(dev) if n <= k else None
    D1 = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    D2 = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    opts = {"VARIANT": variant}
    with gemm_epi.Plan(m, n, k, "bf16", "BIAS", "1N", **opts) as p1, \
            gemm_epi.Plan(m, n, n, "bf16", "GELU_BIAS", "1N", **opts) as p2:
        for _ in range(3):
            A.copy_(q["A"].to(dev))          # torch writes A ...
            bias.copy_(q["bias"].to(dev))    # ... and the bias right before the call
            p1.execute(A, B, bias, D1)
            p2.execute(D1, B2, bias, D2)     # reads the previous call's output
        assert p1.sync_status() == 0 and p2.sync_status() == 0
    cur = {"A": q["A"], "B": p["B"], "bias": q["bias"]}
    from parity_helpers import oracle_ref
    want1, _ = oracle_ref(cur, "bf16", "BIAS", "1N")
    assert rel_err(D1, want1) <= TOL["bf16"]
    want2, _ = oracle_ref({"A": D1.cpu(), "B": B2.cpu(), "bias": q["bias"]}, "bf16", "GELU_BIAS",
                          "1N")
    assert rel_err(D2, want2) <= TOL["bf16"]


# ---- the CTA-pair row-tile kernel (cta_group::2, 256 x 256 tiles) -----------------------------

@pytest.mark.parametrize("bn", [256, 224])
@pytest.mark.parametrize("epilog", EPILOGS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_pair_parity(bn, epilog, dtype):
    m, n, k = 600, 520, 200            # 3 ragged 256-row tiles, 3 ragged column tiles
    layout = "M1" if (EPILOGS.index(epilog) + bn // 32) % 2 else "1N"
    p = _inputs(m, n, k, dtype, layout, seed=61 + EPILOGS.index(epilog) + bn)
    _, _, _, _, desc = check(p, m, n, k, dtype, epilog, layout,
                             options={"VARIANT": 3, "TILE_N": bn})
    assert "variant=row-pair" in desc and f"tile=256x{bn} " in desc


@pytest.mark.parametrize("bn", [256, 224])
@pytest.mark.parametrize("epilog", ["GELU_BIAS", "TANH_BIAS"])
@pytest.mark.parametrize("k,grid", [(200, 0), (264, 6), (520, 0), (600, 4)])
def test_pair_epilogue_warp_variants(bn, epilog, k, grid):
    # GELU_BIAS and TANH_BIAS run 16 epilogue warps (bias shuffled between lanes) when K <= 512
    # and 8 otherwise; both, with a few pairs walking many tiles, and both bias layouts
    m, n = 1280, 1000
    layout = "M1" if (k + bn) % 3 == 0 else "1N"
    p = _inputs(m, n, k, "bf16", layout, seed=k + bn + len(epilog))
    opts = {"VARIANT": 3, "TILE_N": bn}
    if grid:
        opts["GRID"] = grid
    check(p, m, n, k, "bf16", epilog, layout, options=opts)


# ---- the CTA-pair kernel's tile order: static, or handed out by the plan's device counter ----

ORDERS = {"static": 1, "dynamic": 2}


@pytest.mark.parametrize("order", ["static", "dynamic"])
@pytest.mark.parametrize("bn", [256, 224])
@pytest.mark.parametrize("epilog", EPILOGS)
def test_pair_order_parity(order, bn, epilog):
    m, n, k = 1000, 520, 200           # 4 ragged 256-row tiles, ragged N and K
    layout = "M1" if (EPILOGS.index(epilog) + bn // 32) % 2 else "1N"
    p = _inputs(m, n, k, "bf16", layout, seed=161 + EPILOGS.index(epilog) + bn)
    _, _, _, _, desc = check(p, m, n, k, "bf16", epilog, layout,
                             options={"VARIANT": 3, "TILE_N": bn, "TILE_ORDER": ORDERS[order]})
    assert "variant=row-pair" in desc and f"tile=256x{bn} " in desc and f"order={order}" in desc


@pytest.mark.parametrize("grid,group_m", [(2, 1), (4, 2), (8, 3), (12, 8)])
def test_pair_dynamic_walk(grid, group_m):
    # 9 x 5 tiles, 9 K blocks, few pairs: most tiles come from the counter
    m, n, k = 2304, 1000, 520
    p = _inputs(m, n, k, "bf16", "1N", seed=grid + 170)
    check(p, m, n, k, "bf16", "GELU_BIAS", "1N",
          options={"VARIANT": 3, "GRID": grid, "GROUP_M": group_m, "TILE_ORDER": 2})


def test_pair_dynamic_counter_back_at_zero_between_launches():
    # every launch must find the counter at zero: repeated launches of one plan (each on new
    # inputs) and of two plans in turn, all exact on integer inputs
    from parity_helpers import oracle_ref
    dev = torch.device("cuda")
    shapes = [(1536, 776, 136), (768, 1288, 72)]
    plans = [gemm_epi.Plan(m, n, k, "bf16", "RELU_AUX_BIAS", "1N", variant=3, grid=10,
                           tile_order=2) for m, n, k in shapes]
    try:
        for rep in range(4):
            for i, ((m, n, k), plan) in enumerate(zip(shapes, plans)):
                assert "order=dynamic" in plan.describe()
                p = _inputs(m, n, k, "bf16", "1N", seed=500 + 10 * rep + i, kind="int")
                A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
                D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                aux = torch.empty((m, (n + 31) // 32), dtype=torch.int32, device=dev)
                plan.execute(A, B, bias, D, aux=aux)
                assert plan.sync_status() == 0
                want, _ = oracle_ref(p, "bf16", "RELU_AUX_BIAS", "1N")
                assert np.array_equal(D.float().cpu().double().numpy(), want), (rep, i)
    finally:
        for plan in plans:
            plan.free()


def test_pair_dynamic_integer_bit_exact():
    m, n, k = 1024, 264, 64
    p = _inputs(m, n, k, "bf16", "1N", seed=172, kind="int")
    check(p, m, n, k, "bf16", "RELU_AUX_BIAS", "1N", options={"VARIANT": 3, "TILE_ORDER": 2},
          exact=True)


@pytest.mark.parametrize("m,n,order", [(65536, 16384, "dynamic"), (8192, 16384, "dynamic"),
                                       (4096, 4096, "static"), (4096, 1024, "static")])
def test_pair_order_automatic_choice(m, n, order):
    # CTA-pair plans hand out their tiles from the counter from eight waves of tiles over
    # the pairs up, and in the static order below that; the option overrides either way
    with gemm_epi.Plan(m, n, 4096, "bf16", "RELU_BIAS", "1N") as plan:
        d = plan.describe()
        assert "variant=row-pair " in d and f"order={order}" in d, d
        plan.set_option("TILE_ORDER", 1)
        assert "order=static" in plan.describe()
        plan.set_option("TILE_ORDER", 2)
        assert "order=dynamic" in plan.describe()


def test_pair_option_rules():
    with gemm_epi.Plan(1024, 1024, 1024, "e4m3", "RELU_BIAS", "1N") as plan:
        for v in (1, 2, 4):
            with pytest.raises(gemm_epi.GemmEpiError) as e:
                plan.set_option("VARIANT", v)   # E4M3 plans run the CTA-pair kernel only
            assert e.value.status == 1
        assert "variant=row-pair " in plan.describe()
    with gemm_epi.Plan(1024, 1024, 1024, "bf16", "RELU_BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("VARIANT", 4)       # no such kernel
        assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.set_option("TILE_ORDER", 3)
        assert e.value.status == 1
        plan.set_option("VARIANT", 3)
        d = plan.describe()
        grid = int(d.split(" grid=")[1].split()[0])
        assert grid % 2 == 0 and "order=static" in d      # 16 tiles: one wave


@pytest.mark.parametrize("m,n,want", [(4096, 4096, 224), (8192, 16384, 256), (65536, 16384, 256),
                                      (4096, 1024, 256)])
def test_pair_tile_width_choice(m, n, want):
    """The planner trades tile width against wave quantization over the resident pairs."""
    with gemm_epi.Plan(m, n, 1024, "bf16", "RELU_BIAS", "1N", variant=3) as plan:
        desc = plan.describe()
    assert "variant=row-pair" in desc and f"tile=256x{want} " in desc, desc


def test_pair_narrow_tile_persistent_walk():
    m, n, k = 1280, 1000, 264          # 5 x 5 tiles of 256 x 224, 5 K blocks, 3 pairs walking
    p = _inputs(m, n, k, "bf16", "1N", seed=88)
    check(p, m, n, k, "bf16", "RELU_AUX_BIAS", "1N",
          options={"VARIANT": 3, "TILE_N": 224, "GRID": 6, "GROUP_M": 2})


@pytest.mark.parametrize("grid,group_m", [(2, 1), (4, 2), (6, 8)])
def test_pair_persistent_walk(grid, group_m):
    m, n, k = 1280, 768, 520           # 5 x 3 pair tiles, 9 K blocks, few pairs walking them
    p = _inputs(m, n, k, "bf16", "1N", seed=grid + 70)
    check(p, m, n, k, "bf16", "RELU_AUX_BIAS", "1N",
          options={"VARIANT": 3, "GRID": grid, "GROUP_M": group_m})


def test_pair_integer_bit_exact():
    m, n, k = 512, 264, 64
    p = _inputs(m, n, k, "bf16", "1N", seed=72, kind="int")
    check(p, m, n, k, "bf16", "RELU_AUX_BIAS", "1N", options={"VARIANT": 3}, exact=True)


@pytest.mark.parametrize("order", [1, 2])
def test_pair_timeout_path(order):
    # after a launch that ran out its wait limit, the next launch is correct (with the
    # dynamic order: the aborted launch left the tile counter at zero)
    m, n, k = 1024, 768, 128
    p = _inputs(m, n, k, "bf16", "1N", seed=73)
    dev = torch.device("cuda")
    A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
    D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "BIAS", "1N", variant=3, tile_order=order,
                       grid=4) as plan:
        plan.set_option("WAIT_LIMIT_US", 20000)
        plan.set_option("DEBUG_STALL", 1)
        plan.execute(A, B, bias, D)
        assert plan.sync_status() == 8
        plan.set_option("DEBUG_STALL", 0)
        plan.execute(A, B, bias, D)
        assert plan.sync_status() == 0
    from parity_helpers import oracle_ref
    want, _ = oracle_ref(p, "bf16", "BIAS", "1N")
    assert rel_err(D, want) <= TOL["bf16"]


def test_plans_run_concurrently_on_separate_streams():
    # each plan owns its status word, tile counter, workspace and tensor maps: different
    # plans may run at the same time on different streams (a CTA-pair plan with the dynamic
    # tile order, a small-m plan with a device-memory split and a row-tile plan split
    # through a cluster)
    from parity_helpers import oracle_ref
    dev = torch.device("cuda")
    cases = [(4096, 4096, 256, "RELU_AUX_BIAS", {}),
             (24, 776, 1544, "GELU_BIAS", {"SPLIT_K": 4}),
             (1024, 512, 2048, "BIAS", {})]
    plans, outs, ins = [], [], []
    streams = [torch.cuda.Stream() for _ in cases]
    try:
        for i, (m, n, k, epi, opts) in enumerate(cases):
            p = _inputs(m, n, k, "bf16", "1N", seed=300 + i)
            A, B, bias = p["A"].to(dev), p["B"].to(dev), p["bias"].to(dev)
            D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            aux = torch.empty((m, (n + 31) // 32), dtype=torch.int32, device=dev) \
                if epi == "RELU_AUX_BIAS" else None
            plan = gemm_epi.Plan(m, n, k, "bf16", epi, "1N", **opts)
            plans.append(plan)
            ins.append((p, epi))
            outs.append((A, B, bias, D, aux))
        torch.cuda.synchronize()
        for rep in range(3):
            for plan, s, (A, B, bias, D, aux) in zip(plans, streams, outs):
                with torch.cuda.stream(s):
                    plan.execute(A, B, bias, D, aux=aux)
        torch.cuda.synchronize()
        for plan, (p, epi), (A, B, bias, D, aux) in zip(plans, ins, outs):
            assert plan.sync_status() == 0
            want, _ = oracle_ref(p, "bf16", epi, "1N")
            assert rel_err(D.cpu(), want) <= TOL["bf16"], plan.describe()
    finally:
        for plan in plans:
            plan.free()
