"""GPU parity of the LayerNorm row ("Operator fusion in model inference", section 2): the fused
LayerNorm (+ residual) kernel, the per-row statistics, the weight fold, the GEMM with the
LayerNorm folded into its epilogue (LN_GELU_BIAS) on every kernel variant, and the
pre-LayerNorm FFN block, against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi
from parity_helpers import TD, TOL, UNIT_ROUNDOFF, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _ln_inputs(t, d, seed, dtype="bf16", offset=1.5, scale=3.0):
    g = torch.Generator().manual_seed(seed)
    X = (torch.randn(t, d, generator=g) * scale + offset).to(TD[dtype])
    gamma = (1.0 + 0.1 * torch.randn(d, generator=g)).to(TD[dtype])
    beta = (0.1 * torch.randn(d, generator=g)).to(TD[dtype])
    R = torch.randn(t, d, generator=g).to(TD[dtype])
    return X, gamma, beta, R


def _weights(d, f, seed, dtype="bf16", sigma=None):
    g = torch.Generator().manual_seed(seed)
    s = sigma if sigma is not None else 1.0 / np.sqrt(d)
    W = (torch.randn(d, f, generator=g) * s).to(TD[dtype])
    b = (torch.randn(f, generator=g) * 0.1).to(TD[dtype])
    return W, b


# ---- the fused LayerNorm (+ residual) kernel ------------------------------------------------

@pytest.mark.parametrize("t,d,dtype,eps,res", [(1, 8, "bf16", 1e-5, False), (37, 72, "f16", 1e-5, True),
                                               (300, 1024, "bf16", 1e-6, True),
                                               (129, 4096, "bf16", 1e-5, False),
                                               (64, 768, "f16", 0.0, True)])
def test_layernorm_kernel_parity(t, d, dtype, eps, res):
    X, gamma, beta, R = _ln_inputs(t, d, seed=t + d, dtype=dtype)
    dev = torch.device("cuda")
    Xg, gg, bg, Rg = (v.to(dev) for v in (X, gamma, beta, R))
    Y = torch.full((t, d), float("nan"), dtype=TD[dtype], device=dev)
    gemm_epi.gemm_epi_layernorm(t, d, dtype, Xg, Rg if res else None, gg, bg, eps, Y)
    torch.cuda.synchronize()
    want, _ = oracle.layernorm(X, gamma, beta, eps=eps, dtype=dtype, residual=R if res else None)
    assert rel_err(Y, want) <= TOL[dtype]


def test_layernorm_in_place():
    t, d = 50, 256
    X, gamma, beta, R = _ln_inputs(t, d, seed=2)
    dev = torch.device("cuda")
    Xg, gg, bg, Rg = (v.to(dev) for v in (X, gamma, beta, R))
    gemm_epi.gemm_epi_layernorm(t, d, "bf16", Xg, Rg, gg, bg, 1e-5, Rg)   # Y = residual
    torch.cuda.synchronize()
    want, _ = oracle.layernorm(X, gamma, beta, eps=1e-5, dtype="bf16", residual=R)
    assert rel_err(Rg, want) <= TOL["bf16"]


@pytest.mark.parametrize("t,d", [(1, 8), (300, 1024), (77, 4096)])
def test_layernorm_stats(t, d):
    X, _, _, _ = _ln_inputs(t, d, seed=d)
    stats = torch.empty((t, 2), dtype=torch.float32, device="cuda")
    gemm_epi.gemm_epi_layernorm_stats(t, d, "bf16", X.cuda(), 1e-5, stats)
    torch.cuda.synchronize()
    _, want = oracle.layernorm(X, torch.ones(d, dtype=torch.bfloat16),
                               torch.zeros(d, dtype=torch.bfloat16), eps=1e-5, dtype="bf16")
    got = stats.cpu().double().numpy()
    # fp32 sums of d values (relative error well below 1e-5 at these sizes) and rsqrt (~2 ulp)
    sd = 1.0 / want[:, 1]
    assert np.all(np.abs(got[:, 0] - want[:, 0]) <= 1e-5 * (np.abs(want[:, 0]) + sd))
    np.testing.assert_allclose(got[:, 1], want[:, 1], rtol=2e-5)


def test_layernorm_fold():
    d, f = 264, 520
    _, gamma, beta, _ = _ln_inputs(1, d, seed=4)
    W, b = _weights(d, f, seed=5)
    dev = torch.device("cuda")
    Wf = torch.empty((d, f), dtype=torch.bfloat16, device=dev)
    cs = torch.empty(f, dtype=torch.float32, device=dev)
    bf = torch.empty(f, dtype=torch.float32, device=dev)
    gemm_epi.gemm_epi_layernorm_fold(d, f, "bf16", gamma.cuda(), beta.cuda(), W.cuda(), b.cuda(),
                                     Wf, cs, bf)
    torch.cuda.synchronize()
    g64 = gamma.double().numpy()[:, None]
    want_wf = torch.from_numpy((g64 * W.double().numpy()).astype(np.float32)).to(torch.bfloat16)
    # gamma_k W_kj formed in fp32 and rounded once to bf16
    assert torch.equal(Wf.cpu(), want_wf)
    np.testing.assert_allclose(cs.cpu().double().numpy(), want_wf.double().numpy().sum(0),
                               rtol=1e-5, atol=1e-5)
    want_b = beta.double().numpy() @ W.double().numpy() + b.double().numpy()
    np.testing.assert_allclose(bf.cpu().double().numpy(), want_b, rtol=1e-5, atol=1e-5)


def test_layernorm_argument_errors():
    dev = torch.device("cuda")
    X = torch.zeros((4, 16), dtype=torch.bfloat16, device=dev)
    g = torch.ones(16, dtype=torch.bfloat16, device=dev)
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.gemm_epi_layernorm(4, 12, "bf16", X, None, g, g, 1e-5, X)
    assert e.value.status == 2
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.gemm_epi_layernorm(4, 16, "bf16", X, None, g, g, -1.0, X)
    assert e.value.status == 1
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.gemm_epi_layernorm(4, 8, "bf16", X.data_ptr() + 2, None, g, g, 1e-5, X)
    assert e.value.status == 3
    gemm_epi.gemm_epi_layernorm(0, 16, "bf16", None, None, None, None, 1e-5, None)  # empty


# ---- the GEMM with LayerNorm folded into its epilogue --------------------------------------

def _ln_gemm_gpu(X, gamma, beta, W, b, eps, dtype, options=None, unfused=False):
    m, k = X.shape
    n = W.shape[1]
    dev = torch.device("cuda")
    Xg = X.to(dev)
    Wf = torch.empty((k, n), dtype=TD[dtype], device=dev)
    cs = torch.empty(n, dtype=torch.float32, device=dev)
    bf = torch.empty(n, dtype=torch.float32, device=dev)
    stats = torch.empty((m, 2), dtype=torch.float32, device=dev)
    gemm_epi.gemm_epi_layernorm_fold(k, n, dtype, gamma.to(dev), beta.to(dev), W.to(dev),
                                     b.to(dev), Wf, cs, bf)
    gemm_epi.gemm_epi_layernorm_stats(m, k, dtype, Xg, eps, stats)
    D = torch.full((m, n), float("nan"), dtype=TD[dtype], device=dev)
    with gemm_epi.Plan(m, n, k, dtype, "LN_GELU_BIAS", "1N", **(options or {})) as plan:
        if unfused:
            pre = torch.empty((m, n), dtype=TD[dtype], device=dev)
            plan.execute_unfused(Xg, Wf, None, pre, D, ln=(stats, cs, bf))
        else:
            plan.execute(Xg, Wf, None, D, ln=(stats, cs, bf))
        assert plan.sync_status() == 0
        desc = plan.describe()
    return D.cpu(), desc


VARIANTS = [
    ("rowtile64", 300, 264, 136, {"VARIANT": 1, "TILE_N": 64}),
    ("rowtile128", 40, 520, 200, {"VARIANT": 1, "TILE_N": 128}),
    ("rowtile256", 300, 520, 1024, {"VARIANT": 1, "TILE_N": 256}),
    ("pair256", 600, 520, 200, {"VARIANT": 3, "TILE_N": 256}),
    ("pair224", 520, 600, 136, {"VARIANT": 3, "TILE_N": 224}),
    ("pair_static", 1000, 600, 136, {"VARIANT": 3, "TILE_ORDER": 1}),
    ("pair_dynamic_walk", 1000, 600, 136, {"VARIANT": 3, "TILE_ORDER": 2, "GRID": 4}),
    ("split3", 260, 264, 520, {"VARIANT": 1, "TILE_N": 128, "SPLIT_K": 3}),
    ("split3_cluster", 260, 264, 520, {"VARIANT": 1, "TILE_N": 128, "SPLIT_K": 3, "SPLIT_MODE": 1}),
    ("split4_cluster_l2", 260, 264, 520, {"VARIANT": 1, "TILE_N": 128, "SPLIT_K": 4, "SPLIT_MODE": 3}),
    ("auto_split", 1024, 512, 2048, None),
    ("small_m_default", 16, 3072, 768, None),
    ("default", 1000, 776, 328, None),
]


@pytest.mark.parametrize("name,m,n,k,opts", VARIANTS, ids=[v[0] for v in VARIANTS])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_ln_gemm_gelu_parity(name, m, n, k, opts, dtype):
    X, gamma, beta, _ = _ln_inputs(m, k, seed=m + n + k, dtype=dtype)
    W, b = _weights(k, n, seed=k, dtype=dtype)
    D, desc = _ln_gemm_gpu(X, gamma, beta, W, b, 1e-5, dtype, options=opts)
    want = oracle.ln_gemm_gelu(X, gamma, beta, W, b, eps=1e-5, dtype=dtype)
    assert rel_err(D, want) <= TOL[dtype], desc
    if name == "small_m_default":
        assert "variant=row-tile" in desc  # no LayerNorm epilogue on the swapped kernel


def test_ln_gemm_gelu_unfused():
    m, n, k = 300, 264, 136
    X, gamma, beta, _ = _ln_inputs(m, k, seed=11)
    W, b = _weights(k, n, seed=12)
    D, desc = _ln_gemm_gpu(X, gamma, beta, W, b, 1e-5, "bf16", unfused=True)
    want = oracle.ln_gemm_gelu(X, gamma, beta, W, b, eps=1e-5, dtype="bf16")
    # the unfused baseline rounds X . W' (which still holds mu c) to bf16 before correcting
    xabs = np.abs(X.double().numpy()) @ np.abs(gamma.double().numpy()[:, None] * W.double().numpy())
    _, stats = oracle.layernorm(X, gamma, beta, eps=1e-5, dtype="bf16")
    slack = 2 * UNIT_ROUNDOFF["bf16"] * stats[:, 1:2] * xabs
    got = D.double().numpy()
    assert np.all(np.abs(got - want) <= TOL["bf16"] * (np.abs(want) + 1) + slack), desc


def test_ln_plan_rules():
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.Plan(16, 64, 64, "bf16", "LN_GELU_BIAS", "1N", VARIANT=2)
    assert e.value.status == 1
    with pytest.raises(gemm_epi.GemmEpiError) as e:
        gemm_epi.Plan(16, 64, 0, "bf16", "LN_GELU_BIAS", "1N")
    assert e.value.status == 2
    dev = torch.device("cuda")
    A = torch.zeros((16, 64), dtype=torch.bfloat16, device=dev)
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device=dev)
    D = torch.empty((16, 64), dtype=torch.bfloat16, device=dev)
    st = torch.zeros((16, 2), dtype=torch.float32, device=dev)
    cs = torch.zeros(64, dtype=torch.float32, device=dev)
    bias = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(16, 64, 64, "bf16", "LN_GELU_BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:          # LN operands missing
            plan.execute(A, B, None, D)
        assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:          # a 16-bit bias is not used
            plan.execute(A, B, bias, D, ln=(st, cs, cs))
        assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:
            plan.execute(A, B, None, D, ln=(st.data_ptr() + 4, cs, cs))
        assert e.value.status == 3


# ---- the pre-LayerNorm FFN block -----------------------------------------------------------

@pytest.mark.parametrize("t,d,f", [(300, 136, 264), (16, 256, 520), (4096, 1024, 4096)])
def test_ffn_layernorm_parity(t, d, f):
    X, gamma, beta, _ = _ln_inputs(t, d, seed=t + f, offset=0.5, scale=1.0)
    W1, b1 = _weights(d, f, seed=d, sigma=0.02)
    W2, b2 = _weights(f, d, seed=f, sigma=0.02)
    dev = torch.device("cuda")
    Xg, W2g, b2g = X.to(dev), W2.to(dev), b2.to(dev)
    W1f = torch.empty((d, f), dtype=torch.bfloat16, device=dev)
    cs = torch.empty(f, dtype=torch.float32, device=dev)
    b1f = torch.empty(f, dtype=torch.float32, device=dev)
    gemm_epi.gemm_epi_layernorm_fold(d, f, "bf16", gamma.to(dev), beta.to(dev), W1.to(dev),
                                     b1.to(dev), W1f, cs, b1f)
    Y = torch.empty((t, d), dtype=torch.bfloat16, device=dev)
    with gemm_epi.FfnPlan(t, d, f, "bf16", layernorm=True) as plan:
        assert "row statistics" in plan.describe()
        plan.execute_layernorm(Xg, 1e-5, W1f, cs, b1f, W2g, b2g, Xg, Y)   # residual = X
        assert plan.sync_status() == 0
        H = plan.hidden().cpu()
        with pytest.raises(gemm_epi.GemmEpiError):       # a LayerNorm plan needs the LN inputs
            plan.execute(Xg, W1f, b1.to(dev), W2g, b2g, Xg, Y)
    H_bits, H_exact, Y_ref = oracle.ln_ffn(X, gamma, beta, W1, b1, W2, b2, X, eps=1e-5)
    assert rel_err(H, H_exact) <= TOL["bf16"]
    assert rel_err(Y, Y_ref) <= TOL["bf16"]
