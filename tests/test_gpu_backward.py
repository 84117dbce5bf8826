"""GPU parity of the backward epilogues (DRELU_BGRAD, DGELU_BGRAD): D = (A.B) times the ReLU
mask bit or GELU'(stored pre), and the bias gradient, against the CPU oracle; plus the
forward/backward chains RELU_AUX_BIAS -> DRELU_BGRAD and GELU_AUX_BIAS -> DGELU_BGRAD."""
import numpy as np
import pytest
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi, workloads
from parity_helpers import TD, TOL, UNIT_ROUNDOFF, rel_err

pytestmark = pytest.mark.gpu

KINDS = ["DRELU_BGRAD", "DGELU_BGRAD"]

# Bias gradient bound: |got - want| <= DBIAS_TOL * (sum of |terms| + 1).  The terms are fp32
# products of a tensor-core fp32 accumulation (relative error ~1e-6 here) and a factor that is
# exact (the mask bit) or GELU' to ~1e-6; the kernel sums at most a few thousand of them in
# fp32 (32-term butterflies, then atomics: error < terms/32 * 2^-24 relative to the sum of
# |terms|, below 1e-5 at every size tested).  Dropping one row or column of 300 moves the
# sum by ~1/300 of it.
DBIAS_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _bwd_inputs(m, n, k, dtype, seed):
    return workloads.random_backward_problem(m, n, k, dtype=dtype, seed=seed)


def _run_bwd(inp, m, n, k, dtype, kind, layout, unfused=False, options=None):
    dev = torch.device("cuda")
    A, B = inp["A"].to(dev), inp["B"].to(dev)
    if kind == "DRELU_BGRAD":
        aux_in = torch.from_numpy(inp["mask"].view(np.int32).copy()).to(dev)
    else:
        aux_in = inp["pre"].to(dev)
    D = torch.full((m, n), float("nan"), dtype=TD[dtype], device=dev)
    dbias = torch.full((m if layout == "M1" else n,), float("nan"), dtype=torch.float32,
                       device=dev)
    with gemm_epi.Plan(m, n, k, dtype, kind, layout, **(options or {})) as plan:
        if unfused:
            pre = torch.empty((m, n), dtype=TD[dtype], device=dev)
            plan.execute_unfused(A, B, None, pre, D, aux_in=aux_in, dbias=dbias)
        else:
            plan.execute(A, B, None, D, aux_in=aux_in, dbias=dbias)
        status = plan.sync_status()
        desc = plan.describe()
    assert status == 0, f"device status {gemm_epi.status_string(status)} ({desc})"
    return D.cpu(), dbias.cpu().double().numpy(), desc


def _oracle_bwd(inp, dtype, kind, layout):
    return oracle.gemm_bwd(inp["A"], inp["B"], dtype=dtype, kind=kind, bias_layout=layout,
                           mask=inp["mask"] if kind == "DRELU_BGRAD" else None,
                           pre=inp["pre"] if kind == "DGELU_BGRAD" else None)


def _check_bwd(inp, m, n, k, dtype, kind, layout, unfused=False, options=None):
    D, dbias, desc = _run_bwd(inp, m, n, k, dtype, kind, layout, unfused, options)
    want, want_db = _oracle_bwd(inp, dtype, kind, layout)
    slack = 0.0
    if unfused:
        # The unfused baseline multiplies bf16/f16(A.B): one more rounding of A.B per term,
        # scaled by the factor (the mask bit, or GELU' <= 1.13).
        pre0 = oracle.gemm_epi(inp["A"], inp["B"], None, dtype=dtype, epilog="NONE")
        slack = 1.2 * UNIT_ROUNDOFF[dtype] * np.abs(pre0)
    got = D.float().double().numpy()
    bad = np.abs(got - want) > TOL[dtype] * (np.abs(want) + 1.0) + slack
    assert not bad.any(), f"{int(bad.sum())} D values off, rel err {rel_err(D, want):.3e} ({desc})"
    axis = 1 if layout == "M1" else 0
    bound = DBIAS_TOL * (np.abs(want).sum(axis=axis) + 1.0)
    if unfused and m and n:
        bound = bound + slack.sum(axis=axis)
    assert dbias.shape == want_db.shape
    err = np.abs(dbias - want_db)
    assert np.all(err <= bound), f"dbias err {np.max(err / bound):.3f} x bound ({desc})"
    return D, dbias, want, want_db, desc


# ---- every kernel variant, both kinds, both dtypes, both layouts ---------------------------

VARIANTS = [
    ("rowtile64", 300, 264, 136, {"VARIANT": 1, "TILE_N": 64}),
    ("rowtile128", 300, 264, 200, {"VARIANT": 1, "TILE_N": 128}),
    ("rowtile256", 300, 520, 136, {"VARIANT": 1, "TILE_N": 256}),
    ("pair", 600, 520, 200, {"VARIANT": 3}),
    ("pair224", 600, 520, 200, {"VARIANT": 3, "TILE_N": 224}),
    ("pair224_ragged", 520, 600, 136, {"VARIANT": 3, "TILE_N": 224}),
    ("swapped1", 1, 264, 136, {"VARIANT": 2}),
    ("swapped16", 16, 264, 136, {"VARIANT": 2}),
    ("swapped40", 40, 392, 200, {"VARIANT": 2}),
    ("swapped256", 256, 264, 136, {"VARIANT": 2}),
    ("split3_rowtile", 260, 264, 520, {"VARIANT": 1, "TILE_N": 128, "SPLIT_K": 3}),
    ("split2_swapped", 24, 264, 264, {"VARIANT": 2, "SPLIT_K": 2}),
    ("split3_rowtile_cluster", 260, 264, 520, {"VARIANT": 1, "TILE_N": 128, "SPLIT_K": 3,
                                               "SPLIT_MODE": 1}),
    ("split4_rowtile_cluster_l2", 260, 264, 520, {"VARIANT": 1, "TILE_N": 128, "SPLIT_K": 4,
                                                  "SPLIT_MODE": 3}),
    ("split2_swapped_cluster_l2", 40, 392, 776, {"VARIANT": 2, "SPLIT_K": 2, "SPLIT_MODE": 3}),
    ("auto_split_rowtile", 1024, 512, 2048, None),
    ("split6_swapped", 40, 392, 776, {"VARIANT": 2, "TILE_N": 16, "SPLIT_K": 6}),
    ("swapped_narrow", 100, 392, 200, {"VARIANT": 2, "TILE_N": 32}),
    ("pair_static", 1000, 520, 200, {"VARIANT": 3, "TILE_ORDER": 1}),
    ("pair_dynamic_walk", 1000, 520, 200, {"VARIANT": 3, "TILE_ORDER": 2, "GRID": 4}),
    ("persistent", 640, 512, 520, {"VARIANT": 1, "TILE_N": 128, "GRID": 3, "GROUP_M": 2}),
]


@pytest.mark.parametrize("name,m,n,k,opts", VARIANTS, ids=[v[0] for v in VARIANTS])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_backward_parity(name, m, n, k, opts, kind, layout):
    dtype = "f16" if (len(name) + KINDS.index(kind)) % 3 == 0 else "bf16"
    inp = _bwd_inputs(m, n, k, dtype, seed=len(name) * 31 + m + KINDS.index(kind))
    _check_bwd(inp, m, n, k, dtype, kind, layout, options=opts)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("layout", ["M1", "1N"])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_backward_default_plan(kind, layout, dtype):
    m, n, k = 1000, 776, 328
    inp = _bwd_inputs(m, n, k, dtype, seed=4242)
    _check_bwd(inp, m, n, k, dtype, kind, layout)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_backward_unfused(kind, layout):
    m, n, k = 300, 264, 136
    inp = _bwd_inputs(m, n, k, "bf16", seed=17)
    _check_bwd(inp, m, n, k, "bf16", kind, layout, unfused=True)


# ---- integer inputs: every product and sum exact in fp32 -----------------------------------

@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_drelu_integer_bit_exact(variant, layout):
    m = 200 if variant == 2 else 520
    n, k = 264, 64
    p = workloads.random_problem(m, n, k, dtype="bf16", seed=90 + variant, kind="int")
    inp = _bwd_inputs(m, n, k, "bf16", seed=91 + variant)
    inp["A"], inp["B"] = p["A"], p["B"]
    D, dbias, desc = _run_bwd(inp, m, n, k, "bf16", "DRELU_BGRAD", layout,
                              options={"VARIANT": variant})
    want, want_db = _oracle_bwd(inp, "bf16", "DRELU_BGRAD", layout)
    assert np.array_equal(D.float().double().numpy(), want), desc
    assert np.array_equal(dbias, want_db), desc


# ---- edge cases ----------------------------------------------------------------------------

@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_backward_k_zero(kind, layout):
    m, n = 70, 72
    inp = _bwd_inputs(m, n, 0, "bf16", seed=3)
    D, dbias, want, want_db, _ = _check_bwd(inp, m, n, 0, "bf16", kind, layout)
    assert not D.float().abs().sum() and not np.abs(dbias).sum()


@pytest.mark.parametrize("m,n", [(0, 64), (64, 0)])
@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_backward_empty_zeroes_dbias(m, n, layout):
    dev = torch.device("cuda")
    nb = m if layout == "M1" else n
    dbias = torch.full((max(nb, 1),), float("nan"), dtype=torch.float32, device=dev)
    D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    mask = torch.zeros((m, (n + 31) // 32), dtype=torch.int32, device=dev)
    A = torch.empty((m, 64), dtype=torch.bfloat16, device=dev)
    B = torch.empty((64, n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, 64, "bf16", "DRELU_BGRAD", layout) as plan:
        plan.execute(A, B, None, D, aux_in=mask, dbias=dbias)
        assert plan.sync_status() == 0
    got = dbias.cpu()
    if nb:
        assert torch.all(got[:nb] == 0)
    else:
        assert torch.isnan(got[0])  # nothing written


def test_mask_extremes_and_pad_bits():
    """All-ones mask (pad bits too) gives A.B itself; all-zeros gives 0 and dbias 0."""
    m, n, k = 136, 200, 72
    inp = _bwd_inputs(m, n, k, "bf16", seed=8)
    words = (n + 31) // 32
    for fill, name in [(0xFFFFFFFF, "ones"), (0, "zeros")]:
        inp["mask"] = np.full((m, words), fill, np.uint32)
        D, dbias, want, want_db, desc = _check_bwd(inp, m, n, k, "bf16", "DRELU_BGRAD", "1N",
                                                   options={"VARIANT": 1, "TILE_N": 64})
        if name == "zeros":
            assert not D.float().abs().sum() and not np.abs(dbias).sum()
        else:
            plain = oracle.gemm_epi(inp["A"], inp["B"], None, dtype="bf16", epilog="NONE")
            assert rel_err(D, plain) <= TOL["bf16"]


def test_operand_rules():
    dev = torch.device("cuda")
    m, n, k = 64, 64, 64
    A = torch.zeros((m, k), dtype=torch.bfloat16, device=dev)
    B = torch.zeros((k, n), dtype=torch.bfloat16, device=dev)
    D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    mask = torch.zeros((m, 2), dtype=torch.int32, device=dev)
    dbias = torch.zeros((n,), dtype=torch.float32, device=dev)
    bias = torch.zeros((n,), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "DRELU_BGRAD", "1N") as plan:
        for kw in [dict(aux_in=mask), dict(dbias=dbias),
                   dict(aux_in=mask, dbias=dbias, bias=bias),
                   dict(aux_in=mask, dbias=dbias, aux=mask)]:
            b = kw.pop("bias", None)
            with pytest.raises(gemm_epi.GemmEpiError) as e:
                plan.execute(A, B, b, D, **kw)
            assert e.value.status == 1
        with pytest.raises(gemm_epi.GemmEpiError) as e:  # misaligned dbias
            plan.execute(A, B, None, D, aux_in=mask, dbias=dbias.data_ptr() + 2)
        assert e.value.status == 3
    pre = torch.zeros((m, n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "DGELU_BGRAD", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:  # pre must be 16-byte aligned
            plan.execute(A, B, None, D, aux_in=pre.data_ptr() + 2, dbias=dbias)
        assert e.value.status == 3
    with gemm_epi.Plan(m, n, k, "bf16", "GELU_AUX_BIAS", "1N") as plan:
        with pytest.raises(gemm_epi.GemmEpiError) as e:  # GELU_AUX_BIAS needs aux
            plan.execute(A, B, bias, D)
        assert e.value.status == 1


# ---- forward -> backward chains ---------------------------------------------------------

@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_relu_aux_mask_feeds_drelu(layout):
    """The mask RELU_AUX_BIAS writes is the aux_in of DRELU_BGRAD (same words, same layout)."""
    m, n, k = 384, 264, 136
    dev = torch.device("cuda")
    fw = workloads.random_problem(m, n, k, dtype="bf16", bias_layout=layout, seed=123)
    words = torch.empty((m, (n + 31) // 32), dtype=torch.int32, device=dev)
    Y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "RELU_AUX_BIAS", layout) as plan:
        plan.execute(fw["A"].to(dev), fw["B"].to(dev), fw["bias"].to(dev), Y, aux=words)
        assert plan.sync_status() == 0
    # backward through the same layer: dY (m x n) = G . W for some incoming G (m x k2)
    k2 = 200
    bw = workloads.random_problem(m, n, k2, dtype="bf16", seed=124)
    inp = {"A": bw["A"], "B": bw["B"], "mask": words.cpu().numpy().view(np.uint32),
           "pre": None}
    _check_bwd(inp, m, n, k2, "bf16", "DRELU_BGRAD", layout)


@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_gelu_aux_pre_feeds_dgelu(layout):
    m, n, k = 300, 264, 136
    dev = torch.device("cuda")
    fw = workloads.random_problem(m, n, k, dtype="bf16", bias_layout=layout, seed=321)
    pre = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    Y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(m, n, k, "bf16", "GELU_AUX_BIAS", layout) as plan:
        plan.execute(fw["A"].to(dev), fw["B"].to(dev), fw["bias"].to(dev), Y, aux=pre)
        assert plan.sync_status() == 0
    k2 = 72
    bw = workloads.random_problem(m, n, k2, dtype="bf16", seed=322)
    inp = {"A": bw["A"], "B": bw["B"], "mask": None, "pre": pre.cpu()}
    _check_bwd(inp, m, n, k2, "bf16", "DGELU_BGRAD", layout)
