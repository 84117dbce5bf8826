"""Parity past 2^31 output elements.

D, the residual, the stored 16-bit pre-activation and the backward input are indexed as
row * n + column, and the mask words as row * ceil(n/32) + word.  At m x n = 139264 x 16384
(2.28e9 elements, 4.6 GB per 16-bit matrix) every row from 131072 on lies past 2^31.  A
32-bit product would wrap there, so these tests compare sampled rows on both sides of that
line, in every kernel that such a shape can reach: the automatic plan (CTA pairs,
dynamic tile order), the single-CTA row tiles, and the unfused baseline's elementwise kernel.  K = 64
keeps the GEMMs and the oracle's rows cheap.
"""
import numpy as np
import pytest
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi, workloads
from parity_helpers import TD, TOL, UNIT_ROUNDOFF, aux_bad_bits, rel_err

pytestmark = pytest.mark.gpu

M, N, K = 139264, 16384, 64
EDGE = (1 << 31) // N  # the first row whose elements all lie past index 2^31


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


@pytest.fixture(autouse=True)
def _release():
    yield
    torch.cuda.empty_cache()


def _rows(seed):
    rng = np.random.default_rng(seed)
    fixed = [0, EDGE - 1, EDGE, EDGE + 1, M - 129, M - 128, M - 1]
    past = rng.choice(np.arange(EDGE, M), 48, replace=False)
    before = rng.choice(EDGE, 16, replace=False)
    return np.unique(np.concatenate([fixed, past, before])).astype(np.int64)


def _take(t, rows):
    return t.index_select(0, torch.from_numpy(rows).to(t.device)).cpu()


@pytest.mark.parametrize("mode", ["auto", "rowtile", "unfused"])
@pytest.mark.parametrize("epilog", ["RELU_AUX_BIAS", "BIAS_RESIDUAL", "GELU_AUX_BIAS"])
def test_forward_past_2_31_elements(epilog, mode):
    dev = torch.device("cuda")
    inp = workloads.random_problem(M, N, K, dtype="bf16", seed=4100,
                                   residual=epilog == "BIAS_RESIDUAL", device=dev)
    D = torch.full((M, N), float("nan"), dtype=TD["bf16"], device=dev)
    aux = None
    if epilog == "RELU_AUX_BIAS":
        aux = torch.full((M, (N + 31) // 32), -1, dtype=torch.int32, device=dev)
    elif epilog == "GELU_AUX_BIAS":
        aux = torch.full((M, N), float("nan"), dtype=TD["bf16"], device=dev)
    options = {"VARIANT": 1} if mode == "rowtile" else {}
    with gemm_epi.Plan(M, N, K, "bf16", epilog, "1N", **options) as plan:
        if mode == "unfused":
            pre = torch.empty((M, N), dtype=TD["bf16"], device=dev)
            plan.execute_unfused(inp["A"], inp["B"], inp["bias"], pre, D, aux=aux,
                                 residual=inp.get("R"))
            del pre
        else:
            plan.execute(inp["A"], inp["B"], inp["bias"], D, aux=aux, residual=inp.get("R"))
        status = plan.sync_status()
        desc = plan.describe()
    assert status == 0, f"device status {gemm_epi.status_string(status)} ({desc})"
    if mode == "rowtile":
        assert "variant=row-tile" in desc, desc
    rows = _rows(4101)
    want, pre = oracle.gemm_epi(_take(inp["A"], rows), inp["B"].cpu(), inp["bias"].cpu(),
                                dtype="bf16", epilog=epilog, bias_layout="1N",
                                residual=_take(inp["R"], rows) if "R" in inp else None,
                                want_pre=True)
    err = rel_err(_take(D, rows), want)
    assert err <= TOL["bf16"], f"rel err {err:.3e} ({desc})"
    # The unfused baseline decides the mask on, and stores, bf16(A.B) + bias: one more
    # rounding of A.B than the fused kernels.
    ab = 0.0
    if mode == "unfused":
        ab = np.abs(oracle.gemm_epi(_take(inp["A"], rows), inp["B"].cpu(), None, dtype="bf16",
                                    epilog="NONE"))
    if epilog == "RELU_AUX_BIAS":
        words = _take(aux, rows).numpy().view(np.uint32)
        assert aux_bad_bits(words, pre, 1e-3 + 2 * UNIT_ROUNDOFF["bf16"] * ab) == 0, desc
    elif epilog == "GELU_AUX_BIAS":
        stored = _take(aux, rows).float().double().numpy()
        slack = UNIT_ROUNDOFF["bf16"] * ab
        bad = np.abs(stored - pre) > TOL["bf16"] * (np.abs(pre) + 1.0) + slack
        assert not bad.any(), f"{int(bad.sum())} stored pre values off ({desc})"


@pytest.mark.parametrize("kind", ["DRELU_BGRAD", "DGELU_BGRAD"])
def test_backward_past_2_31_elements(kind):
    """(m,1) layout: each row's bias gradient depends on that row alone, so the sampled rows
    check it too."""
    dev = torch.device("cuda")
    inp = workloads.random_backward_problem(M, N, K, dtype="bf16", seed=4200, device=dev)
    if kind == "DRELU_BGRAD":
        aux_in = torch.from_numpy(inp["mask"].view(np.int32)).to(dev)
    else:
        aux_in = inp["pre"]
    D = torch.full((M, N), float("nan"), dtype=TD["bf16"], device=dev)
    dbias = torch.full((M,), float("nan"), dtype=torch.float32, device=dev)
    with gemm_epi.Plan(M, N, K, "bf16", kind, "M1") as plan:
        plan.execute(inp["A"], inp["B"], None, D, aux_in=aux_in, dbias=dbias)
        status = plan.sync_status()
        desc = plan.describe()
    assert status == 0, f"device status {gemm_epi.status_string(status)} ({desc})"
    rows = _rows(4201)
    want, want_db = oracle.gemm_bwd(
        _take(inp["A"], rows), inp["B"].cpu(), dtype="bf16", kind=kind, bias_layout="M1",
        mask=inp["mask"][rows] if kind == "DRELU_BGRAD" else None,
        pre=_take(inp["pre"], rows) if kind == "DGELU_BGRAD" else None)
    got = _take(D, rows).float().double().numpy()
    bad = np.abs(got - want) > TOL["bf16"] * (np.abs(want) + 1.0)
    assert not bad.any(), f"{int(bad.sum())} D values off ({desc})"
    db = dbias.index_select(0, torch.from_numpy(rows).to(dev)).cpu().double().numpy()
    bound = 1e-4 * (np.abs(want).sum(axis=1) + 1.0)
    assert np.all(np.abs(db - want_db) <= bound), desc
