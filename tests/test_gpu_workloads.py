"""Parity at the full sizes of the five seeded workloads, in the launch configuration the
benchmark times (the automatic plan), against the CPU oracle.

The 65536 x 16384 x 8192 problem is too large for the oracle in full: its RELU output and
mask are compared on 256 seeded random rows plus every row on a 128-row tile boundary,
all 16384 columns; and a BIAS run of the same shape is checked everywhere with a
Freivalds test, D.x against A.(B.x) + bias * sum(x) for random +-1 vectors x.
"""
import numpy as np
import pytest
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi, workloads
from parity_helpers import TOL, aux_bad_bits, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _execute(w, inp, dev):
    td = workloads.TORCH_DTYPES[w.dtype]
    D = torch.empty((w.m, w.n), dtype=td, device=dev)
    aux = None
    if w.epilog == "RELU_AUX_BIAS":
        aux = torch.full((w.m, (w.n + 31) // 32), -1, dtype=torch.int32, device=dev)
    with gemm_epi.Plan(w.m, w.n, w.k, w.dtype, w.epilog, w.bias_layout) as plan:
        plan.execute(inp["A"], inp["B"], inp["bias"], D, aux=aux)
        assert plan.sync_status() == 0
        desc = plan.describe()
    return D, aux, desc


@pytest.mark.parametrize("name", [n for n in workloads.GEMMS
                                  if n != "relu_bias_bf16_65536x16384x8192"])
def test_workload_full_parity(name):
    w = workloads.GEMMS[name]
    dev = torch.device("cuda")
    inp = workloads.gemm_inputs(w, device=dev)
    D, aux, desc = _execute(w, inp, dev)
    cpu = {k: v.cpu() for k, v in inp.items()}
    want, pre = oracle.gemm_epi(cpu["A"], cpu["B"], cpu["bias"], dtype=w.dtype, epilog=w.epilog,
                                bias_layout=w.bias_layout, want_pre=True)
    err = rel_err(D, want)
    assert err <= TOL[w.dtype], f"{name}: rel err {err:.3e} ({desc})"
    if aux is not None:
        assert aux_bad_bits(aux.cpu().numpy().view(np.uint32), pre) == 0


def test_ffn_full_parity():
    f = workloads.FFNS["ffn_bf16_4096x1024x4096"]
    dev = torch.device("cuda")
    fi = workloads.ffn_inputs(f, device=dev)
    H = torch.empty((f.t, f.f), dtype=torch.bfloat16, device=dev)
    Y = torch.empty((f.t, f.d), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(f.t, f.f, f.d, "bf16", "GELU_BIAS", "1N") as p1, \
            gemm_epi.Plan(f.t, f.d, f.f, "bf16", "BIAS_RESIDUAL", "1N") as p2:
        p1.execute(fi["X"], fi["W1"], fi["b1"], H)
        p2.execute(H, fi["W2"], fi["b2"], Y, residual=fi["R"])
        assert p1.sync_status() == 0 and p2.sync_status() == 0
    cpu = {k: v.cpu() for k, v in fi.items()}
    H_ref, H_exact, Y_ref = oracle.ffn(**cpu)
    # H from the GPU against GELU(X.W1 + b1) itself
    assert rel_err(H, H_exact) <= TOL["bf16"]
    # Y against the oracle's chain (which stores H in bf16 as the GPU does)
    assert rel_err(Y, Y_ref) <= TOL["bf16"]
    # and GEMM 2 alone on the GPU's own H
    Y2 = oracle.gemm_epi(H.cpu(), cpu["W2"], cpu["b2"], dtype="bf16", epilog="BIAS_RESIDUAL",
                         residual=cpu["R"])
    assert rel_err(Y, Y2) <= TOL["bf16"]


@pytest.mark.parametrize("launches,split2", [(1, 1), (1, 4), (2, 1), (3, 1)])
def test_ffn_full_plan_parity(launches, split2):
    """The FFN plan on the full workload: one launch (both GEMMs in one persistent kernel,
    GEMM 2 whole or in 4 K slices), two launches, and one launch with H kept on chip."""
    f = workloads.FFNS["ffn_bf16_4096x1024x4096"]
    dev = torch.device("cuda")
    fi = workloads.ffn_inputs(f, device=dev)
    Y = torch.empty((f.t, f.d), dtype=torch.bfloat16, device=dev)
    with gemm_epi.FfnPlan(f.t, f.d, f.f, "bf16", launches=launches, split2=split2) as plan:
        if launches == 1:
            assert f"in {split2} K slice" in plan.describe(), plan.describe()
        plan.execute(fi["X"], fi["W1"], fi["b1"], fi["W2"], fi["b2"], fi["R"], Y)
        assert plan.sync_status() == 0
        H = plan.hidden().cpu()
    cpu = {k: v.cpu() for k, v in fi.items()}
    H_ref, H_exact, Y_ref = oracle.ffn(**cpu)
    if launches != 3:                   # (with H on chip the hidden buffer is not written)
        assert rel_err(H, H_exact) <= TOL["bf16"]
    assert rel_err(Y, Y_ref) <= TOL["bf16"]


def _large_rows(w):
    rng = np.random.default_rng(2024)
    rows = set(rng.choice(w.m, size=256, replace=False).tolist())
    for t in range(0, w.m, 128):
        rows.update({t, t + 127})
    return np.array(sorted(r for r in rows if r < w.m), dtype=np.int64)


def test_large_relu_bias_sampled_rows():
    w = workloads.GEMMS["relu_bias_bf16_65536x16384x8192"]
    dev = torch.device("cuda")
    inp = workloads.gemm_inputs(w, device=dev)
    D, _, desc = _execute(w, inp, dev)
    rows = _large_rows(w)
    # every tile-boundary row, but only 64 columns of them; 256 random rows in full
    rng = np.random.default_rng(7)
    full_rows = np.sort(rng.choice(w.m, size=256, replace=False)).astype(np.int64)
    A_rows = inp["A"][torch.from_numpy(full_rows).to(dev)].cpu()
    B = inp["B"].cpu()
    bias = inp["bias"].cpu()
    want = oracle.gemm_epi(A_rows, B, bias, dtype=w.dtype, epilog=w.epilog,
                           bias_layout=w.bias_layout)
    got = D[torch.from_numpy(full_rows).to(dev)]
    assert rel_err(got, want) <= TOL[w.dtype], desc
    cols = np.concatenate([np.arange(0, w.n, 256), np.arange(255, w.n, 256)])[:64]
    cols = np.unique(cols).astype(np.int64)
    A_b = inp["A"][torch.from_numpy(rows).to(dev)].cpu()
    want_b = oracle.gemm_epi(A_b, B, bias, dtype=w.dtype, epilog=w.epilog,
                             bias_layout=w.bias_layout, cols=cols)
    got_b = D[torch.from_numpy(rows).to(dev)][:, torch.from_numpy(cols).to(dev)]
    assert rel_err(got_b, want_b) <= TOL[w.dtype], desc


def test_large_bias_freivalds():
    w = workloads.GEMMS["relu_bias_bf16_65536x16384x8192"]
    dev = torch.device("cuda")
    inp = workloads.gemm_inputs(w, device=dev)
    D = torch.empty((w.m, w.n), dtype=torch.bfloat16, device=dev)
    with gemm_epi.Plan(w.m, w.n, w.k, "bf16", "BIAS", "1N") as plan:
        plan.execute(inp["A"], inp["B"], inp["bias"], D)
        assert plan.sync_status() == 0
    g = torch.Generator().manual_seed(99)
    X = (torch.randint(0, 2, (w.n, 2), generator=g) * 2 - 1).to(torch.float64)
    # right side on the host in float64, from the exact 16-bit inputs, in row blocks
    Bd = oracle.decode("bf16", inp["B"].cpu())                      # k x n
    bx = Bd @ X.numpy()                                              # k x 2
    beta = oracle.decode("bf16", inp["bias"].cpu())                  # n
    sx = beta @ X.numpy()                                            # 2
    Dx = np.empty((w.m, 2))
    Abx = np.empty((w.m, 2))
    step = 4096
    for r0 in range(0, w.m, step):
        Dd = oracle.decode("bf16", D[r0:r0 + step].cpu())
        Dx[r0:r0 + step] = Dd @ X.numpy()
        Ad = oracle.decode("bf16", inp["A"][r0:r0 + step].cpu())
        Abx[r0:r0 + step] = Ad @ bx + sx
        rms = np.sqrt(np.mean(Dd ** 2, axis=1))
        # bf16 output rounding: each element off by <= 2^-8 relative, random signs; six
        # standard deviations of the sum over n columns, plus fp32 accumulation slack
        tol = 6 * 2.0 ** -8 * rms * np.sqrt(w.n) + 1e-3 * np.sqrt(w.n)
        bad = np.abs(Dx[r0:r0 + step] - Abx[r0:r0 + step]) > tol[:, None]
        assert not bad.any(), f"Freivalds check failed in rows {r0}..{r0 + step}"
