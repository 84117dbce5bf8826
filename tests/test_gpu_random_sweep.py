"""A seeded random sweep over shapes, dtypes, epilogs, bias layouts, kernel variants and tile
orders, each case checked element by element against the CPU oracle (the fixed-shape tests
cover the edges deliberately; this covers the combinations between them)."""
import os
import random

import numpy as np
import pytest
import torch

from activation_epilogue_gb300 import workloads
from parity_helpers import check

pytestmark = pytest.mark.gpu

EPILOGS = ["BIAS", "RELU_BIAS", "GELU_BIAS", "RELU_AUX_BIAS", "BIAS_RESIDUAL", "NONE",
           "TANH_BIAS", "GELU_AUX_BIAS"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _case(i):
    r = random.Random(9000 + i)
    variant = r.choice([0, 0, 1, 2, 3, 4])      # 4: the CTA-pair kernel, static tile order
    m = r.choice([1, 7, 64, 129, 200, 256]) if variant == 2 else r.randint(1, 700)
    n = 8 * r.randint(1, 90)
    k = 8 * r.randint(1, 80)
    opts = {}
    if variant:
        opts["VARIANT"] = min(variant, 3)
    if variant in (3, 4):
        opts["TILE_ORDER"] = 2 if variant == 3 else 1
    if variant == 1:
        opts["TILE_N"] = r.choice([64, 128, 256])
    if variant in (3, 4):
        opts["TILE_N"] = r.choice([224, 256])
        if r.random() < 0.3:
            opts["GRID"] = r.choice([4, 8, 12])
    if variant == 2 and r.random() < 0.3:
        opts["TILE_N"] = r.choice([16, 32, 64, 128, 256])
    if variant in (1, 2) and r.random() < 0.3:
        mode = r.choice([1, 2, 3])               # cluster, device memory, cluster via L2
        opts["SPLIT_MODE"] = mode
        opts["SPLIT_K"] = r.randint(2, 8 if mode == 2 else 4)
    return dict(m=m, n=n, k=k, dtype=r.choice(["bf16", "f16"]), epilog=r.choice(EPILOGS),
                layout=r.choice(["M1", "1N"]), opts=opts, unfused=r.random() < 0.15,
                seed=r.randint(0, 10 ** 6))


# GEMM_EPI_SWEEP_SCALE=N runs N times as many cases of every sweep here (a longer stress run;
# 1 by default).
SCALE = max(1, int(os.environ.get("GEMM_EPI_SWEEP_SCALE", "1")))


@pytest.mark.parametrize("i", range(64 * SCALE))
def test_random_case(i):
    c = _case(i)
    p = workloads.random_problem(c["m"], c["n"], c["k"], dtype=c["dtype"], bias_layout=c["layout"],
                                 residual=True, seed=c["seed"])
    check(p, c["m"], c["n"], c["k"], c["dtype"], c["epilog"], c["layout"], unfused=c["unfused"],
          options=c["opts"])


@pytest.mark.parametrize("i", range(24 * SCALE))
def test_random_ffn_case(i):
    """The FFN plan in every mode (automatic; one launch with GEMM 2 whole or in K slices and
    either tile order; two launches; H on chip) on seeded random shapes, both 16-bit types,
    against the oracle's chain."""
    import oracle
    from activation_epilogue_gb300 import gemm_epi
    from parity_helpers import TOL, rel_err
    r = random.Random(5000 + i)
    mode = r.choice([0, 1, 2, 3])
    dtype = r.choice(["bf16", "f16"])
    t = r.randint(1, 700)
    if mode == 3:
        d, f = 256 * r.randint(1, 4), 256 * r.randint(1, 4)
    else:
        d, f = 8 * r.randint(1, 80), 8 * r.randint(1, 160)
    opts = {"launches": mode}
    if mode == 1:
        opts["split2"] = r.choice([1, 1, 2, 4])
        opts["tile_order"] = r.choice([0, 1, 2])
    g = torch.Generator().manual_seed(r.randint(0, 10 ** 6))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16

    def rn(*sh, sc=1.0):
        return (torch.randn(*sh, generator=g) * sc).to(tdt)
    cpu = dict(X=rn(t, d, sc=0.5), W1=rn(d, f, sc=0.05), b1=rn(f, sc=0.1), W2=rn(f, d, sc=0.05),
               b2=rn(d, sc=0.1), R=rn(t, d))
    dev = torch.device("cuda")
    gi = {k: v.to(dev) for k, v in cpu.items()}
    Y = torch.empty((t, d), dtype=tdt, device=dev)
    with gemm_epi.FfnPlan(t, d, f, dtype, **opts) as plan:
        plan.execute(gi["X"], gi["W1"], gi["b1"], gi["W2"], gi["b2"], gi["R"], Y)
        assert plan.sync_status() == 0
        desc = plan.describe()
    _, _, Y_ref = oracle.ffn(**cpu, dtype=dtype)
    assert rel_err(Y, Y_ref) <= TOL[dtype], desc
