"""A seeded random sweep over shapes, dtypes, epilogs, bias layouts, kernel variants and tile
orders, each case checked element by element against the CPU oracle (the fixed-shape tests
cover the edges deliberately; this covers the combinations between them)."""
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
        mode = r.choice([1, 2])                  # cluster, device memory
        opts["SPLIT_MODE"] = mode
        opts["SPLIT_K"] = r.randint(2, 4 if mode == 1 else 8)
    return dict(m=m, n=n, k=k, dtype=r.choice(["bf16", "f16"]), epilog=r.choice(EPILOGS),
                layout=r.choice(["M1", "1N"]), opts=opts, unfused=r.random() < 0.15,
                seed=r.randint(0, 10 ** 6))


@pytest.mark.parametrize("i", range(64))
def test_random_case(i):
    c = _case(i)
    p = workloads.random_problem(c["m"], c["n"], c["k"], dtype=c["dtype"], bias_layout=c["layout"],
                                 residual=True, seed=c["seed"])
    check(p, c["m"], c["n"], c["k"], c["dtype"], c["epilog"], c["layout"], unfused=c["unfused"],
          options=c["opts"])
