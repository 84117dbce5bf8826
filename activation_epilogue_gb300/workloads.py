"""Seeded synthetic inputs for the GEMM + epilogue workloads.

This module only draws random tensors: it holds shapes, distributions and seeds and none
of the method's arithmetic, so that the CUDA path's tests and the CPU oracle can be fed the
same inputs.  Every tensor is drawn in float32 from one ``torch.Generator`` per workload,
seeded with the workload's seed, in the order the workload lists its tensors, scaled by
its standard deviation and then rounded (round-to-nearest-even) to the 16-bit dtype.

Distributions: ``N(0, v)`` with ``v = 1/fan_in`` (1/4096, 1/8192) is read as a variance
(sigma = 1/sqrt(fan_in)); the decimal constants (0.02, 0.1, 1) are standard deviations.

The workloads are the page-1 worked example's shapes (m, n, k = 1024, 512, 2048 with a
(m,1) fp16 bias; "Fusing bias into cuBLASLt matmul with nvmath-python", code example),
a square RELU(_AUX)_BIAS GEMM, the small-batch GELU_BIAS inference shapes, the large
RELU_BIAS GEMM (the 65536 x 16384 output the same page names), and the FFN block of
"Operator fusion in model inference" (section 1 flowchart).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Gemm:
    """One GEMM + epilogue workload: D[m,n] = epi(A[m,k] . B[k,n] + bias)."""
    name: str
    m: int
    n: int
    k: int
    dtype: str
    epilog: str
    bias_layout: str            # "M1" = bias (m,1), "1N" = bias (1,n)
    seed: int
    sigma_a: float
    sigma_b: float
    sigma_bias: float
    sigma_residual: float = 1.0

    @property
    def flops(self) -> int:
        return 2 * self.m * self.n * self.k


@dataclass(frozen=True)
class Ffn:
    """The FFN block: H = GELU(X.W1 + b1) (stored 16-bit), Y = H.W2 + b2 + R."""
    name: str
    t: int
    d: int
    f: int
    dtype: str
    seed: int
    sigma_x: float = 1.0
    sigma_w: float = 0.02
    sigma_r: float = 1.0

    @property
    def flops(self) -> int:
        return 2 * 2 * self.t * self.d * self.f


GEMMS = {
    g.name: g for g in [
        Gemm("bias_f16_1024x512x2048", 1024, 512, 2048, "f16", "BIAS", "M1", 1001,
             1.0, 1.0, 1.0),
        Gemm("relu_bias_bf16_4096", 4096, 4096, 4096, "bf16", "RELU_BIAS", "1N", 1002,
             1 / 64.0, 1 / 64.0, 0.1),
        Gemm("relu_aux_bias_bf16_4096", 4096, 4096, 4096, "bf16", "RELU_AUX_BIAS", "1N",
             1002, 1 / 64.0, 1 / 64.0, 0.1),
        Gemm("gelu_bias_bf16_t16", 16, 3072, 768, "bf16", "GELU_BIAS", "1N", 3016,
             1.0, 0.02, 0.02),
        Gemm("gelu_bias_bf16_t64", 64, 3072, 768, "bf16", "GELU_BIAS", "1N", 3064,
             1.0, 0.02, 0.02),
        Gemm("gelu_bias_bf16_t256", 256, 3072, 768, "bf16", "GELU_BIAS", "1N", 3256,
             1.0, 0.02, 0.02),
        Gemm("relu_bias_bf16_65536x16384x8192", 65536, 16384, 8192, "bf16", "RELU_BIAS",
             "1N", 1004, 1 / math.sqrt(8192.0), 1.0, 1.0),
    ]
}

FFNS = {"ffn_bf16_4096x1024x4096": Ffn("ffn_bf16_4096x1024x4096", 4096, 1024, 4096, "bf16",
                                       1005)}


def _draw(g: torch.Generator, shape, sigma: float, dtype: str, device) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(TORCH_DTYPES[dtype])


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def gemm_inputs(w: Gemm, device="cpu") -> dict:
    """A, B, bias (and R for BIAS_RESIDUAL), drawn in that order."""
    g = _generator(w.seed, device)
    out = {
        "A": _draw(g, (w.m, w.k), w.sigma_a, w.dtype, device),
        "B": _draw(g, (w.k, w.n), w.sigma_b, w.dtype, device),
        "bias": _draw(g, (w.m if w.bias_layout == "M1" else w.n,), w.sigma_bias, w.dtype,
                      device),
    }
    if w.epilog == "BIAS_RESIDUAL":
        out["R"] = _draw(g, (w.m, w.n), w.sigma_residual, w.dtype, device)
    return out


def ffn_inputs(w: Ffn, device="cpu") -> dict:
    """X, W1, b1, W2, b2, R, drawn in that order."""
    g = _generator(w.seed, device)
    return {
        "X": _draw(g, (w.t, w.d), w.sigma_x, w.dtype, device),
        "W1": _draw(g, (w.d, w.f), w.sigma_w, w.dtype, device),
        "b1": _draw(g, (w.f,), w.sigma_w, w.dtype, device),
        "W2": _draw(g, (w.f, w.d), w.sigma_w, w.dtype, device),
        "b2": _draw(g, (w.d,), w.sigma_w, w.dtype, device),
        "R": _draw(g, (w.t, w.d), w.sigma_r, w.dtype, device),
    }


def layer_stack_inputs(t: int, d: int, f: int, layers: int, *, dtype: str = "bf16",
                       seed: int = 0, device="cpu") -> dict:
    """A stack of FFN layers at small batch: X[t,d] ~ N(0,1), then for each layer W1[d,f],
    b1[f], W2[f,d], b2[d] ~ N(0, 0.02) (the small-batch GELU_BIAS workload's and the FFN
    block's distributions), drawn in that order; returns {"X": X, "layers": [(W1, b1, W2,
    b2), ...]}."""
    g = _generator(seed, device)
    X = _draw(g, (t, d), 1.0, dtype, device)
    stack = []
    for _ in range(layers):
        stack.append((_draw(g, (d, f), 0.02, dtype, device), _draw(g, (f,), 0.02, dtype, device),
                      _draw(g, (f, d), 0.02, dtype, device), _draw(g, (d,), 0.02, dtype, device)))
    return {"X": X, "layers": stack}


def random_problem(m: int, n: int, k: int, *, dtype: str = "bf16", bias_layout: str = "1N",
                   residual: bool = False, seed: int = 0, kind: str = "normal",
                   sigma_a: float | None = None, device="cpu") -> dict:
    """Inputs for parity tests at arbitrary shapes.

    kind="normal": A ~ N(0, 1/k) (so A.B is O(1)), B ~ N(0,1), bias and R ~ N(0,1).
    kind="int":    every element an integer drawn uniformly from {-2, ..., 2}; with small k
                   all sums are exact in fp32, which makes any correct result bit-exact.
    """
    g = _generator(seed, device)
    if kind == "int":
        def draw(shape, _sigma):
            x = torch.randint(-2, 3, shape, generator=g, device=device, dtype=torch.int32)
            return x.to(torch.float32).to(TORCH_DTYPES[dtype])
    else:
        def draw(shape, sigma):
            return _draw(g, shape, sigma, dtype, device)
    sa = sigma_a if sigma_a is not None else 1.0 / math.sqrt(max(k, 1))
    out = {
        "A": draw((m, k), sa),
        "B": draw((k, n), 1.0),
        "bias": draw((m if bias_layout == "M1" else n,), 1.0),
    }
    if residual:
        out["R"] = draw((m, n), 1.0)
    return out


def random_backward_problem(m: int, n: int, k: int, *, dtype: str = "bf16", seed: int = 0,
                            device="cpu") -> dict:
    """Inputs of a backward epilogue: A (m x k) and B (k x n) as in random_problem (the
    incoming gradient and the weight), ReLU mask words uint32 [m][ceil(n/32)] with every bit
    (the pad bits too) drawn fair, and a stored pre-activation ~ N(0, 2^2) in dtype."""
    p = random_problem(m, n, k, dtype=dtype, seed=seed, device=device)
    g = _generator(seed + 99991, device)
    words = (n + 31) // 32
    halves = torch.randint(0, 1 << 16, (m, words, 2), generator=g, dtype=torch.int64,
                           device=device)
    mask = (halves[..., 0] | (halves[..., 1] << 16)).to(torch.int64)
    pre = _draw(g, (m, n), 2.0, dtype, device)
    return {"A": p["A"], "B": p["B"],
            "mask": mask.cpu().numpy().astype(np.uint32), "pre": pre}


def random_fp8_problem(m: int, n: int, k: int, *, bias_layout: str = "1N", seed: int = 0,
                       residual: bool = False, device="cpu") -> dict:
    """Inputs of an FP8 GEMM: A (m x k) and Bt (n x k, B transposed) drawn N(0, 1) in fp32 and
    rounded to E4M3 (torch's float8_e4m3fn conversion), per-tensor scales 1/sqrt(k) and 1/2
    (so A.B scaled is O(1)), bias and residual N(0, 1) in bf16."""
    g = _generator(seed, device)
    A = torch.randn((m, k), generator=g, device=device).to(torch.float8_e4m3fn)
    Bt = torch.randn((n, k), generator=g, device=device).to(torch.float8_e4m3fn)
    out = {"A": A, "Bt": Bt, "scale_a": 1.0 / math.sqrt(max(k, 1)), "scale_b": 0.5,
           "bias": _draw(g, (m if bias_layout == "M1" else n,), 1.0, "bf16", device)}
    if residual:
        out["R"] = _draw(g, (m, n), 1.0, "bf16", device)
    return out
