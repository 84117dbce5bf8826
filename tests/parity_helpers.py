"""Shared pieces of the GPU parity tests: run the library through its C ABI and compare
with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi

# Acceptance bound: max |gpu - oracle| / (|oracle| + 1), by output dtype.
TOL = {"f16": 8e-3, "bf16": 2e-2}
# Aux bits may differ from the oracle only where the fp32 pre-activation is this close to 0.
AUX_BAND = 1e-3

TD = {"f16": torch.float16, "bf16": torch.bfloat16}


def rel_err(got: torch.Tensor, want: np.ndarray) -> float:
    g = got.detach().float().cpu().double().numpy()
    if g.size == 0:
        return 0.0
    return float(np.max(np.abs(g - want) / (np.abs(want) + 1.0)))


# Unit roundoff of the 16-bit formats (the unfused baseline stores A.B rounded to these).
UNIT_ROUNDOFF = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def aux_bad_bits(words: np.ndarray, pre: np.ndarray, band=AUX_BAND) -> int:
    """Mask bits that differ from [pre > 0] outside the |pre| < band region (a scalar or an
    array like pre), plus any nonzero pad bit."""
    m, n = pre.shape
    words = np.ascontiguousarray(words).view(np.uint32).reshape(m, -1)
    bits = np.unpackbits(words.view(np.uint8), axis=1, bitorder="little").astype(bool)
    want = np.zeros_like(bits)
    want[:, :n] = pre > 0
    diff = bits != want
    inband = np.zeros_like(bits)
    inband[:, :n] = np.abs(pre) < band
    return int(np.count_nonzero(diff & ~inband))


def run(inputs: dict, m: int, n: int, k: int, dtype: str, epilog: str, layout: str,
        unfused: bool = False, options: dict | None = None, device="cuda"):
    """Execute one plan on `inputs` (CPU tensors); returns (D, aux words, describe)."""
    dev = torch.device(device)
    A = inputs["A"].to(dev)
    B = inputs["B"].to(dev)
    bias = inputs["bias"].to(dev) if epilog != "NONE" else None
    R = inputs["R"].to(dev) if epilog == "BIAS_RESIDUAL" else None
    D = torch.full((m, n), float("nan"), dtype=TD[dtype], device=dev)
    aux = None
    if epilog == "RELU_AUX_BIAS":
        aux = torch.full((m, (n + 31) // 32), -1, dtype=torch.int32, device=dev)
    elif epilog == "GELU_AUX_BIAS":
        aux = torch.full((m, n), float("nan"), dtype=TD[dtype], device=dev)
    with gemm_epi.Plan(m, n, k, dtype, epilog, layout, **(options or {})) as plan:
        if unfused:
            pre = torch.empty((m, n), dtype=TD[dtype], device=dev)
            plan.execute_unfused(A, B, bias, pre, D, aux=aux, residual=R)
        else:
            plan.execute(A, B, bias, D, aux=aux, residual=R)
        status = plan.sync_status()
        desc = plan.describe()
    assert status == 0, f"device status {gemm_epi.status_string(status)} ({desc})"
    if aux is None:
        return D.cpu(), None, desc
    if epilog == "GELU_AUX_BIAS":
        return D.cpu(), aux.cpu(), desc  # the stored 16-bit pre-activation
    return D.cpu(), aux.cpu().numpy().view(np.uint32), desc


def oracle_ref(inputs: dict, dtype: str, epilog: str, layout: str):
    """(D, pre) from the oracle in double."""
    return oracle.gemm_epi(inputs["A"], inputs["B"], None if epilog == "NONE" else inputs["bias"],
                           dtype=dtype, epilog=epilog, bias_layout=layout,
                           residual=inputs.get("R") if epilog == "BIAS_RESIDUAL" else None,
                           want_pre=True)


def check(inputs, m, n, k, dtype, epilog, layout, unfused=False, options=None, exact=False):
    D, words, desc = run(inputs, m, n, k, dtype, epilog, layout, unfused=unfused,
                         options=options)
    want, pre = oracle_ref(inputs, dtype, epilog, layout)
    if exact:
        got = D.float().double().numpy()
        assert np.array_equal(got, want), f"not bit-exact ({desc})"
        assert not np.any(np.signbit(got) & (got == 0) & ~np.signbit(want)), "negative zero"
    else:
        err = rel_err(D, want)
        assert err <= TOL[dtype], f"rel err {err:.3e} > {TOL[dtype]} ({desc})"
    if words is not None and epilog == "GELU_AUX_BIAS":
        # the stored pre-activation: one rounding of the fp32 value to the output format
        # (unfused: of bf16/f16(A.B) + bias, which adds one rounding of A.B)
        got = words.float().double().numpy()
        slack = 0.0
        if unfused:
            pre0 = oracle.gemm_epi(inputs["A"], inputs["B"], None, dtype=dtype, epilog="NONE")
            slack = UNIT_ROUNDOFF[dtype] * np.abs(pre0)
        bad = np.abs(got - pre) > TOL[dtype] * (np.abs(pre) + 1.0) + slack
        assert not bad.any(), f"{int(bad.sum())} stored pre values off ({desc})"
    elif words is not None:
        band = AUX_BAND
        if unfused:
            # The unfused baseline decides the mask on bf16/f16(A.B) + bias: its decision
            # may differ within one rounding of A.B of zero.
            pre0 = oracle.gemm_epi(inputs["A"], inputs["B"], None, dtype=dtype, epilog="NONE")
            band = AUX_BAND + 2 * UNIT_ROUNDOFF[dtype] * np.abs(pre0)
        bad = aux_bad_bits(words, pre, band)
        assert bad == 0, f"{bad} aux bits differ ({desc})"
    return D, words, want, pre, desc
