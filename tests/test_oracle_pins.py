"""Pins for the CPU oracle, against things other than itself (no GPU needed).

Each test checks the oracle against a library routine, a closed form, a textbook value or
an independent brute force, chosen so that a plausible slip in the oracle (a dropped
bias, a wrong broadcast axis, a transposed operand, a wrong GELU form, a wrong bit order)
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from activation_epilogue_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lib_decode(dtype, bits):
    """Decode 16-bit payloads with numpy (binary16) or torch (bfloat16), not the oracle."""
    bits = np.ascontiguousarray(bits, np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _bits_np(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---- 16-bit decode / encode --------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_every_pattern_matches_library(oracle, dtype):
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode(dtype, bits)
    ref = _lib_decode(dtype, bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero is kept
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_encode_f16_matches_numpy_rounding(oracle):
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 6, 200000),
        # exact ties half-way between neighbouring binary16 values, normal and subnormal
        (np.arange(1, 4000, dtype=np.float64) + 0.5) * 2.0 ** -24,
        (np.arange(1024, 3000, dtype=np.float64) + 0.5) * 2.0 ** -10,
        [65504.0, 65519.99, 65520.0, 70000.0, -65520.0, 2.0 ** -25, 2.0 ** -26, 0.0, -0.0],
    ])
    ours = oracle.encode("f16", x)
    ref = x.astype(np.float16).view(np.uint16)      # numpy rounds float64 -> binary16 RNE
    assert np.array_equal(ours, ref)


def test_encode_bf16_matches_torch_on_float32_values(oracle):
    # torch rounds float32 -> bfloat16 to nearest-even; feed float32-exact doubles so the
    # library result is a single correct rounding.
    g = torch.Generator().manual_seed(3)
    x32 = torch.randn(200000, generator=g) * torch.pow(10.0, torch.randint(-30, 30, (200000,),
                                                                              generator=g))
    x32 = torch.cat([x32, torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8),
                                        3.3895314e38, 3.40e38, 1e-40, 0.0, -0.0])])
    ours = oracle.encode("bf16", x32.double().numpy())
    ref = _bits_np(x32.to(torch.bfloat16))
    assert np.array_equal(ours, ref)


def test_encode_bf16_ties_to_even(oracle):
    # 1 + 2^-8 is half-way between 1 and 1 + 2^-7: ties go to the even neighbour, 1.0.
    assert oracle.encode("bf16", np.array([1 + 2 ** -8]))[0] == 0x3F80
    # 1 + 3*2^-8 is half-way between 1 + 2^-7 (odd) and 1 + 2^-6 (even).
    assert oracle.encode("bf16", np.array([1 + 3 * 2 ** -8]))[0] == 0x3F82
    # just above the tie rounds up
    assert oracle.encode("bf16", np.array([1 + 2 ** -8 + 2 ** -30]))[0] == 0x3F81


# ---- GELU ----------------------------------------------------------------------------------

def _phi_table():
    rows = []
    with open(os.path.join(GOLDEN, "standard_normal_cdf.txt")) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                x, p = line.split()
                rows.append((float(x), float(p)))
    return rows


def test_gelu_textbook_points(oracle):
    for x, phi in _phi_table():
        # the table has 10 decimals: |x| * 0.5e-10 is its rounding
        assert abs(oracle.gelu(x) - x * phi) <= 0.6e-10 * max(abs(x), 1.0), x


def test_gelu_matches_library_cdf_and_not_tanh_form(oracle):
    from scipy.special import ndtr
    xs = np.linspace(-8, 8, 4001)
    ours = np.array([oracle.gelu(x) for x in xs])
    ref = xs * ndtr(xs)
    assert np.max(np.abs(ours - ref) / (np.abs(ref) + 1e-300)) < 1e-13 or \
        np.max(np.abs(ours - ref)) < 1e-15
    tanh_form = 0.5 * xs * (1 + np.tanh(math.sqrt(2 / math.pi) * (xs + 0.044715 * xs ** 3)))
    assert np.max(np.abs(ours - tanh_form)) > 1e-4   # the tanh approximation is not GELU here


def test_gelu_closed_forms(oracle):
    assert oracle.gelu(0.0) == 0.0
    for x in [6.0, 8.0, 10.0, 30.0]:
        assert abs(oracle.gelu(x) / x - 1.0) < 1e-8
    for x in [0.1, 0.7, 1.3, 2.9, 5.0]:
        # Phi(-x) = 1 - Phi(x)  =>  GELU(-x) = GELU(x) - x
        assert abs(oracle.gelu(-x) - (oracle.gelu(x) - x)) < 1e-14
    # far left tail keeps relative accuracy: GELU(-10) = -10 * Phi(-10) ~ -7.62e-23
    assert abs(oracle.gelu(-10.0) / (-10.0 * 7.619853024160527e-24) - 1.0) < 1e-9


# ---- the GEMM + epilogue ------------------------------------------------------------------

EPILOGS = ["BIAS", "RELU_BIAS", "GELU_BIAS", "RELU_AUX_BIAS", "BIAS_RESIDUAL", "NONE", "TANH_BIAS"]


def _brute(dtype, epilog, layout, A, B, bias, R):
    """Naive triple loop in Python floats, from the definition (independent of the oracle)."""
    from scipy.special import ndtr
    Ad, Bd = _lib_decode(dtype, _bits_np(A)), _lib_decode(dtype, _bits_np(B))
    bd = _lib_decode(dtype, _bits_np(bias))
    Rd = None if R is None else _lib_decode(dtype, _bits_np(R))
    m, k = Ad.shape
    n = Bd.shape[1]
    pre = np.zeros((m, n))
    D = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            s = 0.0
            for kk in range(k):
                s += Ad[i, kk] * Bd[kk, j]
            if epilog != "NONE":
                s += bd[i] if layout == "M1" else bd[j]
            pre[i, j] = s
            if epilog in ("RELU_BIAS", "RELU_AUX_BIAS"):
                D[i, j] = s if s > 0 else 0.0
            elif epilog == "GELU_BIAS":
                D[i, j] = s * float(ndtr(s))
            elif epilog == "TANH_BIAS":
                D[i, j] = math.tanh(s)
            elif epilog == "BIAS_RESIDUAL":
                D[i, j] = s + Rd[i, j]
            else:
                D[i, j] = s
    return pre, D


def test_brute_force_all_tiny_shapes(oracle):
    combo = 0
    for m in range(1, 10):
        for n in range(1, 10):
            for k in range(1, 10):
                epilog = EPILOGS[combo % len(EPILOGS)]
                layout = "M1" if (combo // len(EPILOGS)) % 2 else "1N"
                dtype = "bf16" if combo % 3 else "f16"
                combo += 1
                p = workloads.random_problem(m, n, k, dtype=dtype, bias_layout=layout,
                                             residual=epilog == "BIAS_RESIDUAL", seed=combo)
                pre_ref, D_ref = _brute(dtype, epilog, layout, p["A"], p["B"], p["bias"],
                                        p.get("R"))
                D, pre = oracle.gemm_epi(p["A"], p["B"], None if epilog == "NONE" else p["bias"],
                                         dtype=dtype, epilog=epilog, bias_layout=layout,
                                         residual=p.get("R"), want_pre=True)
                np.testing.assert_allclose(pre, pre_ref, rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(D, D_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("epilog", EPILOGS)
@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_medium_shapes_match_numpy_float64_matmul(oracle, epilog, layout):
    from scipy.special import ndtr
    m, n, k = 97, 130, 211
    p = workloads.random_problem(m, n, k, dtype="bf16", bias_layout=layout, residual=True,
                                 seed=11)
    Ad, Bd = _lib_decode("bf16", _bits_np(p["A"])), _lib_decode("bf16", _bits_np(p["B"]))
    bd = _lib_decode("bf16", _bits_np(p["bias"]))
    Rd = _lib_decode("bf16", _bits_np(p["R"]))
    pre = Ad @ Bd
    if epilog != "NONE":
        pre = pre + (bd[:, None] if layout == "M1" else bd[None, :])
    ref = {"BIAS": pre, "NONE": pre, "RELU_BIAS": np.maximum(pre, 0),
           "RELU_AUX_BIAS": np.maximum(pre, 0), "GELU_BIAS": pre * ndtr(pre),
           "BIAS_RESIDUAL": pre + Rd, "TANH_BIAS": np.tanh(pre)}[epilog]
    D = oracle.gemm_epi(p["A"], p["B"], None if epilog == "NONE" else p["bias"], dtype="bf16",
                        epilog=epilog, bias_layout=layout, residual=p["R"])
    np.testing.assert_allclose(D, ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_zero_A_gives_broadcast_bias(oracle, layout):
    m, n, k = 40, 70, 33
    p = workloads.random_problem(m, n, k, dtype="f16", bias_layout=layout, seed=5)
    A0 = torch.zeros_like(p["A"])
    bd = _lib_decode("f16", _bits_np(p["bias"]))
    full = np.broadcast_to(bd[:, None] if layout == "M1" else bd[None, :], (m, n))
    D = oracle.gemm_epi(A0, p["B"], p["bias"], dtype="f16", epilog="BIAS", bias_layout=layout)
    assert np.array_equal(D, full)
    D = oracle.gemm_epi(A0, p["B"], p["bias"], dtype="f16", epilog="RELU_BIAS",
                        bias_layout=layout)
    assert np.array_equal(D, np.maximum(full, 0))


@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_identity_B_gives_A_plus_bias(oracle, layout):
    m, n = 37, 48
    p = workloads.random_problem(m, n, n, dtype="bf16", bias_layout=layout, seed=6)
    eye = torch.eye(n, dtype=torch.bfloat16)
    Ad = _lib_decode("bf16", _bits_np(p["A"]))
    bd = _lib_decode("bf16", _bits_np(p["bias"]))
    want = Ad + (bd[:, None] if layout == "M1" else bd[None, :])
    D = oracle.gemm_epi(p["A"], eye, p["bias"], dtype="bf16", epilog="BIAS", bias_layout=layout)
    assert np.array_equal(D, want)


def test_zero_bias_is_plain_gemm_and_rows_permute(oracle):
    m, n, k = 50, 60, 70
    p = workloads.random_problem(m, n, k, dtype="bf16", seed=8)
    zb = torch.zeros_like(p["bias"])
    D0 = oracle.gemm_epi(p["A"], p["B"], zb, dtype="bf16", epilog="BIAS")
    Dn = oracle.gemm_epi(p["A"], p["B"], None, dtype="bf16", epilog="NONE")
    assert np.array_equal(D0, Dn)
    perm = torch.randperm(m, generator=torch.Generator().manual_seed(1))
    Dp = oracle.gemm_epi(p["A"][perm], p["B"], p["bias"], dtype="bf16", epilog="GELU_BIAS")
    D = oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="GELU_BIAS")
    assert np.array_equal(Dp, D[perm.numpy()])


def test_sampled_rows_and_columns_match_full(oracle):
    m, n, k = 64, 96, 80
    p = workloads.random_problem(m, n, k, dtype="bf16", seed=9)
    full = oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="GELU_BIAS")
    rows = np.array([63, 0, 17, 17, 40])
    cols = np.array([95, 1, 2, 64, 31, 32])
    sub = oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="GELU_BIAS",
                          rows=rows, cols=cols)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])


def test_relu_is_max_of_bias_run_with_positive_zero(oracle):
    m, n, k = 33, 65, 40
    p = workloads.random_problem(m, n, k, dtype="bf16", seed=10)
    pre = oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="BIAS")
    relu = oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="RELU_BIAS")
    assert np.array_equal(relu, np.maximum(pre, 0.0))
    assert not np.any(np.signbit(relu))


@pytest.mark.parametrize("n", [1, 31, 32, 33, 64, 100])
def test_aux_pack_matches_packbits(oracle, n):
    rng = np.random.default_rng(n)
    pre = rng.standard_normal((7, n))
    pre[0, :] = 0.0                                   # pre == 0 gives bit 0 (strict >)
    words = oracle.aux_pack(pre)
    # library packing of the definition: LSB first, 32 bits per word, zero padding
    nw = (n + 31) // 32
    padded = np.zeros((7, nw * 32), dtype=bool)
    padded[:, :n] = pre > 0
    ref = np.packbits(padded, axis=1, bitorder="little").view("<u4").reshape(7, nw)
    assert np.array_equal(words, ref)
    assert np.all(words[0] == 0)


def test_aux_bit_order_lsb_is_lowest_column(oracle):
    pre = np.full((1, 40), -1.0)
    pre[0, 0] = 1.0
    pre[0, 33] = 2.0
    w = oracle.aux_pack(pre)
    assert w.tolist() == [[1, 2]]


def test_integer_inputs_are_exact(oracle):
    m, n, k = 20, 24, 32
    p = workloads.random_problem(m, n, k, dtype="bf16", kind="int", seed=12)
    Ai = p["A"].to(torch.int64).numpy()
    Bi = p["B"].to(torch.int64).numpy()
    bi = p["bias"].to(torch.int64).numpy()
    want = Ai @ Bi + bi[None, :]
    D = oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="BIAS")
    assert np.array_equal(D, want.astype(np.float64))


# ---- the FFN block ------------------------------------------------------------------------

def _ffn_inputs(t=24, d=40, f=56, seed=13):
    g = torch.Generator().manual_seed(seed)
    def r(*s, sc=1.0):
        return (torch.randn(*s, generator=g) * sc).to(torch.bfloat16)
    return dict(X=r(t, d), W1=r(d, f, sc=0.2), b1=r(f, sc=0.2), W2=r(f, d, sc=0.2),
                b2=r(d, sc=0.2), R=r(t, d))


def test_ffn_is_two_gemms_with_stored_bf16_hidden(oracle):
    p = _ffn_inputs()
    H, Hx, Y = oracle.ffn(**p)
    H1 = oracle.gemm_epi(p["X"], p["W1"], p["b1"], dtype="bf16", epilog="GELU_BIAS")
    assert np.array_equal(Hx, H1)
    # stored H is the RNE bfloat16 of the exact GELU output (torch rounds float32 RNE, and
    # these values are checked to be float32-exact before comparing)
    assert np.array_equal(H, oracle.encode("bf16", H1))
    Ht = torch.from_numpy(H.view(np.int16).copy()).view(torch.bfloat16)
    Y2 = oracle.gemm_epi(Ht, p["W2"], p["b2"], dtype="bf16", epilog="BIAS_RESIDUAL",
                         residual=p["R"])
    assert np.array_equal(Y, Y2)


def test_ffn_reductions(oracle):
    p = _ffn_inputs()
    t, d = p["X"].shape
    f = p["W1"].shape[1]
    # R = 0 and b2 = 0: Y is GEMM 2 alone on the stored H
    q = dict(p, R=torch.zeros(t, d, dtype=torch.bfloat16), b2=torch.zeros(d, dtype=torch.bfloat16))
    H, _, Y = oracle.ffn(**q)
    Hd = _lib_decode("bf16", H)
    W2d = _lib_decode("bf16", _bits_np(q["W2"]))
    np.testing.assert_allclose(Y, Hd @ W2d, rtol=1e-12, atol=1e-12)
    # W2 = identity slice (f >= d): Y = H[:, :d] + b2 + R
    eye = torch.eye(f, d, dtype=torch.bfloat16)
    H, _, Y = oracle.ffn(**dict(p, W2=eye))
    want = (_lib_decode("bf16", H)[:, :d] + _lib_decode("bf16", _bits_np(p["b2"]))[None, :]
            + _lib_decode("bf16", _bits_np(p["R"])))
    assert np.array_equal(Y, want)


def test_bad_arguments_are_rejected(oracle):
    p = workloads.random_problem(4, 8, 8, seed=1)
    with pytest.raises(ValueError):
        oracle.gemm_epi(p["A"], p["B"], None, dtype="bf16", epilog="BIAS")
    with pytest.raises(ValueError):
        oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="BIAS_RESIDUAL")
    with pytest.raises(ValueError):
        oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="BIAS", rows=[4])


def test_tanh_epilog_closed_forms(oracle):
    # A = 0: D = tanh(bias); odd symmetry: negating A and the bias negates D.
    m, n, k = 12, 40, 24
    p = workloads.random_problem(m, n, k, dtype="bf16", seed=14)
    bd = _lib_decode("bf16", _bits_np(p["bias"]))
    D0 = oracle.gemm_epi(torch.zeros_like(p["A"]), p["B"], p["bias"], dtype="bf16",
                         epilog="TANH_BIAS")
    # C's tanh and numpy's may differ in the last bit
    np.testing.assert_allclose(D0, np.broadcast_to(np.tanh(bd)[None, :], (m, n)), rtol=4e-16,
                               atol=0)
    D = oracle.gemm_epi(p["A"], p["B"], p["bias"], dtype="bf16", epilog="TANH_BIAS")
    Dn = oracle.gemm_epi(-p["A"], p["B"], -p["bias"], dtype="bf16", epilog="TANH_BIAS")
    np.testing.assert_allclose(Dn, -D, rtol=0, atol=1e-15)
    assert np.all(np.abs(D) < 1.0)


# ---- backward epilogues (DRELU_BGRAD, DGELU_BGRAD) -----------------------------------------

def test_gelu_grad_matches_derivative_and_library(oracle):
    from scipy.special import ndtr
    from scipy.stats import norm
    for x in np.linspace(-8, 8, 161):
        h = 1e-5
        num = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
        g = oracle.gelu_grad(x)
        assert abs(g - num) < 1e-8, x
        assert abs(g - (ndtr(x) + x * norm.pdf(x))) < 1e-14, x
    assert oracle.gelu_grad(0.0) == 0.5


def _t64(bits16, dtype="bf16"):
    return torch.from_numpy(_lib_decode(dtype, _bits_np(bits16)))


@pytest.mark.parametrize("layout", ["1N", "M1"])
def test_drelu_bgrad_matches_autograd_of_the_forward_chain(oracle, layout):
    # forward: pre = X.W1 + b1, H = relu(pre), Y = H.W2; backward from dY:
    # dpre = (dY.W2^T) * [pre > 0], db1 = sum of dpre over the broadcast dimension
    t, d, f = 24, 40, 56
    g = torch.Generator().manual_seed(21)
    X = torch.randn(t, d, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(d, f, generator=g) * 0.3).to(torch.bfloat16)
    b1 = torch.randn(t if layout == "M1" else f, generator=g).to(torch.bfloat16)
    W2 = (torch.randn(f, d, generator=g) * 0.3).to(torch.bfloat16)
    dY = torch.randn(t, d, generator=g).to(torch.bfloat16)
    _, pre = oracle.gemm_epi(X, W1, b1, dtype="bf16", epilog="RELU_AUX_BIAS", bias_layout=layout,
                             want_pre=True)
    mask = oracle.aux_pack(pre)
    W2T = W2.t().contiguous()
    D, dbias = oracle.gemm_bwd(dY, W2T, dtype="bf16", kind="DRELU_BGRAD", bias_layout=layout,
                               mask=mask)
    # the same chain with torch autograd in float64
    Xd, W1d, W2d, dYd = _t64(X), _t64(W1), _t64(W2), _t64(dY)
    bd = _t64(b1).requires_grad_(True)
    pre_t = Xd @ W1d + (bd[:, None] if layout == "M1" else bd[None, :])
    pre_t.retain_grad()
    Y = torch.relu(pre_t) @ W2d
    Y.backward(dYd)
    np.testing.assert_allclose(D, pre_t.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dbias, bd.grad.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("layout", ["1N", "M1"])
def test_dgelu_bgrad_matches_autograd_on_the_stored_pre(oracle, layout):
    t, d, f = 20, 32, 48
    g = torch.Generator().manual_seed(22)
    pre16 = (torch.randn(t, f, generator=g) * 2).to(torch.bfloat16)   # the stored pre-activation
    dY = torch.randn(t, d, generator=g).to(torch.bfloat16)
    W2T = (torch.randn(d, f, generator=g) * 0.3).to(torch.bfloat16)
    D, dbias = oracle.gemm_bwd(dY, W2T, dtype="bf16", kind="DGELU_BGRAD", bias_layout=layout,
                               pre=pre16)
    x = _t64(pre16).requires_grad_(True)
    h = torch.nn.functional.gelu(x, approximate="none")
    dH = _t64(dY) @ _t64(W2T)
    h.backward(dH)
    np.testing.assert_allclose(D, x.grad.numpy(), rtol=1e-10, atol=1e-12)
    want_db = x.grad.numpy().sum(axis=1 if layout == "M1" else 0)
    np.testing.assert_allclose(dbias, want_db, rtol=1e-10, atol=1e-10)


def test_drelu_bgrad_brute_force_and_mask_extremes(oracle):
    rng = np.random.default_rng(4)
    for (m, n, k) in [(1, 1, 1), (3, 33, 5), (7, 64, 9), (5, 40, 3)]:
        p = workloads.random_problem(m, n, k, dtype="f16", seed=m * 100 + n)
        Ad, Bd = _lib_decode("f16", _bits_np(p["A"])), _lib_decode("f16", _bits_np(p["B"]))
        bits = rng.integers(0, 2, size=(m, n)).astype(bool)
        padded = np.zeros((m, ((n + 31) // 32) * 32), dtype=bool)
        padded[:, :n] = bits
        mask = np.packbits(padded, axis=1, bitorder="little").view("<u4").reshape(m, -1)
        D, db = oracle.gemm_bwd(p["A"], p["B"], dtype="f16", kind="DRELU_BGRAD", mask=mask)
        want = np.zeros((m, n))
        for i in range(m):
            for j in range(n):
                s = 0.0
                for kk in range(k):
                    s += Ad[i, kk] * Bd[kk, j]
                want[i, j] = s if bits[i, j] else 0.0
        np.testing.assert_allclose(D, want, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(db, want.sum(axis=0), rtol=1e-12, atol=1e-12)
        # all ones: the plain product and its column sums; all zeros: nothing
        ones = np.full_like(mask, 0xFFFFFFFF)
        D1, db1 = oracle.gemm_bwd(p["A"], p["B"], dtype="f16", kind="DRELU_BGRAD", mask=ones)
        np.testing.assert_allclose(D1, Ad @ Bd, rtol=1e-12, atol=1e-12)
        D0, db0 = oracle.gemm_bwd(p["A"], p["B"], dtype="f16", kind="DRELU_BGRAD",
                                  mask=np.zeros_like(mask))
        assert not D0.any() and not db0.any()


# ---- LayerNorm ("Operator fusion in model inference", section 2) ---------------------------

def _ln_inputs(t, d, seed, dtype="bf16", offset=1.5, scale=3.0):
    g = torch.Generator().manual_seed(seed)
    td = workloads.TORCH_DTYPES[dtype]
    X = (torch.randn(t, d, generator=g) * scale + offset).to(td)
    gamma = (1.0 + 0.1 * torch.randn(d, generator=g)).to(td)
    beta = (0.1 * torch.randn(d, generator=g)).to(td)
    R = torch.randn(t, d, generator=g).to(td)
    return X, gamma, beta, R


@pytest.mark.parametrize("d,eps,dtype", [(1, 1e-5, "bf16"), (7, 0.0, "f16"), (64, 1e-5, "bf16"),
                                         (1024, 1e-6, "bf16"), (300, 1e-5, "f16")])
def test_layernorm_matches_torch_float64(oracle, d, eps, dtype):
    X, gamma, beta, R = _ln_inputs(9, d, seed=d, dtype=dtype)
    Xd, gd, bd, Rd = (_t64(x, dtype) for x in (X, gamma, beta, R))
    ref = torch.nn.functional.layer_norm(Xd, (d,), gd, bd, eps).numpy()
    Y, stats = oracle.layernorm(X, gamma, beta, eps=eps, dtype=dtype)
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)
    Yr, _ = oracle.layernorm(X, gamma, beta, eps=eps, dtype=dtype, residual=R)
    np.testing.assert_allclose(Yr, ref + Rd.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(stats[:, 0], Xd.mean(1).numpy(), rtol=1e-13, atol=1e-13)
    var = Xd.var(1, unbiased=False).numpy()
    np.testing.assert_allclose(stats[:, 1], 1.0 / np.sqrt(var + eps), rtol=1e-12)


def test_layernorm_invariants(oracle):
    # integer-valued rows: a shift by an integer and a doubling stay exact in bf16
    g = torch.Generator().manual_seed(3)
    X = torch.randint(-40, 41, (6, 96), generator=g).to(torch.bfloat16)
    ones = torch.ones(96, dtype=torch.bfloat16)
    zeros = torch.zeros(96, dtype=torch.bfloat16)
    Y, stats = oracle.layernorm(X, ones, zeros, eps=1e-5, dtype="bf16")
    Ys, _ = oracle.layernorm(X + 7, ones, zeros, eps=1e-5, dtype="bf16")
    np.testing.assert_allclose(Ys, Y, rtol=0, atol=1e-12)          # shift invariance
    assert np.max(np.abs(Y.mean(1))) < 1e-12                          # centred
    var = _t64(X).var(1, unbiased=False).numpy()
    np.testing.assert_allclose((Y * Y).mean(1), var / (var + 1e-5), rtol=1e-12)
    Y0, _ = oracle.layernorm(X, ones, zeros, eps=0.0, dtype="bf16")
    Y2, _ = oracle.layernorm(X * 2, ones, zeros, eps=0.0, dtype="bf16")
    np.testing.assert_allclose(Y2, Y0, rtol=0, atol=1e-12)          # scale invariance (eps 0)
    # gamma scales, beta shifts, per column
    gam = torch.arange(1, 97).to(torch.bfloat16)
    bet = (torch.arange(96) - 48).to(torch.bfloat16)
    Yg, _ = oracle.layernorm(X, gam, bet, eps=1e-5, dtype="bf16")
    np.testing.assert_allclose(Yg, Y * _t64(gam).numpy() + _t64(bet).numpy(), rtol=1e-13,
                               atol=1e-12)


def test_ln_gemm_gelu_matches_library_chain(oracle):
    from scipy.special import ndtr
    m, k, n = 33, 72, 40
    X, gamma, beta, _ = _ln_inputs(m, k, seed=5)
    g = torch.Generator().manual_seed(6)
    W = (torch.randn(k, n, generator=g) * 0.1).to(torch.bfloat16)
    b = (torch.randn(n, generator=g) * 0.1).to(torch.bfloat16)
    D = oracle.ln_gemm_gelu(X, gamma, beta, W, b, eps=1e-5, dtype="bf16")
    xn = torch.nn.functional.layer_norm(_t64(X), (k,), _t64(gamma), _t64(beta), 1e-5).numpy()
    pre = xn @ _t64(W).numpy() + _t64(b).numpy()
    np.testing.assert_allclose(D, pre * ndtr(pre), rtol=1e-11, atol=1e-12)


def test_ln_ffn_is_the_composition(oracle):
    t, d, f = 17, 48, 64
    X, gamma, beta, R = _ln_inputs(t, d, seed=8)
    g = torch.Generator().manual_seed(9)
    W1 = (torch.randn(d, f, generator=g) * 0.1).to(torch.bfloat16)
    b1 = (torch.randn(f, generator=g) * 0.1).to(torch.bfloat16)
    W2 = (torch.randn(f, d, generator=g) * 0.1).to(torch.bfloat16)
    b2 = (torch.randn(d, generator=g) * 0.1).to(torch.bfloat16)
    H, Hx, Y = oracle.ln_ffn(X, gamma, beta, W1, b1, W2, b2, R, eps=1e-5)
    D = oracle.ln_gemm_gelu(X, gamma, beta, W1, b1, eps=1e-5, dtype="bf16")
    np.testing.assert_array_equal(Hx, D)
    np.testing.assert_array_equal(H, oracle.encode("bf16", D))
    Y2 = oracle.gemm_epi(H, W2, b2, dtype="bf16", epilog="BIAS_RESIDUAL", residual=R)
    np.testing.assert_array_equal(Y, Y2)


# ---- FP8 (E4M3) inputs with per-tensor scales ---------------------------------------------

def test_e4m3_decode_every_pattern_matches_torch(oracle):
    allb = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e4m3(allb)
    want = torch.from_numpy(allb).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))
    # the format's landmarks: largest finite, smallest normal, smallest subnormal, NaN
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and got[0x80] == 0.0


@pytest.mark.parametrize("epilog", ["BIAS", "RELU_BIAS", "GELU_BIAS", "BIAS_RESIDUAL", "NONE",
                                    "TANH_BIAS"])
@pytest.mark.parametrize("layout", ["M1", "1N"])
def test_fp8_gemm_equals_the_bf16_oracle_on_the_same_values(oracle, epilog, layout):
    # every E4M3 value is exact in bfloat16, so with unit scales the FP8 oracle must give
    # the 16-bit oracle's result on A and B = Bt^T carried over exactly
    m, n, k = 9, 40, 48
    p = workloads.random_fp8_problem(m, n, k, bias_layout=layout, seed=len(epilog),
                                     residual=True)
    A16 = p["A"].to(torch.bfloat16)
    B16 = p["Bt"].to(torch.bfloat16).t().contiguous()
    assert torch.equal(A16.double(), p["A"].double()) and torch.equal(B16.t().double(), p["Bt"].double())
    want = oracle.gemm_epi(A16, B16, p["bias"], dtype="bf16", epilog=epilog, bias_layout=layout,
                           residual=p["R"])
    got = oracle.gemm_epi_fp8(p["A"], p["Bt"], p["bias"], scale_a=1.0, scale_b=1.0,
                              epilog=epilog, bias_layout=layout, residual=p["R"])
    assert np.array_equal(got, want)


def test_fp8_gemm_scales_and_library_matmul(oracle):
    m, n, k = 12, 24, 64
    p = workloads.random_fp8_problem(m, n, k, seed=3)
    a = p["A"].double().numpy()
    bt = p["Bt"].double().numpy()
    sa, sb = 0.125, 3.0
    want = sa * sb * (a @ bt.T) + p["bias"].double().numpy()[None, :]
    got = oracle.gemm_epi_fp8(p["A"], p["Bt"], p["bias"], scale_a=sa, scale_b=sb, epilog="BIAS")
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-12)
    # only the product of the scales matters
    got2 = oracle.gemm_epi_fp8(p["A"], p["Bt"], p["bias"], scale_a=sa * 4, scale_b=sb / 4,
                               epilog="BIAS")
    np.testing.assert_array_equal(got2, got)
