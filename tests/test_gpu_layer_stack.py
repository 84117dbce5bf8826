"""A stack of FFN layers at small batch, every GEMM launched as a programmatic dependent of
the one before it on the stream:

    H_l = GELU(X_l . W1_l + b1_l),    X_{l+1} = H_l . W2_l + b2_l + X_l

(the operator-fusion page's FFN chain, section 1 flowchart, repeated as in a decoder; the
small-batch inference shapes of the cuBLASLt page's closing section).  Each GEMM's A is the
previous GEMM's output, so the kernels must not copy A before their predecessor has
finished; with B_READY they copy the weight B before that.  Every intermediate buffer starts
as NaN and every layer's outputs are checked against the oracle on the GPU's own inputs of
that layer: a copy of A taken too early shows up as NaN or as stale values.
"""
import pytest
import torch

import oracle
from activation_epilogue_gb300 import gemm_epi, workloads
from parity_helpers import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from activation_epilogue_gb300 import build
    build.build()
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def run_stack(t, d, f, layers, options, seed, dtype="bf16", graph=False):
    """Queue the stack on the current stream (or capture it in a CUDA graph and replay it
    twice); returns the CPU inputs, the per-layer outputs and both plans' descriptions."""
    dev = torch.device("cuda")
    td = workloads.TORCH_DTYPES[dtype]
    inp = workloads.layer_stack_inputs(t, d, f, layers, dtype=dtype, seed=seed)
    X = [inp["X"].to(dev)] + [torch.full((t, d), float("nan"), dtype=td, device=dev)
                              for _ in range(layers)]
    H = [torch.full((t, f), float("nan"), dtype=td, device=dev) for _ in range(layers)]
    W = [[w.to(dev) for w in layer] for layer in inp["layers"]]
    with gemm_epi.Plan(t, f, d, dtype, "GELU_BIAS", "1N", **options) as up, \
            gemm_epi.Plan(t, d, f, dtype, "BIAS_RESIDUAL", "1N", **options) as down:
        def queue():
            for l in range(layers):
                W1, b1, W2, b2 = W[l]
                up.execute(X[l], W1, b1, H[l])
                down.execute(H[l], W2, b2, X[l + 1], residual=X[l])

        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                queue()  # (warm-up: tensor maps encoded outside the capture)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            for b in X[1:] + H:
                b.fill_(float("nan"))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                queue()
            g.replay()
            g.replay()
        else:
            queue()
        torch.cuda.synchronize()
        assert up.sync_status() == 0 and down.sync_status() == 0
        descs = (up.describe(), down.describe())
    return inp, [x.cpu() for x in X], [h.cpu() for h in H], descs


def check_stack(inp, X, H, dtype, descs):
    for l, (W1, b1, W2, b2) in enumerate(inp["layers"]):
        want_h = oracle.gemm_epi(X[l], W1, b1, dtype=dtype, epilog="GELU_BIAS")
        err = rel_err(H[l], want_h)
        assert err <= TOL[dtype], f"layer {l} H: rel err {err:.3e} ({descs[0]})"
        want_x = oracle.gemm_epi(H[l], W2, b2, dtype=dtype, epilog="BIAS_RESIDUAL",
                                 residual=X[l])
        err = rel_err(X[l + 1], want_x)
        assert err <= TOL[dtype], f"layer {l} X: rel err {err:.3e} ({descs[1]})"


# (t, d, f, layers, options, the kernel the up projection must run)
CASES = [
    (16, 768, 3072, 3, {}, "small-m"),
    (16, 768, 3072, 3, {"B_READY": 1}, "small-m"),
    (5, 768, 3072, 2, {"B_READY": 1}, "small-m"),
    (64, 256, 1024, 3, {"B_READY": 1}, "small-m"),
    (40, 264, 520, 2, {"B_READY": 1, "VARIANT": 2}, "swapped"),
    (200, 256, 512, 2, {"B_READY": 1}, "swapped"),
    (130, 264, 256, 2, {"B_READY": 1, "VARIANT": 1}, "row-tile"),
    (130, 256, 512, 2, {"B_READY": 1, "VARIANT": 1, "SPLIT_K": 2, "SPLIT_MODE": 3},
     "row-tile"),
    (16, 768, 3072, 2, {"B_READY": 1, "PDL": 0}, "small-m"),
]


@pytest.mark.parametrize("t,d,f,layers,options,kernel", CASES)
def test_layer_stack_matches_oracle(t, d, f, layers, options, kernel):
    inp, X, H, descs = run_stack(t, d, f, layers, options, seed=7000 + t + layers)
    assert f"variant={kernel}" in descs[0], descs
    check_stack(inp, X, H, "bf16", descs)


def _random_stack_case(i):
    import random
    r = random.Random(9100 + i)
    t = r.choice([1, 3, 8, 16, 17, 32, 40, 64, 65, 100, 130, 200, 256, 300])
    d = 8 * r.randint(2, 64)
    f = 8 * r.randint(2, 200)
    options = {"B_READY": r.choice([0, 1, 1])}
    if r.random() < 0.3:
        options["PDL"] = r.choice([0, 1])
    if t <= 64 and r.random() < 0.3:
        options["VARIANT"] = 2
    return t, d, f, options


@pytest.mark.parametrize("i", range(24))
def test_random_layer_stacks(i):
    # seeded random shapes (ragged t, d and f) and launch options, three layers each
    t, d, f, options = _random_stack_case(i)
    inp, X, H, descs = run_stack(t, d, f, 3, options, seed=9200 + i)
    check_stack(inp, X, H, "bf16", descs)


@pytest.mark.parametrize("options", [{}, {"B_READY": 1}])
def test_layer_stack_in_a_graph(options):
    inp, X, H, descs = run_stack(16, 768, 3072, 3, options, seed=7101, graph=True)
    check_stack(inp, X, H, "bf16", descs)


def test_layer_stack_f16():
    inp, X, H, descs = run_stack(24, 256, 768, 2, {"B_READY": 1}, seed=7102, dtype="f16")
    check_stack(inp, X, H, "f16", descs)


def test_b_ready_repeats_bit_identical():
    a = run_stack(16, 768, 3072, 2, {"B_READY": 1}, seed=7103)
    b = run_stack(16, 768, 3072, 2, {}, seed=7103)
    for x, y in zip(a[1] + a[2], b[1] + b[2]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("t", [1, 16])
def test_down_projection_plan_widens_the_row_tile(t):
    # t x 768 x 3072: no 16-row slab of the K loop fits shared memory in the 4 slices 16
    # rows allow, so the small-m kernel runs 32-row tiles in 8 slices (6 clusters of 8)
    with gemm_epi.Plan(t, 768, 3072, "bf16", "BIAS_RESIDUAL", "1N") as plan:
        d = plan.describe()
    assert "variant=small-m" in d and "tile=128x32" in d and "split_k=8(cluster)" in d, d
    inp, X, H, descs = run_stack(t, 768, 3072, 2, {"B_READY": 1}, seed=7200 + t)
    assert "tile=128x32" in descs[1], descs
    check_stack(inp, X, H, "bf16", descs)


@pytest.mark.parametrize("t,d,f,b_ready", [(16, 768, 3072, 1), (16, 768, 3072, 0), (40, 264, 520, 1)])
def test_ffn_calls_back_to_back(t, d, f, b_ready):
    # the FFN entry point layer after layer (R = the layer's input), with the weights
    # promised ready: each layer's Y against the oracle's FFN on that layer's GPU input
    dev = torch.device("cuda")
    layers = 3
    inp = workloads.layer_stack_inputs(t, d, f, layers, seed=7300 + t + b_ready)
    X = [inp["X"].to(dev)] + [torch.full((t, d), float("nan"), dtype=torch.bfloat16,
                                         device=dev) for _ in range(layers)]
    W = [[w.to(dev) for w in layer] for layer in inp["layers"]]
    with gemm_epi.FfnPlan(t, d, f, b_ready=b_ready) as plan:
        for l in range(layers):
            W1, b1, W2, b2 = W[l]
            plan.execute(X[l], W1, b1, W2, b2, X[l], X[l + 1])
        torch.cuda.synchronize()
        assert plan.sync_status() == 0
        desc = plan.describe()
    Xc = [x.cpu() for x in X]
    for l, (W1, b1, W2, b2) in enumerate(inp["layers"]):
        _, _, want = oracle.ffn(Xc[l], W1, b1, W2, b2, Xc[l], dtype="bf16")
        err = rel_err(Xc[l + 1], want)
        assert err <= TOL["bf16"], f"layer {l}: rel err {err:.3e} ({desc})"


def test_b_ready_option_values():
    with gemm_epi.Plan(16, 256, 128, "bf16", "BIAS", "1N") as plan:
        plan.set_option("B_READY", 1)
        plan.set_option("B_READY", 0)
        with pytest.raises(gemm_epi.GemmEpiError):
            plan.set_option("B_READY", 2)
    with gemm_epi.FfnPlan(16, 256, 512) as plan:
        gemm_epi.gemm_epi_ffn_set_option(plan.handle, "B_READY", 1)
        with pytest.raises(gemm_epi.GemmEpiError):
            gemm_epi.gemm_epi_ffn_set_option(plan.handle, "B_READY", 2)
