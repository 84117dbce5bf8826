"""Plant mistakes in a copy of the oracle and check that the pins catch every one.

Each mutant is the oracle's C source with one plausible slip written in; it is compiled to
a temporary library and the pin suite is run against it in a subprocess.  The pin suite
must fail for every mutant (and pass for the unmodified source, which the rest of the CPU
suite already checks).
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gemm_epi_oracle.c")

MUTANTS = {
    "bias dropped": ("const double p = acc[c] + beta;", "const double p = acc[c];"),
    "bias axis swapped": ("bias_layout == OR_BIAS_M1 ? bias[i] : bias[j]",
                          "bias_layout != OR_BIAS_M1 && i < n ? bias[i] : bias[j % (n ? n : 1)]"),
    "gelu tanh form": ("return x * 0.5 * erfc(-x / sqrt(2.0));",
                       "return 0.5 * x * (1.0 + tanh(0.7978845608028654 * (x + 0.044715 * x * x * x)));"),
    "gelu sign": ("return x * 0.5 * erfc(-x / sqrt(2.0));", "return x * 0.5 * erfc(x / sqrt(2.0));"),
    "relu negative zero": ("return pre > 0.0 ? pre : 0.0;", "return pre > 0.0 ? pre : -0.0;"),
    "aux bit order": ("words[r * ldw + j / 32] |= 1u << (j % 32);",
                      "words[r * ldw + j / 32] |= 1u << (31 - j % 32);"),
    "aux not strict": ("if (pre[r * n + j] > 0.0)", "if (pre[r * n + j] >= 0.0)"),
    "bf16 exponent bias": ("v = ldexp((double)(frac + 128), expo - 134);",
                           "v = ldexp((double)(frac + 128), expo - 133);"),
    "encode truncates": ("double q = nearbyint(scaled);", "double q = floor(scaled);"),
    "tanh sign": ("return tanh(pre);", "return tanh(-pre);"),
    "gelu grad drops density term": ("return 0.5 * erfc(-x / sqrt(2.0)) + x * phi;",
                                     "return 0.5 * erfc(-x / sqrt(2.0));"),
    "dbias sums the wrong axis": ("dbias[bias_layout == OR_BIAS_M1 ? i : j] += D[i * n + j];",
                                  "dbias[bias_layout == OR_BIAS_M1 ? j % nb : i % nb] += D[i * n + j];"),
    "drelu mask bit order": ("g = (mask[i * ldw + j / 32] >> (j % 32)) & 1u ? 1.0 : 0.0;",
                             "g = (mask[i * ldw + j / 32] >> (31 - j % 32)) & 1u ? 1.0 : 0.0;"),
    "residual dropped": ("d = p + decode(dtype, residual[i * n + j]);", "d = p;"),
    "e4m3 exponent bias": ("v = ldexp((double)(frac + 8), expo - 10);",
                           "v = ldexp((double)(frac + 8), expo - 11);"),
    "fp8 B not transposed": ("acc += oracle_decode_e4m3(A[i * k + q]) * Bd[j * k + q];",
                             "acc += oracle_decode_e4m3(A[i * k + q]) * Bd[(q * n + j) % (n * k)];"),
    "fp8 second scale dropped": ("const double p = sa * sb * acc + beta;",
                                 "const double p = sa * acc + beta;"),
    "layernorm eps dropped": ("const double rstd = 1.0 / sqrt(var + eps);",
                              "const double rstd = 1.0 / sqrt(var);"),
    "layernorm unbiased variance": ("const double var = d > 0 ? ss / (double)d : 0.0;",
                                    "const double var = d > 1 ? ss / (double)(d - 1) : 0.0;"),
    "layernorm gamma and beta swapped": ("* rstd * decode(dtype, gamma[j]) +\n                       decode(dtype, beta[j]);",
                                         "* rstd * decode(dtype, beta[j]) +\n                       decode(dtype, gamma[j]);"),
    "layernorm gemm drops last term": ("for (int64_t q = 0; q < k; ++q) {",
                                       "for (int64_t q = 0; q + 1 < k; ++q) {"),
    "layernorm residual dropped": ("                y += decode(dtype, residual[i * d + j]);",
                                   "                y += 0.0;"),
    "k loop drops last term": ("for (int64_t kk = 0; kk < k; ++kk) {\n                const double a",
                               "for (int64_t kk = 0; kk + 1 < k; ++kk) {\n                const double a"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
                    "-shared", "-o", str(lib), str(mutant_c), "-lm"], check=True)
    env = dict(os.environ, GEMM_EPI_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name!r}:\n{r.stdout[-2000:]}"
