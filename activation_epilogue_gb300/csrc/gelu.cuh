// Activation functions of the epilogues, in fp32.
//
// erf-form GELU, x * Phi(x), branch-free.
//
// Phi is evaluated with formula 7.1.26 of Abramowitz & Stegun, Handbook of Mathematical
// Functions (1964): for z >= 0,
//     erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2) + eps,
//     t = 1 / (1 + p z),  |eps| <= 1.5e-7,
// with p = 0.3275911, a1 = 0.254829592, a2 = -0.284496736, a3 = 1.421413741,
// a4 = -1.453152027, a5 = 1.061405429.  With z = |x| / sqrt(2) the tail
// q = Phi(-|x|) = (a1 t + ... + a5 t^5) exp(-z^2) / 2 comes out directly (no cancellation
// for negative x), and Phi(x) = q for x < 0, 1 - q otherwise.  Every element takes the
// same instruction path, so a thread's 32 columns interleave instead of running the
// branches of a library erf one after another.
#pragma once

namespace gemm_epi {

__device__ __forceinline__ float gelu_erf_fast(float x)
{
    const float z = fabsf(x) * 0.70710678118654752f;
    const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
    float poly = fmaf(t, 1.061405429f, -1.453152027f);
    poly = fmaf(poly, t, 1.421413741f);
    poly = fmaf(poly, t, -0.284496736f);
    poly = fmaf(poly, t, 0.254829592f);
    poly *= t;
    const float q = 0.5f * poly * __expf(-z * z);
    return x * (x < 0.0f ? q : 1.0f - q);
}

// GELU'(x) = Phi(x) + x phi(x), phi(x) = exp(-x^2/2) / sqrt(2 pi): the same tail q =
// Phi(-|x|) (formula 7.1.26), and the density from the exponential it already computes.
__device__ __forceinline__ float gelu_grad_fast(float x)
{
    const float z = fabsf(x) * 0.70710678118654752f;
    const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
    float poly = fmaf(t, 1.061405429f, -1.453152027f);
    poly = fmaf(poly, t, 1.421413741f);
    poly = fmaf(poly, t, -0.284496736f);
    poly = fmaf(poly, t, 0.254829592f);
    poly *= t;
    const float e = __expf(-z * z);  // exp(-x^2 / 2)
    const float q = 0.5f * poly * e;
    const float phi_cdf = x < 0.0f ? q : 1.0f - q;
    return fmaf(x * e, 0.39894228040143268f, phi_cdf);
}

// tanh with the hardware approximation (relative error below 2^-10.9), well inside the
// 16-bit output rounding of a bf16 result and the acceptance bound of an fp16 one.
__device__ __forceinline__ float tanh_fast(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace gemm_epi
