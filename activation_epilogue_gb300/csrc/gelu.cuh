// Activation functions of the epilogues, in fp32.
//
// erf-form GELU, x * Phi(x), in the forward epilogues: Phi from a logistic approximation,
//     Phi(x) ~= 1 / (1 + exp(-x (c1 + c3 s + c5 s^2))),   s = min(x^2, 64),
// the form of Bowling et al., "A logistic approximation to the cumulative normal
// distribution" (J. Industrial Engineering and Management, 2009), with an x^5 term and
// coefficients refitted minimax on [0, 8] (fit_gelu_logistic.py beside this file):
// |Phi error| * max(1, |x|) <= 3.1e-5, so |GELU error| <= 3.1e-5 * max(1, |x|), two orders
// below the rounding of a bf16 result and well inside an f16 result's acceptance bound.
// Beyond |x| = 8 the exponent grows linearly in x with the sign it has at 8, so Phi
// saturates; clamping the square (one min) rather than x (two) gives the same bits for
// |x| <= 8.  Per element: two multiplies, one min, two FMAs, one multiply, one ex2, one
// add, one fast divide: under half the instructions of the formula-7.1.26 version below,
// which matters because the epilogue's instruction count is its cost (it also takes issue
// slots from the MMA warp).  The exponent is odd in x, so Phi(-x) = 1 - Phi(x) holds
// exactly and every element takes the same path.
//
// GELU' in the backward epilogue uses formula 7.1.26 of Abramowitz & Stegun, Handbook of
// Mathematical Functions (1964): for z >= 0,
//     erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2) + eps,
//     t = 1 / (1 + p z),  |eps| <= 1.5e-7,
// with p = 0.3275911, a1 = 0.254829592, a2 = -0.284496736, a3 = 1.421413741,
// a4 = -1.453152027, a5 = 1.061405429.  With z = |x| / sqrt(2) the tail
// q = Phi(-|x|) = (a1 t + ... + a5 t^5) exp(-z^2) / 2 comes out directly (no cancellation
// for negative x), and Phi(x) = q for x < 0, 1 - q otherwise.
#pragma once

namespace gemm_epi {

// 2^x with the hardware approximation (relative error about 2^-22).
__device__ __forceinline__ float exp2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float gelu_erf_fast(float x)
{
    // c1, c3, c5 of the fit times -log2(e): exp(-P(x)) = 2^(x * (k1 + k3 x^2 + k5 x^4))
    constexpr float k1 = -2.3014667034f, k3 = -0.10654459149f, k5 = 0.00098442099988f;
    const float x2 = fminf(x * x, 64.0f);
    const float p = fmaf(fmaf(x2, k5, k3), x2, k1);
    return __fdividef(x, 1.0f + exp2_approx(x * p));
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
