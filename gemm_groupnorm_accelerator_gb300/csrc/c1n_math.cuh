// Device math shared by the tensor-core kernel and the CUDA-core passes.
#pragma once

namespace c1n {

// Exact (erf) GELU, 0.5 z (1 + erf(z / sqrt 2)), with erf from the rational-exponential
// approximation 7.1.26 of Abramowitz & Stegun's Handbook of Mathematical Functions (Hastings):
// erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-x^2), t = 1 / (1 + p x), x >= 0, with
// |error| <= 1.5e-7; odd symmetry for x < 0. The reciprocal and exp2 use the hardware
// approximations (a few ulp), which keeps the GELU error below 1e-6 * |z| -- far inside the fp32
// and bf16 output tolerances -- at about a dozen instructions.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float exp2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// Written as GELU(z) = z * Phi(z) with the normal CDF Phi(z) = 1 - Q (z >= 0) or Q (z < 0), where
// Q = erfc(|z| / sqrt 2) / 2 is the approximation's tail term (its coefficients halved and
// 1/sqrt(2) folded into p; exp(-z^2/2) as exp2). Both cases are max(z, 0) - |z| * Q.
__device__ __forceinline__ float gelu_erf(float z) {
    const float az = fabsf(z);
    const float t = rcp_approx(fmaf(0.3275911f * 0.70710678118654752f, az, 1.0f));
    const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 0.5f * 1.061405429f, 0.5f * -1.453152027f),
                                                0.5f * 1.421413741f), 0.5f * -0.284496736f), 0.5f * 0.254829592f);
    const float q = poly * exp2_approx(z * z * (-0.5f * 1.4426950408889634f));
    return fmaf(-az, q, fmaxf(z, 0.f));
}

}  // namespace c1n
