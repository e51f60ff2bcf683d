// Device math shared by the tensor-core kernel and the CUDA-core passes.
#pragma once

#include <cstdint>

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

// Packed pairs of fp32 for Blackwell's paired fp32 add / sub / mul / fma (one instruction for two
// lanes of arithmetic, each rounded as its scalar form): lo in the low word.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t p, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ float f2_hsum(uint64_t p) {
    float lo, hi;
    f2_unpack(p, lo, hi);
    return lo + hi;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// gelu_erf on a pair, step for step (the same roundings): -|z| by setting the sign bits, the
// polynomial and the products in paired arithmetic, the reciprocal and exp2 per half.
__device__ __forceinline__ uint64_t gelu_erf2(uint64_t z) {
    const uint64_t nz = z | 0x8000000080000000ull;  // -|z|
    const uint64_t u = f2_fma(nz, f2_pack(-0.3275911f * 0.70710678118654752f, -0.3275911f * 0.70710678118654752f),
                              f2_pack(1.0f, 1.0f));
    float ul, uh;
    f2_unpack(u, ul, uh);
    const uint64_t t = f2_pack(rcp_approx(ul), rcp_approx(uh));
    uint64_t p = f2_fma(t, f2_pack(0.5f * 1.061405429f, 0.5f * 1.061405429f),
                        f2_pack(0.5f * -1.453152027f, 0.5f * -1.453152027f));
    p = f2_fma(t, p, f2_pack(0.5f * 1.421413741f, 0.5f * 1.421413741f));
    p = f2_fma(t, p, f2_pack(0.5f * -0.284496736f, 0.5f * -0.284496736f));
    p = f2_fma(t, p, f2_pack(0.5f * 0.254829592f, 0.5f * 0.254829592f));
    p = f2_mul(t, p);
    const uint64_t e = f2_mul(f2_mul(z, z), f2_pack(-0.5f * 1.4426950408889634f, -0.5f * 1.4426950408889634f));
    float el, eh;
    f2_unpack(e, el, eh);
    const uint64_t q = f2_mul(p, f2_pack(exp2_approx(el), exp2_approx(eh)));
    float zl, zh;
    f2_unpack(z, zl, zh);
    return f2_fma(nz, q, f2_pack(fmaxf(zl, 0.f), fmaxf(zh, 0.f)));
}

}  // namespace c1n
