// stress.cuh -- the MLS-MPM elastic stress term of P2G and the deformation
// gradient update of G2P.
//
// Implementation guide ("Implementation -- GPU Optimization & Reference
// Codebases"), section 3.1, Part 2: the Neo-Hookean model with Lame
// constants mu and lambda, J = det F, P = mu (F - F^-T) + lambda ln(J) F^-T,
// sigma = P F^T / J.  In MLS-MPM the stress rides in the same affine scatter
// as APIC's C: a node gains the momentum -dt V sigma D^-1 w (x_i - x_p), with
// V = V0 J and D^-1 = 4/dx^2 for the quadratic B-spline (section 3.3.2,
// "D (= B*4)").  Divided by the particle mass this is a change of C:
//     C' = C - kappa tau,   kappa = dt V0 (4/dx^2) / m,   tau = J sigma = P F^T,
// and P F^T = mu (F F^T - I) + lambda ln(J) I since F^-T F^T = I.  So the
// scatter loop is the APIC one; only the matrix it reads changes.  G2P then
// advances F <- (I + D) F with D = dt C' (section 3.3.2, velocity form).
//
// Every step is one fp32 operation with round-to-nearest-even in a fixed
// order, so the fixed-point shares are reproducible bit for bit:
//   J (3D) = (F00 (F11 F22 - F12 F21) - F01 (F10 F22 - F12 F20)) + F02 (F10 F21 - F11 F20)
//   b_kl   = (F_k0 F_l0 + F_k1 F_l1) + F_k2 F_l2
//   tau_kl = mu b_kl (k != l),  tau_kk = mu (b_kk - 1) + lambda ln J
//   C'_kl  = C_kl - kappa tau_kl,  kappa = ((dt V0) c4s) / m,  c4s = (4 inv_dx) inv_dx
// ln J is not the CUDA math library's: it is the series below, written out
// here so that it rounds the same way on every device and host.
#pragma once

#include "common.cuh"

namespace mpm {

// Material constants and the step's scale factors of the stress term.
struct StressP {
    float mu, lam;  // Lame constants
    float dt;       // time step
    float c4s;      // (4 * inv_dx) * inv_dx
};

// J in the domain of the logarithm: a positive, normal, finite fp32 number
// (false for zero, negatives, subnormals, infinities and NaN).
__device__ __forceinline__ bool log_domain(float J) { return J >= 0x1p-126f && J <= 0x1.fffffep+127f; }

// Natural logarithm of J (in log_domain) from the inverse hyperbolic tangent
// series: J = 2^e r with r in [1/sqrt2, sqrt2), s = (r - 1) / (r + 1),
// ln r = 2 atanh(s) = 2 (s + s^3/3 + s^5/5 + s^7/7 + s^9/9 + ...); |s| <= 0.1716,
// so the terms after s^9/9 are below 2e-9 relative.  ln 2 is split into
// 45426/65536 (exact times any exponent of fp32) plus the fp32 remainder.
__device__ __forceinline__ float series_log(float J) {
    constexpr float kLn2Hi = 0x1.62e4p-1f;     // 45426 / 65536
    constexpr float kLn2Lo = 0x1.7f7d1cp-20f;  // ln 2 - kLn2Hi
    constexpr float kSqrt2 = 0x1.6a09e6p+0f;
    constexpr float k3 = 0x1.555556p-2f, k5 = 0x1.99999ap-3f, k7 = 0x1.24924ap-3f, k9 = 0x1.c71c72p-4f;
    const uint32_t u = __float_as_uint(J);
    int e = (int)(u >> 23) - 127;
    float r = __uint_as_float((u & 0x007FFFFFu) | 0x3F800000u);
    if (r > kSqrt2) {
        r = __fmul_rn(r, 0.5f);
        e += 1;
    }
    const float s = __fdiv_rn(__fsub_rn(r, 1.0f), __fadd_rn(r, 1.0f));
    const float z = __fmul_rn(s, s);
    float p = __fadd_rn(__fmul_rn(k9, z), k7);
    p = __fadd_rn(__fmul_rn(p, z), k5);
    p = __fadd_rn(__fmul_rn(p, z), k3);
    const float lr = __fmul_rn(2.0f, __fadd_rn(s, __fmul_rn(s, __fmul_rn(z, p))));
    const float fe = (float)e;
    return __fadd_rn(__fmul_rn(fe, kLn2Hi), __fadd_rn(__fmul_rn(fe, kLn2Lo), lr));
}

// C <- C - kappa tau for one particle (F and C row-major dim x dim).  Returns
// false, leaving C as it is, when det F is outside log_domain.
template <int DIM>
__device__ __forceinline__ bool fold_stress(const StressP &sp, const float (&F)[DIM * DIM], float vol, float m,
                                            float (&C)[DIM * DIM]) {
    float J;
    if constexpr (DIM == 3) {
        const float c0 = __fsub_rn(__fmul_rn(F[4], F[8]), __fmul_rn(F[5], F[7]));
        const float c1 = __fsub_rn(__fmul_rn(F[3], F[8]), __fmul_rn(F[5], F[6]));
        const float c2 = __fsub_rn(__fmul_rn(F[3], F[7]), __fmul_rn(F[4], F[6]));
        J = __fadd_rn(__fsub_rn(__fmul_rn(F[0], c0), __fmul_rn(F[1], c1)), __fmul_rn(F[2], c2));
    } else {
        J = __fsub_rn(__fmul_rn(F[0], F[3]), __fmul_rn(F[1], F[2]));
    }
    if (!log_domain(J)) return false;
    const float lj = __fmul_rn(sp.lam, series_log(J));
    const float kappa = __fdiv_rn(__fmul_rn(__fmul_rn(sp.dt, vol), sp.c4s), m);
#pragma unroll
    for (int k = 0; k < DIM; ++k)
#pragma unroll
        for (int l = 0; l < DIM; ++l) {
            float b = __fadd_rn(__fmul_rn(F[k * DIM + 0], F[l * DIM + 0]), __fmul_rn(F[k * DIM + 1], F[l * DIM + 1]));
            if constexpr (DIM == 3) b = __fadd_rn(b, __fmul_rn(F[k * DIM + 2], F[l * DIM + 2]));
            const float tau = k == l ? __fadd_rn(__fmul_rn(sp.mu, __fsub_rn(b, 1.0f)), lj) : __fmul_rn(sp.mu, b);
            C[k * DIM + l] = __fsub_rn(C[k * DIM + l], __fmul_rn(kappa, tau));
        }
    return true;
}

// F' = (I + D) F with D = dt C (C the particle's new affine matrix):
// F'_kl = fma(D_k2, F_2l, fma(D_k1, F_1l, fma(D_k0, F_0l, F_kl))).
template <int DIM>
__device__ __forceinline__ void advance_F(float dt, const float (&C)[DIM * DIM], const float (&F)[DIM * DIM],
                                          float (&Fn)[DIM * DIM]) {
    float D[DIM * DIM];
#pragma unroll
    for (int j = 0; j < DIM * DIM; ++j) D[j] = __fmul_rn(dt, C[j]);
#pragma unroll
    for (int k = 0; k < DIM; ++k)
#pragma unroll
        for (int l = 0; l < DIM; ++l) {
            float t = __fmaf_rn(D[k * DIM + 0], F[0 * DIM + l], F[k * DIM + l]);
            t = __fmaf_rn(D[k * DIM + 1], F[1 * DIM + l], t);
            if constexpr (DIM == 3) t = __fmaf_rn(D[k * DIM + 2], F[2 * DIM + l], t);
            Fn[k * DIM + l] = t;
        }
}

}  // namespace mpm
