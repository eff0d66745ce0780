// range.cuh -- the per-particle range behind the P2G bound, and the exact
// rounding of a product for shares of any size.
//
// "particle to grid transfer in checked integer arithmetic", the program: the
// bounds line runs before any particle is scattered and, when it fails,
// nothing is.  A particle's quantity is spread over a quadratic stencil with
// an affine term, so its range is
//   r_k = |v_k| + h*((|C_k0| + |C_k1|) + |C_k2|),  h = 1.5*dx,
//   R_p = max(|m| * max(1, r_0, .., r_dim-1), |q|)   (q: rest volume in cells),
// in fp32 in this order, and the absolute values of one particle's shares of
// any channel sum to at most S*R_p*(1 + 2^-10) + 28.  Every value here is
// non-negative (or a NaN without sign bit, which is how the GPU makes NaN),
// so the maximum of such values is the maximum of their bit patterns as
// unsigned integers, with NaN above every number: a NaN anywhere makes the
// maximum NaN and fails the bound.
#pragma once

#include "common.cuh"

namespace mpm {

__device__ __forceinline__ uint32_t max_bits(uint32_t a, float b) { return max(a, __float_as_uint(b)); }

// max(1, r_0, .., r_dim-1) as fp32 bits; C is the matrix the scatter uses.
template <int DIM>
__device__ __forceinline__ uint32_t range_r_bits(const float (&v)[DIM], const float (&C)[DIM * DIM], float h) {
    uint32_t r = __float_as_uint(1.0f);
#pragma unroll
    for (int k = 0; k < DIM; ++k) {
        float sc = __fadd_rn(fabsf(C[k * DIM + 0]), fabsf(C[k * DIM + 1]));
        if (DIM == 3) sc = __fadd_rn(sc, fabsf(C[k * DIM + 2]));
        r = max_bits(r, __fadd_rn(fabsf(v[k]), __fmul_rn(h, sc)));
    }
    return r;
}

// R_p as fp32 bits from max(1, r_k) (bits), m and, with the volume channel, q.
template <bool VC>
__device__ __forceinline__ uint32_t particle_range_bits(uint32_t r_bits, float m, float q) {
    uint32_t R = __float_as_uint(__fmul_rn(fabsf(m), __uint_as_float(r_bits)));
    if (isnan(m)) R = 0x7FFFFFFFu;
    if constexpr (VC) R = max_bits(R, fabsf(q));
    return R;
}

// Warp maximum of bit patterns, added to a status word by lane 0.
__device__ __forceinline__ void warp_max_to(uint32_t bits, uint32_t *word) {
    bits = __reduce_max_sync(0xFFFFFFFFu, bits);
    if (lane_id() == 0 && bits) atomicMax(word, bits);
}

// rint(a*b) of the exact product, ties to even: the 24-bit significands
// multiplied as integers (48 bits, exact), then shifted to the binary point
// with round-half-even.  |a*b| must stay below 2^62 (the bound sees to it).
__device__ __forceinline__ long long rint_prod64(float a, float b) {
    const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
    const uint32_t ea = (ua >> 23) & 0xFFu, eb = (ub >> 23) & 0xFFu;
    const uint32_t ma = (ua & 0x7FFFFFu) | (ea ? 0x800000u : 0u);
    const uint32_t mb = (ub & 0x7FFFFFu) | (eb ? 0x800000u : 0u);
    // a = ma * 2^(e - 150) for a normal number, (ua & 0x7FFFFF) * 2^-149 for a subnormal one
    const int sh = (int)max(ea, 1u) + (int)max(eb, 1u) - 300;
    const unsigned long long prod = (unsigned long long)ma * (unsigned long long)mb;  // < 2^48
    unsigned long long mag;
    if (sh >= 0) {
        mag = prod << sh;
    } else if (sh > -50) {
        const int k = -sh;
        const unsigned long long q = prod >> k;
        const unsigned long long rem = prod & ((1ull << k) - 1ull);
        const unsigned long long half = 1ull << (k - 1);
        mag = q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
    } else {
        mag = 0;  // prod < 2^48 <= 2^(k-2): the product is below 1/4
    }
    return ((ua ^ ub) >> 31) ? -(long long)mag : (long long)mag;
}

}  // namespace mpm
