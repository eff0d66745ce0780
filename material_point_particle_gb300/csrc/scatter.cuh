// scatter.cuh -- one particle's fixed-point P2G shares into a shared-memory
// accumulator (used by the P2G kernels and by the fused gather-scatter step).
//
// Shares follow "particle to grid transfer in checked integer arithmetic":
// split rather than weight, so each particle's shares sum exactly to its
// quantity and the grid is the same in every order.  The momentum is the
// APIC/MLS affine momentum of the implementation guide, section 3.1; elastic
// particles scatter the stress-folded affine matrix (stress.cuh).
#pragma once

#include "common.cuh"
#include "range.cuh"
#include "stress.cuh"

namespace mpm {

// The stencil base cell b and fraction f of position x, true when the
// particle is in the domain and b lies in the box [o, o + TB) per axis.
template <int DIM, int TB>
__device__ __forceinline__ bool in_box_x(const GridP &g, const float *x, const int o[3], int b[3], float f[3]) {
    bool ok = true;
#pragma unroll
    for (int l = 0; l < DIM; ++l) {
        ok = ok && base_frac(x[l], g.inv_dx, g.n[l], b[l], f[l]);
        ok = ok && b[l] >= o[l] && b[l] < o[l] + TB;
    }
    return ok;
}

// Share encode: rint(a * b) for |a*b| < 2^22, exact product rounded once (RNE).
__device__ __forceinline__ int32_t rint_mul(float a, float b) {
    return __float_as_int(__fmaf_rn(a, b, kMagic)) - kMagicBits;
}
__device__ __forceinline__ int32_t rint_f(float a) { return __float_as_int(__fadd_rn(a, kMagic)) - kMagicBits; }

// Where a share goes: add<C, A>(v) adds share v of channel C to stencil node
// A (A = a0*9 + a1*3 + a2 in 3D, a0*3 + a1 in 2D; a0 along x).
//
// SharedAdd: a shared-memory accumulator of layout Hl; `base` is the shared
// address of the stencil's first node (constant offsets from one base).
template <typename Hl>
struct SharedAdd {
    uint32_t base;
    template <int C, int A>
    __device__ __forceinline__ void add(int32_t v) const {
        red_shared_add<4 * (Hl::off(A) + C * Hl::SIZE)>(base, v);
    }
};

// GlobalAdd: the int64 grid itself, node0 = the stencil's first node.
template <int DIM>
struct GlobalAdd {
    long long *acc;
    int64_t nodes, n0, n01, node0;
    template <int C, int A>
    __device__ __forceinline__ void add(int32_t v) const {
        constexpr int a0 = DIM == 3 ? A / 9 : A / 3;
        constexpr int a1 = DIM == 3 ? (A / 3) % 3 : A % 3;
        constexpr int a2 = DIM == 3 ? A % 3 : 0;
        atomicAdd(reinterpret_cast<unsigned long long *>(acc + C * nodes + node0 + a0 + a1 * n0 + a2 * n01),
                  (unsigned long long)(long long)v);
    }
};

// The particle's affine matrix as P2G scatters it: C, and for elastic
// particles C minus the stress term (stress.cuh); counts the elastic
// particles whose det F leaves them unstressed.
template <int DIM, bool EL, bool VC, typename Rec>
__device__ __forceinline__ void load_affine(const Rec &rec, const StressP &sp, float (&C)[DIM * DIM],
                                            uint32_t &degenerate) {
    using Fl = P2GFields<DIM, EL, VC>;
#pragma unroll
    for (int j = 0; j < DIM * DIM; ++j) C[j] = rec(2 * DIM + j);
    if constexpr (EL) {
        float F[DIM * DIM];
#pragma unroll
        for (int j = 0; j < DIM * DIM; ++j) F[j] = rec(Fl::BASE + j);
        if (!fold_stress<DIM>(sp, F, rec(Fl::VOLF), rec(2 * DIM + DIM * DIM), C)) ++degenerate;
    }
}

// True when every share of the particle stays below 2^22 in magnitude:
// wmax*|Mt| and wmax*|Mt|*(|v_k| + 1.5 dx sum_l |C_kl|) (and wmax*|Vt|) at most
// 2^22 - 4096, which also keeps the centre's remainder below 2^22.
template <int DIM, bool VC>
__device__ __forceinline__ bool shares_fit_22(const GridP &g, const float (&v)[DIM], const float (&C)[DIM * DIM],
                                              float Mt, float Vt) {
    const float h = __fmul_rn(1.5f, g.dx);
    const float aM = fabsf(Mt);
    bool ok = __fmul_rn(g.wmax, aM) <= kShareLimit;
    if constexpr (VC) ok = ok && __fmul_rn(g.wmax, fabsf(Vt)) <= kShareLimit;
#pragma unroll
    for (int k = 0; k < DIM; ++k) {
        float sc = __fadd_rn(fabsf(C[k * DIM + 0]), fabsf(C[k * DIM + 1]));
        if (DIM == 3) sc = __fadd_rn(sc, fabsf(C[k * DIM + 2]));
        const float R = __fmul_rn(aM, __fadd_rn(fabsf(v[k]), __fmul_rn(h, sc)));
        ok = ok && (__fmul_rn(g.wmax, R) <= kShareLimit);
    }
    return ok;
}

// One particle's fixed-point shares below 2^22, handed to `ad` as they are
// formed (the arithmetic the oracle states; one fp32 fma against 1.5*2^23
// leaves rint of the exact product in the low mantissa bits).  The caller
// guarantees the range (the P2G bound), or asks for the test (CHECK: the
// fused kernels, whose new state is formed in the same kernel); then the
// function returns false and adds nothing for a particle out of that range.
// f: the fractions of its stencil base cell.
// rec(f) reads field f of the particle (P2GFields: x[dim], v[dim],
// C[dim*dim], m, then F[dim*dim] for elastic particles, and vol).  With the
// volume channel (VC) the rest volume in cells, Vt = (vol * inv_dx^dim) * S,
// is split over the stencil as the mass is, into channel dim + 1.
template <int DIM, bool EL, bool VC, bool CHECK, typename Rec, typename Add>
__device__ __forceinline__ bool scatter_shares(const GridP &g, const Rec &rec, const float (&f)[3], const Add &ad,
                                               const StressP &sp, uint32_t &degenerate) {
    using Fl = P2GFields<DIM, EL, VC>;
    using St = Stencil<DIM>;
    float v[DIM], C[DIM * DIM];
#pragma unroll
    for (int k = 0; k < DIM; ++k) v[k] = rec(DIM + k);
    load_affine<DIM, EL, VC>(rec, sp, C, degenerate);
    const float Mt = __fmul_rn(rec(2 * DIM + DIM * DIM), g.S);
    [[maybe_unused]] float Vt = 0.f;
    if constexpr (VC) Vt = __fmul_rn(__fmul_rn(rec(Fl::VOLF), g.vcell), g.S);
    if constexpr (CHECK)
        if (!shares_fit_22<DIM, VC>(g, v, C, Mt, Vt)) return false;
    float w[3][3], dd[3][3];
#pragma unroll
    for (int l = 0; l < DIM; ++l) {
        quad_weights(f[l], w[l]);
#pragma unroll
        for (int a = 0; a < 3; ++a) dd[l][a] = __fmul_rn(__fsub_rn((float)a, f[l]), g.dx);
    }
    int32_t rest[St::NC + 1];
    rest[0] = __float2int_rn(Mt);
    rest[St::NC] = VC ? __float2int_rn(Vt) : 0;
#pragma unroll
    for (int k = 0; k < DIM; ++k) rest[1 + k] = __float2int_rn(__fmul_rn(Mt, v[k]));
    // the x and y momentum channels go through packed fp32x2 arithmetic,
    // which rounds each lane exactly as the scalar operation
    const float2 magic2 = make_float2(kMagic, kMagic);
    float2 Cxy[3] = {make_float2(C[0], C[DIM + 0]), make_float2(C[1], C[DIM + 1]), make_float2(0.f, 0.f)};
    if constexpr (DIM == 3) Cxy[2] = make_float2(C[2], C[5]);
    static_for<3>([&](auto A0) {
        constexpr int a0 = decltype(A0)::value;
        const float Wx = __fmul_rn(w[0][a0], Mt);
        // lane y carries the volume weight with the volume channel, else the mass weight again
        const float2 Wx2 = make_float2(Wx, VC ? __fmul_rn(w[0][a0], Vt) : Wx);
        const float2 h0xy = __ffma2_rn(Cxy[0], make_float2(dd[0][a0], dd[0][a0]), make_float2(v[0], v[1]));
        [[maybe_unused]] float h0z = 0.f;
        if constexpr (DIM == 3) h0z = __fmaf_rn(C[6], dd[0][a0], v[2]);
        static_for<3>([&](auto A1) {
            constexpr int a1 = decltype(A1)::value;
            const float2 Wxy = __fmul2_rn(Wx2, make_float2(w[1][a1], w[1][a1]));
            const float2 h1xy = __ffma2_rn(Cxy[1], make_float2(dd[1][a1], dd[1][a1]), h0xy);
            [[maybe_unused]] float h1z = 0.f;
            if constexpr (DIM == 3) h1z = __fmaf_rn(C[7], dd[1][a1], h0z);
            static_for<(DIM == 3 ? 3 : 1)>([&](auto A2) {
                constexpr int a2 = decltype(A2)::value;
                constexpr int a = DIM == 3 ? (a0 * 9 + a1 * 3 + a2) : (a0 * 3 + a1);
                if constexpr (a != St::CENTRE) {
                    const float2 Wt = DIM == 3 ? __fmul2_rn(Wxy, make_float2(w[2][a2], w[2][a2])) : Wxy;
                    const int32_t sm = rint_f(Wt.x);
                    rest[0] -= sm;
                    ad.template add<0, a>(sm);
                    if constexpr (VC) {
                        const int32_t sv = rint_f(Wt.y);
                        rest[St::NC] -= sv;
                        ad.template add<DIM + 1, a>(sv);
                    }
                    const float2 Wm = VC ? make_float2(Wt.x, Wt.x) : Wt;
                    const float2 velxy =
                        DIM == 3 ? __ffma2_rn(Cxy[2], make_float2(dd[2][a2], dd[2][a2]), h1xy) : h1xy;
                    const float2 bxy = __ffma2_rn(Wm, velxy, magic2);
                    const int32_t sx = __float_as_int(bxy.x) - kMagicBits, sy = __float_as_int(bxy.y) - kMagicBits;
                    rest[1] -= sx;
                    rest[2] -= sy;
                    ad.template add<1, a>(sx);
                    ad.template add<2, a>(sy);
                    if constexpr (DIM == 3) {
                        const float velz = __fmaf_rn(C[8], dd[2][a2], h1z);
                        const int32_t sz = rint_mul(Wt.x, velz);
                        rest[3] -= sz;
                        ad.template add<3, a>(sz);
                    }
                }
            });
        });
    });
    ad.template add<0, St::CENTRE>(rest[0]);
    ad.template add<1, St::CENTRE>(rest[1]);
    ad.template add<2, St::CENTRE>(rest[2]);
    if constexpr (DIM == 3) ad.template add<3, St::CENTRE>(rest[3]);
    if constexpr (VC) ad.template add<DIM + 1, St::CENTRE>(rest[St::NC]);
    return true;
}

// --------------------------------------------------------------------------
// Shares of any size (up to the bound): the same values as scatter_shares,
// each the exact product rounded once (rint_prod64), as int64.

// A 64-bit share into the shared-memory tile accumulator: split as
// s = hi * 2^22 + lo, lo the sign-extended low 22 bits, each half added to its
// own int32 plane (lo planes at channel c, hi planes at NCH + c).  Between two
// flushes at most 512 shares reach one entry, so the lo sums stay below 2^30
// and the hi sums below 2^31 for shares below 2^43.  The x offset a0 of the
// stencil node is a run-time value (the wide path keeps its outer loop
// rolled, see scatter_shares_wide); a1 and a2 are compile-time.
template <typename Hl, int NCH>
struct SharedAdd64 {
    uint32_t base;
    template <int C, int A12>
    __device__ __forceinline__ void add(int a0, long long s) const {
        const int32_t lo = ((int32_t)((uint32_t)s << 10)) >> 10;
        const int32_t hi = (int32_t)((s - lo) >> 22);
        const uint32_t at = base + 4u * (uint32_t)a0;
        red_shared_add<4 * (Hl::off(A12) + C * Hl::SIZE)>(at, lo);
        red_shared_add<4 * (Hl::off(A12) + (NCH + C) * Hl::SIZE)>(at, hi);
    }
};

// A 64-bit share straight into the global grid (int64, or int32 where the
// bound keeps every node sum in range); node0 = the stencil's first node,
// A12 = a1*3 + a2 (3D) or a1 (2D).
template <int DIM, typename AccT>
struct GlobalAdd64 {
    AccT *acc;
    int64_t nodes, n0, n01, node0;
    template <int C, int A12>
    __device__ __forceinline__ void add(int a0, long long s) const {
        constexpr int a1 = DIM == 3 ? A12 / 3 : A12;
        constexpr int a2 = DIM == 3 ? A12 % 3 : 0;
        AccT *at = acc + C * nodes + node0 + a0 + a1 * n0 + a2 * n01;
        if constexpr (sizeof(AccT) == 8)
            atomicAdd(reinterpret_cast<unsigned long long *>(at), (unsigned long long)s);
        else
            atomicAdd(reinterpret_cast<int *>(at), (int)s);
    }
};

// One particle's shares of any size, handed to `ad` as 64-bit integers:
// s_m(a) = rint(Wt(a)) and s_k(a) = rint(Wt(a) * vel_k(a)) of the exact
// product, the centre the remainder, in the same order of fp32 operations as
// scatter_shares, so the values are the same wherever both apply.  The loop
// over a0 stays rolled: fully unrolled, the 27 nodes' integer products made
// the kernel too large for the instruction cache (its warps stalled mostly
// waiting for instructions).  Ad::add takes a0 at run time and (a1, a2) as
// compile-time A12 = a1*3 + a2 (3D) or a1 (2D).
template <int DIM, bool EL, bool VC, typename Rec, typename Add>
__device__ __forceinline__ void scatter_shares_wide(const GridP &g, const Rec &rec, const float (&f)[3],
                                                    const Add &ad, const float (&v)[DIM],
                                                    const float (&C)[DIM * DIM]) {
    using Fl = P2GFields<DIM, EL, VC>;
    using St = Stencil<DIM>;
    const float Mt = __fmul_rn(rec(2 * DIM + DIM * DIM), g.S);
    [[maybe_unused]] float Vt = 0.f;
    if constexpr (VC) Vt = __fmul_rn(__fmul_rn(rec(Fl::VOLF), g.vcell), g.S);
    float w[3][3], dd[3][3];
#pragma unroll
    for (int l = 0; l < DIM; ++l) {
        quad_weights(f[l], w[l]);
#pragma unroll
        for (int a = 0; a < 3; ++a) dd[l][a] = __fmul_rn(__fsub_rn((float)a, f[l]), g.dx);
    }
    long long rest[St::NC + 1];
    rest[0] = __float2ll_rn(Mt);
    rest[St::NC] = VC ? __float2ll_rn(Vt) : 0ll;
#pragma unroll
    for (int k = 0; k < DIM; ++k) rest[1 + k] = __float2ll_rn(__fmul_rn(Mt, v[k]));
    constexpr int A12C = DIM == 3 ? 4 : 1;  // (a1, a2) = (1, 1) (3D) or a1 = 1 (2D): the centre with a0 = 1
#pragma unroll 1
    for (int a0 = 0; a0 < 3; ++a0) {
        const float wx = a0 == 0 ? w[0][0] : (a0 == 1 ? w[0][1] : w[0][2]);
        const float dx0 = a0 == 0 ? dd[0][0] : (a0 == 1 ? dd[0][1] : dd[0][2]);
        const float Wx = __fmul_rn(wx, Mt);
        [[maybe_unused]] float Vx = 0.f;
        if constexpr (VC) Vx = __fmul_rn(wx, Vt);
        float h0[DIM];
#pragma unroll
        for (int k = 0; k < DIM; ++k) h0[k] = __fmaf_rn(C[k * DIM + 0], dx0, v[k]);
        static_for<3>([&](auto A1) {
            constexpr int a1 = decltype(A1)::value;
            const float Wxy = __fmul_rn(Wx, w[1][a1]);
            [[maybe_unused]] float Vxy = 0.f;
            if constexpr (VC) Vxy = __fmul_rn(Vx, w[1][a1]);
            float h1[DIM];
#pragma unroll
            for (int k = 0; k < DIM; ++k) h1[k] = __fmaf_rn(C[k * DIM + 1], dd[1][a1], h0[k]);
            static_for<(DIM == 3 ? 3 : 1)>([&](auto A2) {
                constexpr int a2 = decltype(A2)::value;
                constexpr int A12 = DIM == 3 ? a1 * 3 + a2 : a1;
                if (A12 != A12C || a0 != 1) {
                    const float Wt = DIM == 3 ? __fmul_rn(Wxy, w[2][a2]) : Wxy;
                    const long long sm = __float2ll_rn(Wt);
                    rest[0] -= sm;
                    ad.template add<0, A12>(a0, sm);
                    if constexpr (VC) {
                        const long long sv = __float2ll_rn(DIM == 3 ? __fmul_rn(Vxy, w[2][a2]) : Vxy);
                        rest[St::NC] -= sv;
                        ad.template add<DIM + 1, A12>(a0, sv);
                    }
                    static_for<DIM>([&](auto K) {
                        constexpr int k = decltype(K)::value;
                        const float vel = DIM == 3 ? __fmaf_rn(C[k * DIM + 2], dd[2][a2], h1[k]) : h1[k];
                        const long long sk = rint_prod64(Wt, vel);
                        rest[1 + k] -= sk;
                        ad.template add<1 + k, A12>(a0, sk);
                    });
                }
            });
        });
    }
    ad.template add<0, A12C>(1, rest[0]);
    static_for<DIM>([&](auto K) {
        constexpr int k = decltype(K)::value;
        ad.template add<1 + k, A12C>(1, rest[1 + k]);
    });
    if constexpr (VC) ad.template add<DIM + 1, A12C>(1, rest[St::NC]);
}

}  // namespace mpm
