// p2g.cu -- particle-to-grid scatter.
//
// Implementation guide ("Implementation -- GPU Optimization & Reference
// Codebases"), section 1: P2G is the hot spot because many particles add into
// the same nodes; section 2.1: sort + tile + stage the tile in shared memory,
// combine within a warp before any atomic, accumulate fixed-point integers,
// flush each tile once.  Shares follow "particle to grid transfer in checked
// integer arithmetic": split rather than weight, so each particle's shares
// sum exactly to its quantity and the grid is the same in every order.
//
// Work item: a slice of at most 256 consecutive sorted particles of one tile
// (T^dim base cells).  A CTA zeroes the tile's (T+2)^dim x (dim+1) int32
// accumulators in shared memory, each thread computes its particle's shares,
// warps whose 32 particles share one base cell add each share with one
// redux.sync and one shared atomic, the others add lane by lane, and the CTA
// flushes every nonzero node once with a global atomic add (neighbouring
// slices and tiles overlap on halo nodes, so the flush must add).
#include "common.cuh"
#include "internal.h"

namespace mpm {

// Share encode: rint(a * b) for |a*b| < 2^22, exact product rounded once (RNE).
__device__ __forceinline__ int32_t rint_mul(float a, float b) {
    return __float_as_int(__fmaf_rn(a, b, kMagic)) - kMagicBits;
}
__device__ __forceinline__ int32_t rint_f(float a) { return __float_as_int(__fadd_rn(a, kMagic)) - kMagicBits; }

template <int DIM>
struct Stencil {
    static constexpr int NA = DIM == 3 ? 27 : 9;
    static constexpr int NC = DIM + 1;
    static constexpr int CENTRE = DIM == 3 ? 13 : 4;  // a = (1,1,1) / (1,1)
};

// Loads particle `pid`, checks the domain and the share range, and computes
// its NC x NA integer shares (fixed point) -- the arithmetic the oracle states.
// Returns 0 = ok, 1 = outside the domain, 2 = out of range.
template <int DIM>
__device__ __forceinline__ int particle_shares(const GridP &g, const PartsF &p, uint32_t pid, int b[3],
                                               int32_t sh[Stencil<DIM>::NC][Stencil<DIM>::NA]) {
    using St = Stencil<DIM>;
    float f[3] = {0.f, 0.f, 0.f};
    b[2] = 0;
#pragma unroll
    for (int l = 0; l < DIM; ++l)
        if (!base_frac(p.x[l][pid], g.inv_dx, g.n[l], b[l], f[l])) return 1;
    float v[DIM], C[DIM * DIM];
#pragma unroll
    for (int k = 0; k < DIM; ++k) v[k] = p.v[k][pid];
#pragma unroll
    for (int j = 0; j < DIM * DIM; ++j) C[j] = p.C[j][pid];
    const float Mt = __fmul_rn(p.m[pid], g.S);
    // range: wmax*|Mt| and wmax*|Mt|*(|v_k| + 1.5 dx sum_l |C_kl|) below 2^22 - 4096
    const float h = __fmul_rn(1.5f, g.dx);
    const float aM = fabsf(Mt);
    bool ok = __fmul_rn(g.wmax, aM) <= kShareLimit;
#pragma unroll
    for (int k = 0; k < DIM; ++k) {
        float sc = __fadd_rn(fabsf(C[k * DIM + 0]), fabsf(C[k * DIM + 1]));
        if (DIM == 3) sc = __fadd_rn(sc, fabsf(C[k * DIM + 2]));
        const float R = __fmul_rn(aM, __fadd_rn(fabsf(v[k]), __fmul_rn(h, sc)));
        ok = ok && (__fmul_rn(g.wmax, R) <= kShareLimit);
    }
    if (!ok) return 2;
    float w[3][3], dd[3][3];
#pragma unroll
    for (int l = 0; l < DIM; ++l) {
        quad_weights(f[l], w[l]);
#pragma unroll
        for (int a = 0; a < 3; ++a) dd[l][a] = __fmul_rn(__fsub_rn((float)a, f[l]), g.dx);
    }
    int32_t Q[St::NC];
    Q[0] = __float2int_rn(Mt);
#pragma unroll
    for (int k = 0; k < DIM; ++k) Q[1 + k] = __float2int_rn(__fmul_rn(Mt, v[k]));
    int32_t rest[St::NC];
#pragma unroll
    for (int c = 0; c < St::NC; ++c) rest[c] = Q[c];
#pragma unroll
    for (int a0 = 0; a0 < 3; ++a0) {
        const float Wx = __fmul_rn(w[0][a0], Mt);
        float h0[DIM];
#pragma unroll
        for (int k = 0; k < DIM; ++k) h0[k] = __fmaf_rn(C[k * DIM + 0], dd[0][a0], v[k]);
#pragma unroll
        for (int a1 = 0; a1 < 3; ++a1) {
            const float Wxy = __fmul_rn(Wx, w[1][a1]);
            float h1[DIM];
#pragma unroll
            for (int k = 0; k < DIM; ++k) h1[k] = __fmaf_rn(C[k * DIM + 1], dd[1][a1], h0[k]);
#pragma unroll
            for (int a2 = 0; a2 < (DIM == 3 ? 3 : 1); ++a2) {
                const int a = DIM == 3 ? (a0 * 9 + a1 * 3 + a2) : (a0 * 3 + a1);
                if (a == St::CENTRE) continue;
                const float Wt = DIM == 3 ? __fmul_rn(Wxy, w[2][a2]) : Wxy;
                const int32_t sm = rint_f(Wt);
                sh[0][a] = sm;
                rest[0] -= sm;
#pragma unroll
                for (int k = 0; k < DIM; ++k) {
                    const float vel = DIM == 3 ? __fmaf_rn(C[k * DIM + 2], dd[2][a2], h1[k]) : h1[k];
                    const int32_t s = rint_mul(Wt, vel);
                    sh[1 + k][a] = s;
                    rest[1 + k] -= s;
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < St::NC; ++c) sh[c][St::CENTRE] = rest[c];
    return 0;
}

// Shared-memory halo offset of stencil node a relative to the base node.
template <int DIM, int H>
__device__ __forceinline__ constexpr int halo_off(int a) {
    return DIM == 3 ? ((a / 9) + (a / 3 % 3) * H + (a % 3) * H * H) : ((a / 3) + (a % 3) * H);
}

template <int DIM, int T, typename AccT>
__global__ void __launch_bounds__(kSliceParticles) k_p2g_fixed(GridP g, PartsF p, const uint32_t *__restrict__ perm,
                                                               const uint32_t *__restrict__ slices,
                                                               const uint32_t *__restrict__ start,
                                                               uint32_t *__restrict__ status, AccT *__restrict__ acc) {
    using St = Stencil<DIM>;
    constexpr int H = T + 2;
    constexpr int HN = DIM == 3 ? H * H * H : H * H;
    __shared__ int32_t sacc[St::NC * HN];
    if (status[MPM_ST_FLAGS] & kFlagNoScatter) return;
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    const uint32_t lane = lane_id();
    for (uint32_t s = blockIdx.x; s < nslices; s += gridDim.x) {
        const uint32_t t = slices[2 * (size_t)s], first = slices[2 * (size_t)s + 1];
        const uint32_t beg = start[t] + first;
        const uint32_t cnt = min((uint32_t)kSliceParticles, start[t + 1] - beg);
        int o[3];
        tile_origin(g, t, o);
        for (int i = threadIdx.x; i < St::NC * HN; i += blockDim.x) sacc[i] = 0;
        __syncthreads();

        int32_t sh[St::NC][St::NA];
        int b[3] = {0, 0, 0};
        int res = 1;
        if (threadIdx.x < cnt) res = particle_shares<DIM>(g, p, perm[beg + threadIdx.x], b, sh);
        if (threadIdx.x < cnt && res == 2) {
            atomicAdd(&status[MPM_ST_N_OUT_OF_RANGE], 1u);
            set_flag(status, MPM_E_BOUND);
        }
        const bool ok = res == 0;
        const int hb = DIM == 3 ? ((b[2] - o[2]) * H + (b[1] - o[1])) * H + (b[0] - o[0])
                                : (b[1] - o[1]) * H + (b[0] - o[0]);
        const int hb0 = __shfl_sync(0xFFFFFFFFu, hb, 0);
        const bool uniform = __all_sync(0xFFFFFFFFu, ok && hb == hb0);
        if (uniform) {
            // one base cell for the whole warp: reduce each share across lanes
#pragma unroll
            for (int c = 0; c < St::NC; ++c)
#pragma unroll
                for (int a = 0; a < St::NA; ++a) {
                    const uint32_t r = __reduce_add_sync(0xFFFFFFFFu, (uint32_t)sh[c][a]);
                    if (lane == (uint32_t)((c * St::NA + a) & 31))
                        atomicAdd(&sacc[c * HN + hb0 + halo_off<DIM, H>(a)], (int32_t)r);
                }
        } else if (ok) {
#pragma unroll
            for (int c = 0; c < St::NC; ++c)
#pragma unroll
                for (int a = 0; a < St::NA; ++a) atomicAdd(&sacc[c * HN + hb + halo_off<DIM, H>(a)], sh[c][a]);
        }
        __syncthreads();
        for (int h = threadIdx.x; h < HN; h += blockDim.x) {
            const int hx = h % H, hy = (h / H) % H, hz = DIM == 3 ? h / (H * H) : 0;
            const int gx = o[0] + hx, gy = o[1] + hy, gz = o[2] + hz;
            if (gx >= g.n[0] || gy >= g.n[1] || (DIM == 3 && gz >= g.n[2])) continue;
            const int64_t node = node_index(g, gx, gy, gz);
#pragma unroll
            for (int c = 0; c < St::NC; ++c) {
                const int32_t val = sacc[c * HN + h];
                if (val == 0) continue;
                if constexpr (sizeof(AccT) == 8)
                    atomicAdd(reinterpret_cast<unsigned long long *>(acc + c * g.nodes + node),
                              (unsigned long long)(long long)val);
                else
                    atomicAdd(reinterpret_cast<int *>(acc + c * g.nodes + node), val);
            }
        }
        __syncthreads();
    }
}

// Float-atomic P2G (comparison variant: fp32 adds, order dependent).
template <int DIM, int T>
__global__ void __launch_bounds__(kSliceParticles) k_p2g_float(GridP g, PartsF p, const uint32_t *__restrict__ perm,
                                                               const uint32_t *__restrict__ slices,
                                                               const uint32_t *__restrict__ start,
                                                               const uint32_t *__restrict__ status,
                                                               float *__restrict__ acc) {
    using St = Stencil<DIM>;
    constexpr int H = T + 2;
    constexpr int HN = DIM == 3 ? H * H * H : H * H;
    __shared__ float sacc[St::NC * HN];
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    for (uint32_t s = blockIdx.x; s < nslices; s += gridDim.x) {
        const uint32_t t = slices[2 * (size_t)s], first = slices[2 * (size_t)s + 1];
        const uint32_t beg = start[t] + first;
        const uint32_t cnt = min((uint32_t)kSliceParticles, start[t + 1] - beg);
        int o[3];
        tile_origin(g, t, o);
        for (int i = threadIdx.x; i < St::NC * HN; i += blockDim.x) sacc[i] = 0.f;
        __syncthreads();
        if (threadIdx.x < cnt) {
            const uint32_t pid = perm[beg + threadIdx.x];
            int b[3] = {0, 0, 0};
            float f[3] = {0.f, 0.f, 0.f};
            bool ok = true;
#pragma unroll
            for (int l = 0; l < DIM; ++l) ok = ok && base_frac(p.x[l][pid], g.inv_dx, g.n[l], b[l], f[l]);
            if (ok) {
                float v[DIM], C[DIM * DIM], w[3][3], dd[3][3];
#pragma unroll
                for (int k = 0; k < DIM; ++k) v[k] = p.v[k][pid];
#pragma unroll
                for (int j = 0; j < DIM * DIM; ++j) C[j] = p.C[j][pid];
                const float m = p.m[pid];
#pragma unroll
                for (int l = 0; l < DIM; ++l) {
                    quad_weights(f[l], w[l]);
#pragma unroll
                    for (int a = 0; a < 3; ++a) dd[l][a] = __fmul_rn(__fsub_rn((float)a, f[l]), g.dx);
                }
                const int hb = DIM == 3 ? ((b[2] - o[2]) * H + (b[1] - o[1])) * H + (b[0] - o[0])
                                        : (b[1] - o[1]) * H + (b[0] - o[0]);
#pragma unroll
                for (int a0 = 0; a0 < 3; ++a0) {
                    const float Wx = __fmul_rn(w[0][a0], m);
                    float h0[DIM];
#pragma unroll
                    for (int k = 0; k < DIM; ++k) h0[k] = __fmaf_rn(C[k * DIM + 0], dd[0][a0], v[k]);
#pragma unroll
                    for (int a1 = 0; a1 < 3; ++a1) {
                        const float Wxy = __fmul_rn(Wx, w[1][a1]);
                        float h1[DIM];
#pragma unroll
                        for (int k = 0; k < DIM; ++k) h1[k] = __fmaf_rn(C[k * DIM + 1], dd[1][a1], h0[k]);
#pragma unroll
                        for (int a2 = 0; a2 < (DIM == 3 ? 3 : 1); ++a2) {
                            const int a = DIM == 3 ? (a0 * 9 + a1 * 3 + a2) : (a0 * 3 + a1);
                            const float W = DIM == 3 ? __fmul_rn(Wxy, w[2][a2]) : Wxy;
                            const int off = hb + halo_off<DIM, H>(a);
                            atomicAdd(&sacc[off], W);
#pragma unroll
                            for (int k = 0; k < DIM; ++k) {
                                const float vel = DIM == 3 ? __fmaf_rn(C[k * DIM + 2], dd[2][a2], h1[k]) : h1[k];
                                atomicAdd(&sacc[(1 + k) * HN + off], __fmul_rn(W, vel));
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();
        for (int h = threadIdx.x; h < HN; h += blockDim.x) {
            const int hx = h % H, hy = (h / H) % H, hz = DIM == 3 ? h / (H * H) : 0;
            const int gx = o[0] + hx, gy = o[1] + hy, gz = o[2] + hz;
            if (gx >= g.n[0] || gy >= g.n[1] || (DIM == 3 && gz >= g.n[2])) continue;
            const int64_t node = node_index(g, gx, gy, gz);
#pragma unroll
            for (int c = 0; c < St::NC; ++c) {
                const float val = sacc[c * HN + h];
                if (val != 0.f) atomicAdd(acc + c * g.nodes + node, val);
            }
        }
        __syncthreads();
    }
}

mpm_status launch_p2g(const GridP &g, const PartsF &p, const WsView &w, void *grid_acc, const DeviceInfo &dev,
                      cudaStream_t st) {
    const int blocks = dev.sms * 4;
    if (g.dim == 3 && g.T == 4) {
        if (g.acc_mode == MPM_ACC_I64)
            k_p2g_fixed<3, 4, int64_t><<<blocks, kSliceParticles, 0, st>>>(g, p, w.perm, w.slices, w.start, w.status,
                                                                          (int64_t *)grid_acc);
        else if (g.acc_mode == MPM_ACC_I32)
            k_p2g_fixed<3, 4, int32_t><<<blocks, kSliceParticles, 0, st>>>(g, p, w.perm, w.slices, w.start, w.status,
                                                                          (int32_t *)grid_acc);
        else
            k_p2g_float<3, 4><<<blocks, kSliceParticles, 0, st>>>(g, p, w.perm, w.slices, w.start, w.status,
                                                                 (float *)grid_acc);
    } else if (g.dim == 2 && g.T == 8) {
        if (g.acc_mode == MPM_ACC_I64)
            k_p2g_fixed<2, 8, int64_t><<<blocks, kSliceParticles, 0, st>>>(g, p, w.perm, w.slices, w.start, w.status,
                                                                          (int64_t *)grid_acc);
        else if (g.acc_mode == MPM_ACC_I32)
            k_p2g_fixed<2, 8, int32_t><<<blocks, kSliceParticles, 0, st>>>(g, p, w.perm, w.slices, w.start, w.status,
                                                                          (int32_t *)grid_acc);
        else
            k_p2g_float<2, 8><<<blocks, kSliceParticles, 0, st>>>(g, p, w.perm, w.slices, w.start, w.status,
                                                                 (float *)grid_acc);
    } else {
        return MPM_E_ARG;
    }
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

// --------------------------------------------------------------------------
// Integer cloud-in-cell transfer ("particle to grid transfer in checked
// integer arithmetic").  The bounds line runs first, over all particles, and
// the scatter kernel does nothing if it failed.

// Round-half-even quotient of a / b for b != 0 (exact integer arithmetic).
__device__ __forceinline__ long long div_rne(long long a, long long b) {
    long long q = a / b, r = a % b;
    unsigned long long ar = r < 0 ? 0ull - (unsigned long long)r : (unsigned long long)r;
    unsigned long long br = b < 0 ? 0ull - (unsigned long long)b : (unsigned long long)b;
    unsigned long long other = br - ar;
    if (ar > other || (ar == other && (q & 1))) q += ((a < 0) != (b < 0)) ? -1 : 1;
    return q;
}

// scratch[0] = max |m|, scratch[1] = max |v| (as uint64); status counts positions off the grid.
__global__ void k_cic_bound_reduce(GridP g, PartsI p, unsigned long long *scratch, uint32_t *status) {
    unsigned long long mm = 0, vm = 0;
    uint32_t off = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += (int64_t)gridDim.x * blockDim.x) {
        long long m = p.m[i];
        unsigned long long am = m < 0 ? 0ull - (unsigned long long)m : (unsigned long long)m;
        mm = am > mm ? am : mm;
        for (int k = 0; k < g.dim; ++k) {
            long long v = p.v[k][i];
            unsigned long long av = v < 0 ? 0ull - (unsigned long long)v : (unsigned long long)v;
            vm = av > vm ? av : vm;
        }
        bool bad = false;
        for (int l = 0; l < g.dim; ++l) {
            int32_t X = p.X[l][i];
            bad = bad || X < 0 || (X >> 16) > g.n[l] - 2;
        }
        off += bad ? 1u : 0u;
    }
    for (int d = 16; d > 0; d >>= 1) {
        mm = max(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, d));
        vm = max(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, d));
        off += __shfl_xor_sync(0xFFFFFFFFu, off, d);
    }
    if (lane_id() == 0) {
        atomicMax(&scratch[0], mm);
        atomicMax(&scratch[1], vm);
        if (off) atomicAdd(&status[MPM_ST_N_OUTSIDE], off);
    }
}

__global__ void k_cic_bound_check(int64_t n, const unsigned long long *scratch, uint32_t *status) {
    // count * max|m| * max|v| must fit int64, and so must every product q * F
    const unsigned __int128 mm = scratch[0];
    const unsigned __int128 vm = scratch[1] > 1 ? scratch[1] : 1;
    const unsigned __int128 lim = (unsigned __int128)0x7FFFFFFFFFFFFFFFull;
    const unsigned __int128 q = mm * vm;  // < 2^128
    bool ok = q <= lim / 65536u && q * (unsigned __int128)n <= lim;
    if (status[MPM_ST_N_OUTSIDE]) {
        status[MPM_ST_FLAGS] |= (1u << MPM_E_DOMAIN) | kFlagNoScatter;
    }
    if (!ok) status[MPM_ST_FLAGS] |= (1u << MPM_E_BOUND) | kFlagNoScatter;
    status[MPM_ST_N_VALID] = (uint32_t)n;
}

template <int DIM>
__device__ void cic_split_add(const GridP &g, int64_t *plane, const int c[3], const int32_t F[3], long long q) {
    // split along x, then each part along y (then z); upper node gets rdiv(q*F, 65536)
    long long parts[1 << DIM];
    parts[0] = q;
    int count = 1;
#pragma unroll
    for (int axis = 0; axis < DIM; ++axis) {
#pragma unroll
        for (int j = (1 << axis) - 1; j >= 0; --j) {
            const long long far = div_rne(parts[j] * (long long)F[axis], 65536);
            parts[j + (1 << axis)] = far;
            parts[j] = parts[j] - far;
        }
        count <<= 1;
    }
#pragma unroll
    for (int s = 0; s < (1 << DIM); ++s) {
        const int i = c[0] + (s & 1), j = c[1] + ((s >> 1) & 1), k = DIM == 3 ? c[2] + ((s >> 2) & 1) : 0;
        atomicAdd(reinterpret_cast<unsigned long long *>(plane + node_index(g, i, j, k)),
                  (unsigned long long)parts[s]);
    }
    (void)count;
}

template <int DIM>
__global__ void k_cic_scatter(GridP g, PartsI p, int64_t *acc, const uint32_t *status) {
    if (status[MPM_ST_FLAGS] & kFlagNoScatter) return;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += (int64_t)gridDim.x * blockDim.x) {
        int c[3] = {0, 0, 0};
        int32_t F[3] = {0, 0, 0};
#pragma unroll
        for (int l = 0; l < DIM; ++l) {
            c[l] = p.X[l][i] >> 16;
            F[l] = p.X[l][i] & 0xFFFF;
        }
        const long long m = p.m[i];
        cic_split_add<DIM>(g, acc, c, F, m);
#pragma unroll
        for (int k = 0; k < DIM; ++k) cic_split_add<DIM>(g, acc + (1 + k) * g.nodes, c, F, m * p.v[k][i]);
    }
}

mpm_status launch_cic_int_p2g(const GridP &g, const PartsI &p, int64_t *acc, uint32_t *status, uint64_t *scratch,
                              const DeviceInfo &dev, cudaStream_t st) {
    cudaMemsetAsync(status, 0, MPM_STATUS_WORDS * sizeof(uint32_t), st);
    cudaMemsetAsync(scratch, 0, 2 * sizeof(uint64_t), st);
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((p.n + 255) / 256, dev.sms * 4));
    k_cic_bound_reduce<<<blocks, 256, 0, st>>>(g, p, (unsigned long long *)scratch, status);
    k_cic_bound_check<<<1, 1, 0, st>>>(p.n, (const unsigned long long *)scratch, status);
    if (g.dim == 3)
        k_cic_scatter<3><<<blocks, 256, 0, st>>>(g, p, acc, status);
    else
        k_cic_scatter<2><<<blocks, 256, 0, st>>>(g, p, acc, status);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
