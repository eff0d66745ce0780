// iterate.cu -- the transfer loop at fixed positions.
//
// Implementation guide ("Implementation -- GPU Optimization & Reference
// Codebases"), section 3.3.2: the position-based solver runs P2G -> grid
// update -> G2P iterationCount times per substep with the particles in
// place, the particle carrying a displacement d and its gradient D where the
// velocity form carries v and C (the transfer arithmetic is the same:
// momentum(d + D * offset) out, d and D = B * 4 back); section 2.1: this
// loop is where one fused kernel per iteration pays most, since the gather
// and the scatter of an iteration use the same positions and the same tile.
//
// One iteration is one kernel: a block per slice loads the tile's halo of
// the accumulators R applying the grid update (mass-normalise and boundary;
// gravity is not applied inside the loop), each thread gathers its
// particle's new (d, D) and writes it in place, then scatters it at the same
// position into the tile's shared accumulator, which the block adds to the
// accumulators W once.  The last iteration only gathers.  After each
// iteration a second kernel clears R.  The material projections the page
// runs between the transfers are not part of it.
#include "common.cuh"
#include "gather.cuh"
#include "internal.h"
#include "scatter.cuh"

namespace mpm {

template <int DIM, int T, bool SCATTER>
__global__ void __launch_bounds__(kG2PThreads, 2)
    k_iterate(GridP g, PartsF p, const long long *__restrict__ accR, long long *__restrict__ accW,
              const uint32_t *__restrict__ perm, const uint32_t *__restrict__ slices,
              const uint32_t *__restrict__ start, uint32_t *__restrict__ status, float c4) {
    using Hl = HaloU<DIM, T>;
    using St = Stencil<DIM>;
    constexpr int NQ = kSliceParticles / kG2PThreads;
    constexpr int NF = DIM + 1;  // staged: x, m
    constexpr int XW = SCATTER ? St::NC * Hl::SIZE : 1;
    __shared__ float sv_x[Hl::SIZE], sv_y[Hl::SIZE], sv_z[DIM == 3 ? Hl::SIZE : 1];
    const VelHalo<DIM, T> sv{sv_x, sv_y, sv_z, nullptr};
    __shared__ float sbuf[NF * kSliceParticles];
    __shared__ __align__(16) int32_t sacc[XW];
    __shared__ uint32_t item_sh;
    const uint32_t lane = lane_id();
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    const uint32_t halo = (uint32_t)__cvta_generic_to_shared(sacc);
    const StressP sp{0.f, 0.f, 0.f, 0.f};
    uint32_t bad = 0, unused = 0;
    if constexpr (SCATTER)
        for (int i = threadIdx.x; i < XW; i += blockDim.x) sacc[i] = 0;
    int o[3];
    auto flush = [&]() {
        for (int h = threadIdx.x; h < Hl::NODES; h += blockDim.x) {
            int hx, hy, hz;
            Hl::node(h, hx, hy, hz);
            const int gx = o[0] + hx, gy = o[1] + hy, gz = o[2] + hz;
            const bool on = gx < g.n[0] && gy < g.n[1] && (DIM == 2 || gz < g.n[2]);
            const int64_t node = on ? node_index(g, gx, gy, gz) : 0;
#pragma unroll
            for (int c = 0; c < St::NC; ++c) {
                const int32_t val = sacc[c * Hl::SIZE + h];
                if (val == 0) continue;
                sacc[c * Hl::SIZE + h] = 0;
                if (on)
                    atomicAdd(reinterpret_cast<unsigned long long *>(accW + c * g.nodes + node),
                              (unsigned long long)(long long)val);
            }
        }
    };
    uint32_t next = 0;
    for (uint32_t s = grab_item(&status[MPM_ST_WORK_G2P], &item_sh); s < nslices; s = publish_item(next, &item_sh)) {
        next = ask_item(&status[MPM_ST_WORK_G2P]);
        const uint32_t t = slices[2 * (size_t)s], first = slices[2 * (size_t)s + 1];
        const uint32_t beg = start[t] + first;
        const uint32_t cnt = min((uint32_t)kSliceParticles, start[t + 1] - beg);
        tile_origin(g, t, o);
        uint32_t pids[NQ];
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            const uint32_t r = threadIdx.x + qi * kG2PThreads;
            pids[qi] = r < cnt ? perm[beg + r] : 0u;
            if (r < cnt) {
#pragma unroll
                for (int f = 0; f < DIM; ++f) cp_async4(&sbuf[f * kSliceParticles + r], p.x[f] + pids[qi]);
                cp_async4(&sbuf[DIM * kSliceParticles + r], p.m + pids[qi]);
            }
        }
        cp_async_commit();
        // the halo's node values, the grid update (without gravity) applied on load
        for (int h = threadIdx.x; h < Hl::NODES; h += blockDim.x) {
            int hx, hy, hz;
            Hl::node(h, hx, hy, hz);
            const int gi[3] = {o[0] + hx, o[1] + hy, o[2] + hz};
            float v[3] = {0.f, 0.f, 0.f};
            if (gi[0] < g.n[0] && gi[1] < g.n[1] && (DIM == 2 || gi[2] < g.n[2])) {
                const int64_t node = node_index(g, gi[0], gi[1], gi[2]);
                const float M = __ll2float_rn(accR[node]);
                if (M != 0.f) {
#pragma unroll
                    for (int l = 0; l < DIM; ++l) {
                        float vl = __fadd_rn(__fdiv_rn(__ll2float_rn(accR[(1 + l) * g.nodes + node]), M), 0.f);
                        if ((gi[l] < g.boundary && vl < 0.f) || (gi[l] > g.n[l] - 1 - g.boundary && vl > 0.f))
                            vl = 0.f;
                        v[l] = vl;
                    }
                }
            }
            sv_x[h] = v[0];
            sv_y[h] = v[1];
            if (DIM == 3) sv_z[h] = v[2];
        }
        cp_async_wait<0>();
        __syncthreads();
        // gather: the new (d, D) of each particle, written in place
#pragma unroll 1
        for (int qi = 0; qi < NQ; ++qi) {
            const uint32_t r = threadIdx.x + qi * kG2PThreads;
            if (r >= cnt) continue;
            const uint32_t pid = perm[beg + r];
            float x[DIM], f[3] = {0.f, 0.f, 0.f};
            int b[3] = {0, 0, 0};
#pragma unroll
            for (int l = 0; l < DIM; ++l) x[l] = sbuf[l * kSliceParticles + r];
            if (!in_box_x<DIM, T>(g, x, o, b, f)) continue;
            float w[3][3], we[3][3];
#pragma unroll
            for (int l = 0; l < DIM; ++l) {
                quad_weights(f[l], w[l]);
#pragma unroll
                for (int a = 0; a < 3; ++a) we[l][a] = __fmul_rn(w[l][a], __fsub_rn((float)a, f[l]));
            }
            const int hb = DIM == 3 ? (b[0] - o[0]) + (b[1] - o[1]) * Hl::SY + (b[2] - o[2]) * Hl::SZ
                                    : (b[0] - o[0]) + (b[1] - o[1]) * Hl::SY;
            float vn[DIM], Bm[DIM][DIM];
            gather_vB<DIM, T>(sv, hb, w, we, vn, Bm);
#pragma unroll
            for (int k = 0; k < DIM; ++k) {
                p.v[k][pid] = vn[k];
#pragma unroll
                for (int l = 0; l < DIM; ++l) p.C[k * DIM + l][pid] = __fmul_rn(Bm[k][l], c4);
            }
        }
        if constexpr (SCATTER) {
            // scatter the new (d, D) at the same positions (read back from this thread's own writes)
#pragma unroll 1
            for (int qi = 0; qi < NQ; ++qi) {
                const uint32_t r = threadIdx.x + qi * kG2PThreads;
                if (r < cnt) {
                    const uint32_t pid = perm[beg + r];
                    float rec_v[P2GFields<DIM>::NF];
#pragma unroll
                    for (int l = 0; l < DIM; ++l) {
                        rec_v[l] = sbuf[l * kSliceParticles + r];
                        rec_v[DIM + l] = p.v[l][pid];
                    }
#pragma unroll
                    for (int j = 0; j < DIM * DIM; ++j) rec_v[2 * DIM + j] = p.C[j][pid];
                    rec_v[2 * DIM + DIM * DIM] = sbuf[DIM * kSliceParticles + r];
                    auto rec = [&](int fi) { return rec_v[fi]; };
                    float xs[DIM], f[3] = {0.f, 0.f, 0.f};
                    int b[3] = {0, 0, 0};
#pragma unroll
                    for (int l = 0; l < DIM; ++l) xs[l] = rec_v[l];
                    if (in_box_x<DIM, T>(g, xs, o, b, f)) {
                        const int hb = DIM == 3 ? (b[0] - o[0]) + (b[1] - o[1]) * Hl::SY + (b[2] - o[2]) * Hl::SZ
                                                : (b[0] - o[0]) + (b[1] - o[1]) * Hl::SY;
                        const SharedAdd<Hl> ad{halo + 4u * (uint32_t)hb};
                        if (!scatter_shares<DIM, false, false>(g, rec, f, ad, sp, unused)) ++bad;
                    }
                }
                // int32 accumulators: at most 512 shares below 2^22 reach one entry between two flushes
                if (qi == 1 && cnt > 2u * kG2PThreads) {
                    __syncthreads();
                    flush();
                    __syncthreads();
                }
            }
            __syncthreads();
            flush();
        }
    }
    if constexpr (SCATTER) {
        bad = __reduce_add_sync(0xFFFFFFFFu, bad);
        if (bad && lane == 0) {
            atomicAdd(&status[MPM_ST_N_OUT_OF_RANGE], bad);
            set_flag(status, MPM_E_BOUND);
        }
    }
}

template <int DIM, int T>
void launch_iterations(const GridP &g, const PartsF &p, const WsView &w, long long *a, long long *b, int iterations,
                       const DeviceInfo &dev, cudaStream_t st) {
    const float c4 = 4.0f * g.inv_dx;
    const int blocks = dev.sms * 2;
    for (int it = 0; it < iterations; ++it) {
        cudaMemsetAsync(&w.status[MPM_ST_WORK_G2P], 0, sizeof(uint32_t), st);
        if (it + 1 < iterations)
            k_iterate<DIM, T, true><<<blocks, kG2PThreads, 0, st>>>(g, p, a, b, w.perm, w.slices, w.start, w.status,
                                                                    c4);
        else
            k_iterate<DIM, T, false><<<blocks, kG2PThreads, 0, st>>>(g, p, a, b, w.perm, w.slices, w.start,
                                                                     w.status, c4);
        launch_clear_blocks(g, a, w, dev, st);
        std::swap(a, b);
    }
}

mpm_status launch_iterate(const GridP &g, const PartsF &p, const WsView &w, void *acc_a, void *acc_b,
                          int iterations, const DeviceInfo &dev, cudaStream_t st) {
    auto *a = static_cast<long long *>(acc_a), *b = static_cast<long long *>(acc_b);
    if (g.dim == 3 && g.T == 4)
        launch_iterations<3, 4>(g, p, w, a, b, iterations, dev, st);
    else if (g.dim == 2 && g.T == 8)
        launch_iterations<2, 8>(g, p, w, a, b, iterations, dev, st);
    else
        return MPM_E_ARG;
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
