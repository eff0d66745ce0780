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
// One iteration is one kernel with one warp per work item (a slice of a
// tile, the P2G kernel's shape): the warp loads the tile's halo of the
// accumulators R applying the grid update (mass-normalise and boundary;
// gravity is not applied inside the loop) into its own shared-memory
// velocity halo, then, 32 particles a round (each lane's next position and
// mass loaded into registers while the current particle is processed), each
// lane gathers its particle's new (d, D), writes it in place and scatters it
// from its registers at the same position into the warp's own accumulator
// halo, which the warp adds to
// the accumulators W after every 512 particles and at the end.  No block
// barrier couples the warps.  The last iteration only gathers.  R is cleared
// as the iteration goes by its readers' count (release_blocks: the last work
// item to load a node block clears it).  The material projections the page
// runs between the transfers are not part of it.
#include "common.cuh"
#include "gather.cuh"
#include "internal.h"
#include "scatter.cuh"

namespace mpm {

// Per warp: a velocity halo and an accumulator halo.
template <int DIM, int T, bool SCATTER>
__global__ void __launch_bounds__(kP2GThreads, 3)
    k_iterate_w(GridP g, PartsF p, const long long *__restrict__ accR, long long *__restrict__ accW,
                uint32_t *__restrict__ readers, const uint32_t *__restrict__ count,
                const uint32_t *__restrict__ perm, const uint32_t *__restrict__ slices,
                const uint32_t *__restrict__ start, uint32_t *__restrict__ status, float c4) {
    using Hl = HaloU<DIM, T>;
    using St = Stencil<DIM>;
    constexpr int NW = kP2GThreads / 32;
    constexpr int VW = DIM * Hl::SIZE;                       // velocity words per warp
    constexpr int AW = SCATTER ? St::NC * Hl::SIZE : 1;      // accumulator words per warp
    __shared__ float svel[NW][VW];
    __shared__ __align__(16) int32_t sacc[NW][AW];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    float *vw = svel[warp];
    const VelHalo<DIM, T> sv{vw, vw + Hl::SIZE, DIM == 3 ? vw + 2 * Hl::SIZE : vw, nullptr};
    int32_t *wh = sacc[warp];
    const uint32_t halo = (uint32_t)__cvta_generic_to_shared(wh);
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    uint32_t *work = &status[MPM_ST_WORK_G2P];
    const StressP sp{0.f, 0.f, 0.f, 0.f};
    const float kNoGravity[3] = {0.f, 0.f, 0.f};  // the loop adds gravity only at integration
    uint32_t bad = 0, unused = 0;
    if constexpr (SCATTER)
        for (int i = lane; i < AW; i += 32) wh[i] = 0;
    __syncwarp();
    int o[3];
    auto flush = [&]() {
        __syncwarp();
        for (int h = lane; h < Hl::NODES; h += 32) {
            int hx, hy, hz;
            Hl::node(h, hx, hy, hz);
            const int gx = o[0] + hx, gy = o[1] + hy, gz = o[2] + hz;
            const bool on = gx < g.n[0] && gy < g.n[1] && (DIM == 2 || gz < g.n[2]);
            const int64_t node = on ? node_index(g, gx, gy, gz) : 0;
#pragma unroll
            for (int c = 0; c < St::NC; ++c) {
                const int32_t val = wh[c * Hl::SIZE + h];
                if (val == 0) continue;
                wh[c * Hl::SIZE + h] = 0;
                if (on)
                    atomicAdd(reinterpret_cast<unsigned long long *>(accW + c * g.nodes + node),
                              (unsigned long long)(long long)val);
            }
        }
        __syncwarp();
    };
    uint32_t s = 0;
    if (lane == 0) s = atomicAdd(work, 1u);
    s = __shfl_sync(0xFFFFFFFFu, s, 0);
    while (s < nslices) {
        const uint32_t ask = lane == 0 ? atomicAdd(work, 1u) : 0u;
        const uint32_t t = slices[2 * (size_t)s];
        const uint32_t beg = start[t] + slices[2 * (size_t)s + 1];
        const uint32_t cnt = min((uint32_t)kSliceParticles, start[t + 1] - beg);
        tile_origin(g, t, o);
        // positions and masses in registers a round ahead, perm two rounds ahead
        uint32_t pid = lane < cnt ? perm[beg + lane] : 0u;
        uint32_t pid_next = lane + 32 < cnt ? perm[beg + lane + 32] : 0u;
        float xc[DIM + 1], xn[DIM + 1];
#pragma unroll
        for (int l = 0; l < DIM; ++l) xc[l] = lane < cnt ? p.x[l][pid] : 0.f;
        xc[DIM] = lane < cnt ? p.m[pid] : 0.f;
        // the halo's node values, the grid update (without gravity) applied on load
        load_halo<DIM, T, false, 1, 2>(g, accR, kNoGravity, o, vw, (int)lane, 32);
        __syncwarp();
        // this work item has read its blocks of R: the last reader of a block clears it
        release_blocks<DIM, T, long long, DIM + 1>(g, t, readers, count, const_cast<long long *>(accR), lane);
        const uint32_t rounds = (cnt + 31) / 32;
        for (uint32_t q = 0; q < rounds; ++q) {
            const uint32_t r = q * 32 + lane;
#pragma unroll
            for (int l = 0; l < DIM; ++l) xn[l] = r + 32 < cnt ? p.x[l][pid_next] : 0.f;
            xn[DIM] = r + 32 < cnt ? p.m[pid_next] : 0.f;
            const uint32_t pid_after = r + 64 < cnt ? perm[beg + r + 64] : 0u;
            if (r < cnt) {
                float x[DIM], f[3] = {0.f, 0.f, 0.f};
                int b[3] = {0, 0, 0};
#pragma unroll
                for (int l = 0; l < DIM; ++l) x[l] = xc[l];
                if (in_box_x<DIM, T>(g, x, o, b, f)) {
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
                    float rec_v[P2GFields<DIM>::NF];
#pragma unroll
                    for (int k = 0; k < DIM; ++k) {
                        p.v[k][pid] = vn[k];
                        rec_v[DIM + k] = vn[k];
#pragma unroll
                        for (int l = 0; l < DIM; ++l) {
                            const float c = __fmul_rn(Bm[k][l], c4);
                            p.C[k * DIM + l][pid] = c;
                            rec_v[2 * DIM + k * DIM + l] = c;
                        }
                    }
                    if constexpr (SCATTER) {
#pragma unroll
                        for (int l = 0; l < DIM; ++l) rec_v[l] = x[l];
                        rec_v[2 * DIM + DIM * DIM] = xc[DIM];
                        auto rec = [&](int fi) { return rec_v[fi]; };
                        const SharedAdd<Hl> ad{halo + 4u * (uint32_t)hb};
                        if (!scatter_shares<DIM, false, false, true>(g, rec, f, ad, sp, unused)) ++bad;
                    }
                }
            }
#pragma unroll
            for (int l = 0; l <= DIM; ++l) xc[l] = xn[l];
            pid = pid_next;
            pid_next = pid_after;
            // int32 accumulators: at most 512 shares below 2^22 reach one entry between two flushes
            if constexpr (SCATTER)
                if ((q + 1) % 16 == 0 && q + 1 < rounds) flush();
        }
        if constexpr (SCATTER) flush();
        __syncwarp();
        s = __shfl_sync(0xFFFFFFFFu, ask, 0);
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
    const int blocks = dev.sms * 4;
    // the block reader counts start at zero; each iteration's readers leave them at zero again
    cudaMemsetAsync(w.readers, 0, (size_t)g.nblocks * sizeof(uint32_t), st);
    for (int it = 0; it < iterations; ++it) {
        cudaMemsetAsync(&w.status[MPM_ST_WORK_G2P], 0, sizeof(uint32_t), st);
        // R = a is read and cleared as the iteration goes (release_blocks), W = b written
        if (it + 1 < iterations)
            k_iterate_w<DIM, T, true><<<blocks, kP2GThreads, 0, st>>>(g, p, a, b, w.readers, w.count, w.perm,
                                                                      w.slices, w.start, w.status, c4);
        else
            k_iterate_w<DIM, T, false><<<blocks, kP2GThreads, 0, st>>>(g, p, a, b, w.readers, w.count, w.perm,
                                                                       w.slices, w.start, w.status, c4);
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
