// g2p2g.cu -- the fused gather-scatter step.
//
// Implementation guide ("Implementation -- GPU Optimization & Reference
// Codebases"), section 2.1, the worked shape of "sort + tile + stage in shared
// memory": the whole transfer is one kernel per step; it loads a tile's nodes
// and their halo applying the grid update as it loads (so the read is the
// grid pass), gathers each particle, updates it and scatters it into a
// shared-memory accumulator that is added to the global grid once.
//
// In the guide's position-based solver the particles do not move inside the
// loop, so gather and scatter share one tile.  Here, in the velocity form,
// the gather reads the accumulators R of the P2G at the binned positions x,
// and the scatter writes the next accumulators W at the advected positions
// x' = fma(dt, v', x).  The scatter uses the same tile's accumulator while a
// particle's new base cell stays in the tile; a particle that left the tile
// (a few in ten thousand per step) is scattered straight into the global
// grid, with the same shares.  Shares, velocities and the new state are bit
// for bit those of mpm_bin + mpm_p2g + mpm_grid_update + mpm_g2p_binned, then
// mpm_p2g on the new state.  R is only read (several work items read each
// halo node); a second kernel clears it afterwards, so that it can be the
// next step's W (the guide's rotation of grid buffers).  Clearing R inside
// this kernel by its readers' count, as mpm_g2p_update and the transfer loop
// do (release_blocks), measured slower here: 1.56 ms per step on the 16.7M
// blobs against 1.44 ms with the second kernel.
#include "common.cuh"
#include "gather.cuh"
#include "internal.h"
#include "scatter.cuh"

namespace mpm {

// A particle's shares straight into the global grid (the rare particle whose
// new base cell left its tile); out of line, so that its registers do not
// weigh on the kernel's common path.  False when out of range.
template <int DIM>
__device__ __noinline__ bool scatter_global(const GridP &g, const float (&rec_v)[P2GFields<DIM>::NF],
                                            const int (&b)[3], const float (&f)[3], long long *acc) {
    const GlobalAdd<DIM> ad{acc, g.nodes, g.n[0], (int64_t)g.n[0] * g.n[1],
                            node_index(g, b[0], b[1], DIM == 3 ? b[2] : 0)};
    const StressP sp{0.f, 0.f, 0.f, 0.f};
    uint32_t unused = 0;
    auto rec = [&](int fi) { return rec_v[fi]; };
    return scatter_shares<DIM, false, false, true>(g, rec, f, ad, sp, unused);
}

// The fused step with one warp per work item (the P2G kernel's shape): each
// warp owns a velocity halo of its tile, an accumulator halo of the same
// tile and a double buffer of its lanes' x, m and id, so no block barrier
// couples the warps.  32 particles a round, a lane gathers its particle at x,
// writes the new state at the particle's place in bin order (coalesced; the
// order inside a tile is the input's, so a bank-class interleave written by
// the sorted G2P carries over) and scatters the new state from its
// registers: into the warp's halo while the new base cell is still in the
// tile, else straight into the global grid.
template <int DIM, int T>
__global__ void __launch_bounds__(kP2GThreads, 3)
    k_g2p2g_w(GridP g, PartsF p, PartsF q, const long long *__restrict__ accR, long long *__restrict__ accW,
              float dtg0, float dtg1, float dtg2, const uint32_t *__restrict__ perm,
              const uint32_t *__restrict__ slices, const uint32_t *__restrict__ start,
              uint32_t *__restrict__ status, float dt, float c4) {
    using Hl = HaloU<DIM, T>;
    using St = Stencil<DIM>;
    constexpr int NW = kP2GThreads / 32;
    constexpr int VW = DIM * Hl::SIZE;     // velocity words per warp
    constexpr int AW = St::NC * Hl::SIZE;  // accumulator words per warp
    constexpr int NF = DIM + 2;            // staged: x, m, id
    __shared__ float svel[NW][VW];
    __shared__ __align__(16) int32_t sacc[NW][AW];
    __shared__ float sbuf[NW][2 * NF * 32];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    float *vw = svel[warp];
    const VelHalo<DIM, T> sv{vw, vw + Hl::SIZE, DIM == 3 ? vw + 2 * Hl::SIZE : vw, nullptr};
    int32_t *wh = sacc[warp];
    float *wb = sbuf[warp];
    const uint32_t halo = (uint32_t)__cvta_generic_to_shared(wh);
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    uint32_t *work = &status[MPM_ST_WORK_G2P];
    const float dtg[3] = {dtg0, dtg1, dtg2};
    const StressP sp{0.f, 0.f, dt, 0.f};
    float smax = 0.f;
    uint32_t bad = 0, escaped = 0, unused = 0;
    for (int i = lane; i < AW; i += 32) wh[i] = 0;
    __syncwarp();
    auto at = [&](int stage, int f) { return wb + (stage * NF + f) * 32 + lane; };
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
        const uint32_t rounds = (cnt + 31) / 32;
        tile_origin(g, t, o);
        auto issue = [&](int stage, uint32_t r) {
            const uint32_t pid = perm[beg + r];
#pragma unroll
            for (int f = 0; f < DIM; ++f) cp_async4(at(stage, f), p.x[f] + pid);
            cp_async4(at(stage, DIM), p.m + pid);
            if (p.id) cp_async4(at(stage, DIM + 1), p.id + pid);
            return pid;
        };
        uint32_t pid_next = lane < cnt ? issue(0, lane) : 0u;
        cp_async_commit();
        // node velocities of the tile's halo, the grid update applied on load
        load_halo<DIM, T, false, 1, 2>(g, accR, dtg, o, vw, (int)lane, 32);
        __syncwarp();
        int stage = 0;
        for (uint32_t qr = 0; qr < rounds; ++qr) {
            const uint32_t r = qr * 32 + lane;
            const uint32_t pid = pid_next;
            if (qr + 1 < rounds && r + 32 < cnt) pid_next = issue(stage ^ 1, r + 32);
            cp_async_commit();
            cp_async_wait<1>();
            if (r < cnt) {
                const uint32_t dst = beg + r;  // bin order
                float x[DIM], f[3] = {0.f, 0.f, 0.f};
                int b[3] = {0, 0, 0};
#pragma unroll
                for (int l = 0; l < DIM; ++l) x[l] = *at(stage, l);
                const float m = *at(stage, DIM);
                const_cast<float *>(q.m)[dst] = m;
                if (q.id) q.id[dst] = __float_as_uint(*at(stage, DIM + 1));
                float rec_v[P2GFields<DIM>::NF];
                rec_v[2 * DIM + DIM * DIM] = m;
                if (!in_box_x<DIM, T>(g, x, o, b, f)) {
                    // not binned into this tile from these positions: carried as it is
#pragma unroll
                    for (int l = 0; l < DIM; ++l) {
                        rec_v[l] = x[l];
                        rec_v[DIM + l] = p.v[l][pid];
                    }
#pragma unroll
                    for (int j = 0; j < DIM * DIM; ++j) rec_v[2 * DIM + j] = p.C[j][pid];
                } else {
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
                    float sv2 = 0.f, sc2 = 0.f;
#pragma unroll
                    for (int k = 0; k < DIM; ++k) {
                        rec_v[DIM + k] = vn[k];
                        sv2 = __fadd_rn(sv2, __fmul_rn(vn[k], vn[k]));
#pragma unroll
                        for (int l = 0; l < DIM; ++l) {
                            const float c = __fmul_rn(Bm[k][l], c4);
                            rec_v[2 * DIM + k * DIM + l] = c;
                            sc2 = __fadd_rn(sc2, __fmul_rn(c, c));
                        }
                    }
                    smax = fmaxf(smax, __fadd_rn(__fsqrt_rn(sv2), __fmul_rn(__fmul_rn(1.5f, g.dx), __fsqrt_rn(sc2))));
#pragma unroll
                    for (int l = 0; l < DIM; ++l) rec_v[l] = __fmaf_rn(dt, vn[l], x[l]);
                }
#pragma unroll
                for (int l = 0; l < DIM; ++l) {
                    q.x[l][dst] = rec_v[l];
                    q.v[l][dst] = rec_v[DIM + l];
                }
#pragma unroll
                for (int j = 0; j < DIM * DIM; ++j) q.C[j][dst] = rec_v[2 * DIM + j];
                // the scatter of the new state (the P2G's arithmetic)
                auto rec = [&](int fi) { return rec_v[fi]; };
                int b2[3] = {0, 0, 0};
                float f2v[3] = {0.f, 0.f, 0.f};
                bool inside = true;
#pragma unroll
                for (int l = 0; l < DIM; ++l) inside = inside && base_frac(rec_v[l], g.inv_dx, g.n[l], b2[l], f2v[l]);
                if (inside) {
                    bool in_tile = true;
#pragma unroll
                    for (int l = 0; l < DIM; ++l) in_tile = in_tile && b2[l] >= o[l] && b2[l] < o[l] + T;
                    if (in_tile) {
                        const int hb2 = DIM == 3 ? (b2[0] - o[0]) + (b2[1] - o[1]) * Hl::SY + (b2[2] - o[2]) * Hl::SZ
                                                 : (b2[0] - o[0]) + (b2[1] - o[1]) * Hl::SY;
                        const SharedAdd<Hl> ad{halo + 4u * (uint32_t)hb2};
                        if (!scatter_shares<DIM, false, false, true>(g, rec, f2v, ad, sp, unused)) ++bad;
                    } else if (scatter_global<DIM>(g, rec_v, b2, f2v, accW)) {
                        ++escaped;
                    } else {
                        ++bad;
                    }
                }
            }
            stage ^= 1;
            // int32 accumulators: at most 512 shares below 2^22 reach one entry between two flushes
            if ((qr + 1) % 16 == 0 && qr + 1 < rounds) flush();
        }
        flush();
        s = __shfl_sync(0xFFFFFFFFu, ask, 0);
    }
    cp_async_wait<0>();
    bad = __reduce_add_sync(0xFFFFFFFFu, bad);
    escaped = __reduce_add_sync(0xFFFFFFFFu, escaped);
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(smax));
    if (lane == 0) {
        if (bad) {  // the new state does not fit 22-bit shares: this step's scatter is undone
            atomicAdd(&status[MPM_ST_N_OUT_OF_RANGE], bad);
            atomicOr(&status[MPM_ST_FLAGS], (1u << MPM_E_BOUND) | kFlagRollback);
        }
        if (escaped) atomicAdd(&status[MPM_ST_N_ESCAPED], escaped);
        if (wmax) atomicMax(&status[MPM_ST_MAX_SPEED], wmax);
    }
}

// Clears the accumulators of the node blocks that the binned tiles' stencils
// reach (the blocks the grid update visits), every channel.
template <int DIM, int T>
__global__ void k_clear_blocks(GridP g, long long *__restrict__ acc, const uint32_t *__restrict__ count) {
    constexpr int ROWS = DIM == 3 ? T * T : T;  // grid rows of one block row
    const uint32_t lane = lane_id();
    // work item: a brick of 32 nodes in x (one per lane) by one row of node blocks, as the grid update
    const uint32_t runs = ((uint32_t)g.n[0] + 31) / 32, nb1 = (uint32_t)g.nb[1];
    const uint32_t items = runs * nb1 * (DIM == 3 ? (uint32_t)g.nb[2] : 1u);
    const uint32_t warps = gridDim.x * (blockDim.x >> 5);
    for (uint32_t it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
        const uint32_t rest = it / runs;
        const int gx = (int)(it - rest * runs) * 32 + (int)lane;
        const int by = DIM == 3 ? (int)(rest % nb1) : (int)rest;
        const int bz = DIM == 3 ? (int)(rest / nb1) : 0;
        // the node's block received shares only from tiles (block - delta), delta in {0,1}^dim
        bool act = false;
        if (gx < g.n[0]) {
            const int bx = gx / T;
#pragma unroll
            for (int d = 0; d < (1 << DIM); ++d) {
                const int tx = bx - (d & 1), ty = by - ((d >> 1) & 1), tz = bz - ((d >> 2) & 1);
                if (tx >= 0 && ty >= 0 && tz >= 0 && tx < g.nt[0] && ty < g.nt[1] && (DIM == 2 || tz < g.nt[2]))
                    act = act || count[((int64_t)tz * g.nt[1] + ty) * g.nt[0] + tx] > 0;
            }
        }
        if (!act) continue;
#pragma unroll 4
        for (int r = 0; r < ROWS; ++r) {
            const int gy = by * T + r % T, gz = DIM == 3 ? bz * T + r / T : 0;
            if (gy >= g.n[1] || (DIM == 3 && gz >= g.n[2])) continue;
            const int64_t node = node_index(g, gx, gy, gz);
#pragma unroll
            for (int c = 0; c <= DIM; ++c) acc[c * g.nodes + node] = 0;
        }
    }
}

void launch_clear_blocks(const GridP &g, long long *acc, const WsView &w, const DeviceInfo &dev, cudaStream_t st) {
    if (g.dim == 3)
        k_clear_blocks<3, 4><<<dev.sms * 8, 256, 0, st>>>(g, acc, w.count);
    else
        k_clear_blocks<2, 8><<<dev.sms * 8, 256, 0, st>>>(g, acc, w.count);
}

mpm_status launch_g2p2g(const GridP &g, const PartsF &in, const PartsF &out, const WsView &w, void *acc_read,
                        void *acc_write, float dt, const float dtg[3], const DeviceInfo &dev, cudaStream_t st) {
    const float c4 = 4.0f * g.inv_dx;
    const int blocks = dev.sms * 4;
    static_assert(MPM_ST_MAX_SPEED == MPM_ST_WORK_G2P + 1, "adjacent status words");
    cudaMemsetAsync(&w.status[MPM_ST_WORK_G2P], 0, 2 * sizeof(uint32_t), st);  // work counter, max speed
    cudaMemsetAsync(&w.status[MPM_ST_N_OUT_OF_RANGE], 0, sizeof(uint32_t), st);
    const auto *R = static_cast<const long long *>(acc_read);
    auto *Wr = static_cast<long long *>(acc_write);
    if (g.dim == 3 && g.T == 4) {
        k_g2p2g_w<3, 4><<<blocks, kP2GThreads, 0, st>>>(g, in, out, R, Wr, dtg[0], dtg[1], dtg[2], w.perm,
                                                        w.slices, w.start, w.status, dt, c4);
    } else if (g.dim == 2 && g.T == 8) {
        k_g2p2g_w<2, 8><<<blocks, kP2GThreads, 0, st>>>(g, in, out, R, Wr, dtg[0], dtg[1], dtg[2], w.perm,
                                                        w.slices, w.start, w.status, dt, c4);
    } else {
        return MPM_E_ARG;
    }
    launch_copy_rest(g, in, out, w, dev, st);
    launch_clear_blocks(g, const_cast<long long *>(R), w, dev, st);
    launch_rollback(g, Wr, w.status, dev, st);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
