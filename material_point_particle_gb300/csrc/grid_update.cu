// grid_update.cu -- the grid update.
//
// Implementation guide, section 2.1 item 1 and section 3.3.2: mass-normalise,
// add gravity (rule 7: a solver parameter), apply the velocity-form boundary
// sign test; each accumulator is read once and written back to zero (section
// 2.1, "the grid clear can ride along"; rule 4).  Only node blocks next to a
// tile that holds particles are visited.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace mpm {

// Work item: a brick of 32 nodes in x (one per lane) by one row of node
// blocks (T rows in y, T planes in z), visited when a tile next to one of its
// blocks holds particles: each lane reads consecutive nodes of a grid row, so
// a warp's loads cover 256 contiguous bytes of a plane, and two rows' loads
// are in flight before any store.  A node block receives shares only from the
// tiles (block - delta), delta in {0,1}^dim.
template <int DIM, int T, typename AccT, bool VC>
__global__ void __launch_bounds__(256, 4)
    k_grid_update(GridP g, AccT *__restrict__ acc, float *__restrict__ vel, float dtg0, float dtg1, float dtg2,
                  const uint32_t *__restrict__ count) {
    constexpr int NCH = DIM + 1 + (VC ? 1 : 0);
    constexpr int ROWS = DIM == 3 ? T * T : T;  // grid rows of one block row
    constexpr int G = 2;                        // rows whose loads are in flight together
    static_assert(ROWS % G == 0, "whole row groups");
    const uint32_t lane = lane_id();
    const float dtg[3] = {dtg0, dtg1, dtg2};
    // 32-bit item arithmetic: the descriptor bounds the block count well below 2^32
    const uint32_t runs = ((uint32_t)g.n[0] + 31) / 32, nb1 = (uint32_t)g.nb[1];
    const uint32_t items = runs * nb1 * (DIM == 3 ? (uint32_t)g.nb[2] : 1u);
    const uint32_t warps = gridDim.x * (blockDim.x >> 5);
    for (uint32_t it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
        const uint32_t rest = it / runs;
        const int gx = (int)(it - rest * runs) * 32 + (int)lane;
        const int by = DIM == 3 ? (int)(rest % nb1) : (int)rest;
        const int bz = DIM == 3 ? (int)(rest / nb1) : 0;
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
        if (!__any_sync(0xFFFFFFFFu, act)) continue;
#pragma unroll 1
        for (int r0 = 0; r0 < ROWS; r0 += G) {
            AccT a[G][NCH];
            int64_t node[G];
            bool in[G];
#pragma unroll
            for (int k = 0; k < G; ++k) {
                const int gy = by * T + (r0 + k) % T, gz = DIM == 3 ? bz * T + (r0 + k) / T : 0;
                in[k] = act && gy < g.n[1] && (DIM == 2 || gz < g.n[2]);
                node[k] = in[k] ? node_index(g, gx, gy, gz) : 0;
#pragma unroll
                for (int c = 0; c < NCH; ++c) a[k][c] = in[k] ? acc[c * g.nodes + node[k]] : (AccT)0;
            }
#pragma unroll
            for (int k = 0; k < G; ++k) {
                if (!in[k]) continue;
                const int idx[3] = {gx, by * T + (r0 + k) % T, DIM == 3 ? bz * T + (r0 + k) / T : 0};
                bool any = false;
#pragma unroll
                for (int c = 0; c < NCH; ++c) any = any || a[k][c] != (AccT)0;
                const float M = acc_to_float(a[k][0]);
#pragma unroll
                for (int l = 0; l < DIM; ++l) {
                    float v = 0.f;
                    if (M != 0.f) {
                        v = __fadd_rn(__fdiv_rn(acc_to_float(a[k][1 + l]), M), dtg[l]);
                        if ((idx[l] < g.boundary && v < 0.f) || (idx[l] > g.n[l] - 1 - g.boundary && v > 0.f))
                            v = 0.f;
                    }
                    vel[l * g.nodes + node[k]] = v;
                }
                // volume fraction: the sum in cells, the fixed-point scale removed
                if constexpr (VC) vel[DIM * g.nodes + node[k]] = __fmul_rn(acc_to_float(a[k][DIM + 1]), g.inv_S);
                if (any) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c) acc[c * g.nodes + node[k]] = (AccT)0;
                }
            }
        }
    }
}

template <int DIM, int T, typename AccT>
void launch_grid_update_t(const GridP &g, void *grid_acc, float *vel, const float dtg[3], const WsView &w, int blocks,
                          cudaStream_t st) {
    if (g.vc)
        k_grid_update<DIM, T, AccT, true><<<blocks, 256, 0, st>>>(g, (AccT *)grid_acc, vel, dtg[0], dtg[1], dtg[2],
                                                                  w.count);
    else
        k_grid_update<DIM, T, AccT, false><<<blocks, 256, 0, st>>>(g, (AccT *)grid_acc, vel, dtg[0], dtg[1], dtg[2],
                                                                   w.count);
}

mpm_status launch_grid_update(const GridP &g, void *grid_acc, float *vel, const float dtg[3], const WsView &w,
                              const DeviceInfo &dev, cudaStream_t st) {
    const int blocks = dev.sms * 8;
    if (g.dim == 3 && g.T == 4) {
        if (g.acc_mode == MPM_ACC_I64)
            launch_grid_update_t<3, 4, long long>(g, grid_acc, vel, dtg, w, blocks, st);
        else if (g.acc_mode == MPM_ACC_I32)
            launch_grid_update_t<3, 4, int>(g, grid_acc, vel, dtg, w, blocks, st);
        else
            launch_grid_update_t<3, 4, float>(g, grid_acc, vel, dtg, w, blocks, st);
    } else if (g.dim == 2 && g.T == 8) {
        if (g.acc_mode == MPM_ACC_I64)
            launch_grid_update_t<2, 8, long long>(g, grid_acc, vel, dtg, w, blocks, st);
        else if (g.acc_mode == MPM_ACC_I32)
            launch_grid_update_t<2, 8, int>(g, grid_acc, vel, dtg, w, blocks, st);
        else
            launch_grid_update_t<2, 8, float>(g, grid_acc, vel, dtg, w, blocks, st);
    } else {
        return MPM_E_ARG;
    }
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
