// g2p_update.cu -- G2P with the grid update applied as each tile's halo loads
// (implementation guide, section 2.1, the worked shape: the load is the grid
// pass; "the grid clear can ride along"): the G2P kernels of g2p_kernels.cuh
// reading the P2G accumulators instead of a velocity grid, and clearing them
// as they go, so that neither a grid-update pass nor a velocity grid is
// needed.  The bits of every particle are those of mpm_grid_update followed
// by mpm_g2p (or mpm_g2p_sorted).
#include "g2p_kernels.cuh"

namespace mpm {

template <int DIM, int T, bool SORTED, bool EL, bool VC, int UPD>
void launch_g2p_update_t(const GridP &g, const void *acc, const float dtg[3], const PartsF &in, const PartsF &out,
                         const WsView &w, float dt, bool next_keys, const DeviceInfo &dev, cudaStream_t st) {
    const float c4 = 4.0f * g.inv_dx;  // one fp32 rounding, as the oracle
    if constexpr (SORTED) {
        k_g2p<DIM, T, EL, VC, UPD><<<dev.sms * (1024 / kG2PThreads), kG2PThreads, 0, st>>>(
            g, in, out, acc, dtg[0], dtg[1], dtg[2], w.readers, w.count, w.perm, w.key, w.slices, w.start, w.status,
            dt, c4);
        launch_copy_rest(g, in, out, w, dev, st);
    } else {
        if constexpr (UPD == 1) {
            if (next_keys) {
                // the histogram of the next keys: the particles outside the domain stay there, with their count
                const int64_t nb = g.ntiles + 1;
                cudaMemsetAsync(w.count_next, 0, g.ntiles * sizeof(uint32_t), st);
                cudaMemcpyAsync(&w.count_next[nb - 1], &w.count[nb - 1], sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                                st);
                k_g2p_w<DIM, T, false, EL, VC, UPD, true><<<dev.sms * 4, kP2GThreads, 0, st>>>(
                    g, in, out, acc, dtg[0], dtg[1], dtg[2], w.readers, w.count, w.perm, w.slices, w.start, w.status,
                    dt, c4, w.key, w.count_next);
                return;
            }
        }
        k_g2p_w<DIM, T, false, EL, VC, UPD><<<dev.sms * 4, kP2GThreads, 0, st>>>(
            g, in, out, acc, dtg[0], dtg[1], dtg[2], w.readers, w.count, w.perm, w.slices, w.start, w.status, dt, c4);
    }
}

template <int DIM, int T, bool SORTED, int UPD>
void launch_g2p_update_m(const GridP &g, const void *acc, const float dtg[3], const PartsF &in, const PartsF &out,
                         const WsView &w, float dt, bool next_keys, const DeviceInfo &dev, cudaStream_t st) {
    const bool el = in.F[0] != nullptr;
    if (el && g.vc)
        launch_g2p_update_t<DIM, T, SORTED, true, true, UPD>(g, acc, dtg, in, out, w, dt, next_keys, dev, st);
    else if (el)
        launch_g2p_update_t<DIM, T, SORTED, true, false, UPD>(g, acc, dtg, in, out, w, dt, next_keys, dev, st);
    else if (g.vc)
        launch_g2p_update_t<DIM, T, SORTED, false, true, UPD>(g, acc, dtg, in, out, w, dt, next_keys, dev, st);
    else
        launch_g2p_update_t<DIM, T, SORTED, false, false, UPD>(g, acc, dtg, in, out, w, dt, next_keys, dev, st);
}

template <int DIM, int T, bool SORTED>
void launch_g2p_update_d(const GridP &g, const void *acc, const float dtg[3], const PartsF &in, const PartsF &out,
                         const WsView &w, float dt, bool next_keys, const DeviceInfo &dev, cudaStream_t st) {
    if (g.acc_mode == MPM_ACC_I64)
        launch_g2p_update_m<DIM, T, SORTED, 1>(g, acc, dtg, in, out, w, dt, next_keys, dev, st);
    else
        launch_g2p_update_m<DIM, T, SORTED, 2>(g, acc, dtg, in, out, w, dt, false, dev, st);
}

mpm_status launch_g2p_update(const GridP &g, const void *acc, const float dtg[3], const PartsF &in, const PartsF &out,
                             const WsView &w, float dt, bool sorted, bool next_keys, const DeviceInfo &dev,
                             cudaStream_t st) {
    if (g.acc_mode != MPM_ACC_I64 && g.acc_mode != MPM_ACC_I32) return MPM_E_ARG;
    static_assert(MPM_ST_MAX_SPEED == MPM_ST_WORK_G2P + 1, "adjacent status words");
    cudaMemsetAsync(&w.status[MPM_ST_WORK_G2P], 0, 2 * sizeof(uint32_t), st);  // work counter, max speed
    cudaMemsetAsync(&w.status[MPM_ST_G2P_RANGE], 0, sizeof(uint32_t), st);
    cudaMemsetAsync(w.readers, 0, (size_t)g.nblocks * sizeof(uint32_t), st);
    if (g.dim == 3 && g.T == 4) {
        if (sorted)
            launch_g2p_update_d<3, 4, true>(g, acc, dtg, in, out, w, dt, false, dev, st);
        else
            launch_g2p_update_d<3, 4, false>(g, acc, dtg, in, out, w, dt, next_keys, dev, st);
    } else if (g.dim == 2 && g.T == 8) {
        if (sorted)
            launch_g2p_update_d<2, 8, true>(g, acc, dtg, in, out, w, dt, false, dev, st);
        else
            launch_g2p_update_d<2, 8, false>(g, acc, dtg, in, out, w, dt, next_keys, dev, st);
    } else {
        return MPM_E_ARG;
    }
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
