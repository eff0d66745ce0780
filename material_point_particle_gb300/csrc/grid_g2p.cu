// grid_g2p.cu -- grid-to-particle gather from the velocity grid (the G2P
// kernels are in g2p_kernels.cuh), the copy of the particles outside the
// domain, the permutation of a particle set, and the integer cloud-in-cell
// gather.
#include "g2p_kernels.cuh"

namespace mpm {

template <int DIM>
__global__ void k_copy_rest(PartsF p, PartsF q, const uint32_t *__restrict__ perm, const uint32_t *__restrict__ status) {
    for (int64_t j = (int64_t)status[MPM_ST_N_VALID] + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < p.n;
         j += (int64_t)gridDim.x * blockDim.x)
        copy_particle<DIM>(p, q, perm[j], (uint32_t)j);
}

void launch_copy_rest(const GridP &g, const PartsF &in, const PartsF &out, const WsView &w, const DeviceInfo &dev,
                      cudaStream_t st) {
    if (g.dim == 3)
        k_copy_rest<3><<<dev.sms, 256, 0, st>>>(in, out, w.perm, w.status);
    else
        k_copy_rest<2><<<dev.sms, 256, 0, st>>>(in, out, w.perm, w.status);
}

// Where G2P writes the new state: in place (out = in), in bin order
// (out[j] = new state of in[perm[j]]), or sorted (bin order with the
// bank-class interleave inside each slice).
enum G2POut { kInPlace, kBinOrder, kSorted };

template <int DIM, int T, int OUT, bool EL, bool VC>
void launch_g2p_t(const GridP &g, const float *vel, const PartsF &in, const PartsF &out, const WsView &w, float dt,
                  const DeviceInfo &dev, cudaStream_t st) {
    const float c4 = 4.0f * g.inv_dx;  // one fp32 rounding, as the oracle
    if constexpr (OUT == kSorted)
        k_g2p<DIM, T, EL, VC, 0><<<dev.sms * (1024 / kG2PThreads), kG2PThreads, 0, st>>>(
            g, in, out, vel, 0.f, 0.f, 0.f, nullptr, w.count, w.perm, w.key, w.slices, w.start, w.status, dt, c4);
    else
        k_g2p_w<DIM, T, OUT == kBinOrder, EL, VC, 0><<<dev.sms * 4, kP2GThreads, 0, st>>>(
            g, in, out, vel, 0.f, 0.f, 0.f, nullptr, w.count, w.perm, w.slices, w.start, w.status, dt, c4);
    if constexpr (OUT != kInPlace) k_copy_rest<DIM><<<dev.sms, 256, 0, st>>>(in, out, w.perm, w.status);
}

template <int DIM, int T, int OUT>
void launch_g2p_dt(const GridP &g, const float *vel, const PartsF &in, const PartsF &out, const WsView &w, float dt,
                   const DeviceInfo &dev, cudaStream_t st) {
    const bool el = in.F[0] != nullptr;
    if (el && g.vc)
        launch_g2p_t<DIM, T, OUT, true, true>(g, vel, in, out, w, dt, dev, st);
    else if (el)
        launch_g2p_t<DIM, T, OUT, true, false>(g, vel, in, out, w, dt, dev, st);
    else if (g.vc)
        launch_g2p_t<DIM, T, OUT, false, true>(g, vel, in, out, w, dt, dev, st);
    else
        launch_g2p_t<DIM, T, OUT, false, false>(g, vel, in, out, w, dt, dev, st);
}

template <int OUT>
mpm_status launch_g2p_any(const GridP &g, const float *vel, const PartsF &in, const PartsF &out, const WsView &w,
                          float dt, const DeviceInfo &dev, cudaStream_t st) {
    static_assert(MPM_ST_MAX_SPEED == MPM_ST_WORK_G2P + 1, "adjacent status words");
    cudaMemsetAsync(&w.status[MPM_ST_WORK_G2P], 0, 2 * sizeof(uint32_t), st);  // work counter, max speed
    cudaMemsetAsync(&w.status[MPM_ST_G2P_RANGE], 0, sizeof(uint32_t), st);
    if (g.dim == 3 && g.T == 4)
        launch_g2p_dt<3, 4, OUT>(g, vel, in, out, w, dt, dev, st);
    else if (g.dim == 2 && g.T == 8)
        launch_g2p_dt<2, 8, OUT>(g, vel, in, out, w, dt, dev, st);
    else
        return MPM_E_ARG;
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

mpm_status launch_g2p_binned(const GridP &g, const float *vel, const PartsF &in, const PartsF &out, const WsView &w,
                             float dt, const DeviceInfo &dev, cudaStream_t st) {
    return launch_g2p_any<kBinOrder>(g, vel, in, out, w, dt, dev, st);
}

mpm_status launch_g2p(const GridP &g, const float *vel, const PartsF &p, const WsView &w, float dt,
                      const DeviceInfo &dev, cudaStream_t st) {
    return launch_g2p_any<kInPlace>(g, vel, p, p, w, dt, dev, st);
}

mpm_status launch_g2p_sorted(const GridP &g, const float *vel, const PartsF &in, const PartsF &out, const WsView &w,
                             float dt, const DeviceInfo &dev, cudaStream_t st) {
    return launch_g2p_any<kSorted>(g, vel, in, out, w, dt, dev, st);
}

// --------------------------------------------------------------------------
__global__ void k_permute(int ncomp, PartsF in, PartsF out, const uint32_t *__restrict__ perm, int64_t n) {
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t src = perm[j];
        for (int c = 0; c < ncomp; ++c) {
            const float *s;
            float *d;
            if (c < 3) {
                s = in.x[c];
                d = out.x[c];
            } else if (c < 6) {
                s = in.v[c - 3];
                d = out.v[c - 3];
            } else if (c < 15) {
                s = in.C[c - 6];
                d = out.C[c - 6];
            } else if (c == 15) {
                s = in.m;
                d = const_cast<float *>(out.m);
            } else if (c < 25) {
                s = in.F[c - 16];
                d = out.F[c - 16];
            } else if (c == 25) {
                s = in.vol;
                d = out.vol;
            } else {
                s = in.phi;
                d = out.phi;
            }
            if (s && d) d[j] = s[src];
        }
        if (in.id && out.id) out.id[j] = in.id[src];
    }
}

mpm_status launch_permute(const GridP &g, const PartsF &in, const PartsF &out, const uint32_t *perm,
                          const DeviceInfo &dev, cudaStream_t st) {
    const int blocks = dev.sms * 8;
    k_permute<<<blocks, 256, 0, st>>>(27, in, out, perm, in.n);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

// --------------------------------------------------------------------------
__device__ __forceinline__ long long div_rne_g(long long a, long long b) {
    long long q = a / b, r = a % b;
    unsigned long long ar = r < 0 ? 0ull - (unsigned long long)r : (unsigned long long)r;
    unsigned long long br = b < 0 ? 0ull - (unsigned long long)b : (unsigned long long)b;
    unsigned long long other = br - ar;
    if (ar > other || (ar == other && (q & 1))) q += ((a < 0) != (b < 0)) ? -1 : 1;
    return q;
}

template <int DIM>
__global__ void k_cic_gather(GridP g, PartsI p, const int64_t *__restrict__ acc) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += (int64_t)gridDim.x * blockDim.x) {
        int c[3] = {0, 0, 0};
        bool on_grid = true;
#pragma unroll
        for (int l = 0; l < DIM; ++l) {
            const int32_t X = p.X[l][i];
            c[l] = X >> 16;
            on_grid = on_grid && X >= 0 && c[l] <= g.n[l] - 2;
        }
        if (!on_grid) continue;  // positions off the grid: left unchanged
        long long M = 0, P[DIM];
#pragma unroll
        for (int k = 0; k < DIM; ++k) P[k] = 0;
#pragma unroll
        for (int s = 0; s < (1 << DIM); ++s) {
            const int64_t node = node_index(g, c[0] + (s & 1), c[1] + ((s >> 1) & 1), DIM == 3 ? c[2] + ((s >> 2) & 1) : 0);
            M += acc[node];
#pragma unroll
            for (int k = 0; k < DIM; ++k) P[k] += acc[(1 + k) * g.nodes + node];
        }
#pragma unroll
        for (int k = 0; k < DIM; ++k) p.v[k][i] = M != 0 ? div_rne_g(P[k], M) : 0;
    }
}

mpm_status launch_cic_int_gather(const GridP &g, const PartsI &p, const int64_t *acc, const DeviceInfo &dev,
                                 cudaStream_t st) {
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((p.n + 255) / 256, dev.sms * 4));
    if (g.dim == 3)
        k_cic_gather<3><<<blocks, 256, 0, st>>>(g, p, acc);
    else
        k_cic_gather<2><<<blocks, 256, 0, st>>>(g, p, acc);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
