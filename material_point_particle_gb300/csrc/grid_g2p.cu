// grid_g2p.cu -- grid-to-particle gather.
//
// G2P (implementation guide, section 1: a gather, every particle writes only itself; section 3.1
// Part 1 and 3.3.2 "gather d and D (= B*4)"): new velocity, APIC affine matrix
// C = B * 4/dx^2 in cell units, advection x += dt v; for elastic particles
// also F <- (I + dt C) F (section 3.3.2; stress.cuh).
#include "common.cuh"
#include "gather.cuh"
#include "internal.h"
#include "range.cuh"
#include "stress.cuh"

namespace mpm {

// --------------------------------------------------------------------------
// Whole-state copy of particle `src` of p to entry `dst` of q.
template <int DIM>
__device__ __forceinline__ void copy_particle(const PartsF &p, const PartsF &q, uint32_t src, uint32_t dst) {
#pragma unroll
    for (int l = 0; l < DIM; ++l) {
        q.x[l][dst] = p.x[l][src];
        q.v[l][dst] = p.v[l][src];
    }
#pragma unroll
    for (int j = 0; j < DIM * DIM; ++j) q.C[j][dst] = p.C[j][src];
    const_cast<float *>(q.m)[dst] = p.m[src];
    if (q.id && p.id) q.id[dst] = p.id[src];
    if (q.F[0] && p.F[0]) {
#pragma unroll
        for (int j = 0; j < DIM * DIM; ++j) q.F[j][dst] = p.F[j][src];
    }
    if (q.vol && p.vol) q.vol[dst] = p.vol[src];
    if (q.phi && p.phi) q.phi[dst] = p.phi[src];
}

// One particle's gather from the tile's velocity halo in shared memory.  The
// new state of particle `pid` of `p` goes to entry `dst` of `q` (the same
// arrays and index in place; the sorted output otherwise, m and id with it).
// rec(f): the particle's staged fields x[dim], then (sorted output) m and the
// id bits.  The x and y components go through packed fp32x2 arithmetic, which
// rounds each lane exactly as the scalar operation.  Elastic particles (EL)
// read F (and, sorted, vol) of `pid` from global memory and write F'; with
// the volume channel (VC) the particle's grid-recovered volume fraction is
// gathered as v is and written to phi.
template <int DIM, int T, bool MOVED, bool EL, bool VC, typename Rec>
__device__ __forceinline__ void gather_one(const GridP &g, const PartsF &p, const PartsF &q, uint32_t pid,
                                           uint32_t dst, const Rec &rec, const int o[3], const VelHalo<DIM, T> &sv,
                                           float dt, float c4, float &smax, uint32_t &rmax) {
    using Hl = HaloU<DIM, T>;
    float x[DIM], f[3] = {0.f, 0.f, 0.f};
    int b[3] = {0, 0, 0};
#pragma unroll
    for (int l = 0; l < DIM; ++l) x[l] = rec(l);
    if (!in_tile_x<DIM>(g, x, o, b, f)) {
        if constexpr (MOVED) copy_particle<DIM>(p, q, pid, dst);
        return;
    }
    [[maybe_unused]] float Fo[EL ? DIM * DIM : 1];
    if constexpr (EL) {
#pragma unroll
        for (int j = 0; j < DIM * DIM; ++j) Fo[j] = p.F[j][pid];
    }
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
    // the advective bound's term |v'| + 1.5 dx |C'|_F, sums in index order
    float sv2 = 0.f, sc2 = 0.f;
    float Cn[DIM * DIM];
#pragma unroll
    for (int k = 0; k < DIM; ++k) {
        q.v[k][dst] = vn[k];
        sv2 = __fadd_rn(sv2, __fmul_rn(vn[k], vn[k]));
#pragma unroll
        for (int l = 0; l < DIM; ++l) {
            const float c = __fmul_rn(Bm[k][l], c4);
            Cn[k * DIM + l] = c;
            q.C[k * DIM + l][dst] = c;
            sc2 = __fadd_rn(sc2, __fmul_rn(c, c));
        }
    }
    if constexpr (EL) {
        float Fn[DIM * DIM];
        advance_F<DIM>(dt, Cn, Fo, Fn);
#pragma unroll
        for (int j = 0; j < DIM * DIM; ++j) q.F[j][dst] = Fn[j];
    }
    if constexpr (MOVED && (EL || VC)) q.vol[dst] = p.vol[pid];
    if constexpr (VC) q.phi[dst] = gather_phi<DIM, T>(sv, hb, w);
    smax = fmaxf(smax, __fadd_rn(__fsqrt_rn(sv2), __fmul_rn(__fmul_rn(1.5f, g.dx), __fsqrt_rn(sc2))));
    // the range the next P2G's bound may take from this record: max(1, |v'_k| + 1.5 dx sum_l |C'_kl|)
    rmax = max(rmax, range_r_bits<DIM>(vn, Cn, __fmul_rn(1.5f, g.dx)));
#pragma unroll
    for (int l = 0; l < DIM; ++l) q.x[l][dst] = __fmaf_rn(dt, vn[l], x[l]);
    if constexpr (MOVED) {
        const_cast<float *>(q.m)[dst] = rec(DIM);
        if (q.id) q.id[dst] = __float_as_uint(rec(DIM + 1));
    }
}


// The sorted G2P.  Work item as in P2G: one slice of a tile.  The CTA stages
// the tile's halo of node velocities in shared memory, the slice's x, m and
// id in bin order, and counting-sorts the slice by bank class; thread t then
// computes the particles that go to places t, t + 256, ... of the interleaved
// slice, so that its writes are coalesced and its reads of the velocity halo
// meet few bank conflicts.  A slice of at most 32 particles is one round and
// keeps bin order.
template <int DIM, int T, bool EL, bool VC>
__global__ void __launch_bounds__(kG2PThreads) k_g2p(GridP g, PartsF p, PartsF q, const float *__restrict__ vel,
                                                     const uint32_t *__restrict__ perm,
                                                     const uint32_t *__restrict__ key,
                                                     const uint32_t *__restrict__ slices,
                                                     const uint32_t *__restrict__ start,
                                                     uint32_t *__restrict__ status, float dt, float c4) {
    using Hl = HaloU<DIM, T>;
    constexpr int NQ = kSliceParticles / kG2PThreads;
    constexpr int NWARP = kG2PThreads / 32;
    static_assert(NQ * NWARP == 32, "one warp-scan lane per (round, warp)");
    constexpr int NF = DIM + 2;  // x, m, id of the whole slice
    constexpr int BUF = NF * kSliceParticles;
    __shared__ float sv_x[Hl::SIZE], sv_y[Hl::SIZE], sv_z[DIM == 3 ? Hl::SIZE : 1], sv_phi[VC ? Hl::SIZE : 1];
    const VelHalo<DIM, T> sv{sv_x, sv_y, sv_z, sv_phi};
    __shared__ float sbuf[BUF];
    // [(qi, warp)][class], rows padded to 33 words: the scan reads a column
    __shared__ uint32_t hist[NQ * NWARP * 33];
    __shared__ uint32_t cstart[32];
    // sorted entry e -> bin-order entry, at e + e / 32: the interleaved reads
    // take entries R apart
    __shared__ uint32_t order[kSliceParticles + kSliceParticles / 32];
    const uint32_t lane = lane_id();
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    __shared__ uint32_t item_sh;
    float smax = 0.f;  // the advective bound's largest term among this thread's particles
    uint32_t rmax = 0;  // the range record's largest term
    uint32_t next = 0;
    for (uint32_t s = grab_item(&status[MPM_ST_WORK_G2P], &item_sh); s < nslices; s = publish_item(next, &item_sh)) {
        next = ask_item(&status[MPM_ST_WORK_G2P]);
        const uint32_t t = slices[2 * (size_t)s], first = slices[2 * (size_t)s + 1];
        const uint32_t beg = start[t] + first;
        const uint32_t cnt = min((uint32_t)kSliceParticles, start[t + 1] - beg);
        int o[3];
        tile_origin(g, t, o);
        uint32_t pids[NQ];
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            const uint32_t r = threadIdx.x + qi * kG2PThreads;
            pids[qi] = r < cnt ? perm[beg + r] : 0u;
        }
        // the slice's x, m, id in bin order
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            const uint32_t r = threadIdx.x + qi * kG2PThreads;
            if (r < cnt) {
#pragma unroll
                for (int f = 0; f < DIM; ++f) cp_async4(&sbuf[f * kSliceParticles + r], p.x[f] + pids[qi]);
                cp_async4(&sbuf[DIM * kSliceParticles + r], p.m + pids[qi]);
                if (p.id) cp_async4(&sbuf[(DIM + 1) * kSliceParticles + r], p.id + pids[qi]);
            }
        }
        cp_async_commit();
        for (int h = threadIdx.x; h < Hl::NODES; h += blockDim.x) {
            int hx, hy, hz;
            Hl::node(h, hx, hy, hz);
            const int gx = o[0] + hx, gy = o[1] + hy, gz = o[2] + hz;
            const bool in = gx < g.n[0] && gy < g.n[1] && (DIM == 2 || gz < g.n[2]);
            const int64_t node = in ? node_index(g, gx, gy, gz) : 0;
            sv_x[h] = in ? vel[node] : 0.f;
            sv_y[h] = in ? vel[g.nodes + node] : 0.f;
            if (DIM == 3) sv_z[h] = in ? vel[2 * g.nodes + node] : 0.f;
            if (VC) sv_phi[h] = in ? vel[DIM * g.nodes + node] : 0.f;
        }
        if (cnt <= 32u) {
            // one round: the order inside it does not matter, bin order is kept
            cp_async_wait<0>();
            __syncthreads();
            if (threadIdx.x < cnt) {
                const uint32_t r = threadIdx.x;
                auto rec = [&](int f) { return sbuf[f * kSliceParticles + r]; };
                gather_one<DIM, T, true, EL, VC>(g, p, q, pids[0], beg + r, rec, o, sv, dt, c4, smax, rmax);
            }
        } else {
            class_order<DIM, T, kG2PThreads>(key, pids, cnt, hist, cstart, order);
            cp_async_wait<0>();
            __syncthreads();
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                const uint32_t pos = threadIdx.x + qi * kG2PThreads;
                if (pos < cnt) {
                    const uint32_t e = interleave_entry(pos, cnt);
                    const uint32_t r = order[e + (e >> 5)];
                    auto rec = [&](int f) { return sbuf[f * kSliceParticles + r]; };
                    gather_one<DIM, T, true, EL, VC>(g, p, q, perm[beg + r], beg + pos, rec, o, sv, dt, c4, smax, rmax);
                }
            }
        }
    }
    // non-negative fp32 values order as their bit patterns
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(smax));
    if (lane == 0 && wmax) atomicMax(&status[MPM_ST_MAX_SPEED], wmax);
    warp_max_to(rmax, &status[MPM_ST_G2P_RANGE]);
}

// G2P with one warp per work item (the P2G kernel's shape), in place or in
// bin order.  Each warp stages its tile's velocity halo in shared memory and
// takes 32 particles a round; each lane gathers its particle (gather_one, the
// same arithmetic).  In place, the new state overwrites the particle's own
// entry (the mpm_g2p contract), and each lane loads its next particle's
// position into registers while the current one gathers.  In bin order
// (BINORDER), out[j] = the new state of in[perm[j]]: x, m and id are copied
// into a per-warp double buffer in shared memory a round ahead, and
// consecutive lanes write consecutive places.  No block barrier couples the
// warps.
template <int DIM, int T, bool BINORDER, bool EL, bool VC>
__global__ void __launch_bounds__(kP2GThreads) k_g2p_w(GridP g, PartsF p, PartsF q, const float *__restrict__ vel,
                                                       const uint32_t *__restrict__ perm,
                                                       const uint32_t *__restrict__ slices,
                                                       const uint32_t *__restrict__ start,
                                                       uint32_t *__restrict__ status, float dt, float c4) {
    using Hl = HaloU<DIM, T>;
    constexpr int NW = kP2GThreads / 32;
    constexpr int NCH = DIM + (VC ? 1 : 0);
    constexpr int NF = BINORDER ? DIM + 2 : DIM;  // staged: x (and m, id)
    __shared__ float svel[NW][NCH * Hl::SIZE];
    __shared__ float sbuf[NW][BINORDER ? 2 * NF * 32 : 1];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    float *vw = svel[warp];
    const VelHalo<DIM, T> sv{vw, vw + Hl::SIZE, DIM == 3 ? vw + 2 * Hl::SIZE : vw, VC ? vw + DIM * Hl::SIZE : vw};
    float *wb = sbuf[warp];
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    uint32_t *work = &status[MPM_ST_WORK_G2P];
    float smax = 0.f;
    uint32_t rmax = 0;
    auto at = [&](int stage, int f) { return wb + (stage * NF + f) * 32 + lane; };
    uint32_t s = 0;
    if (lane == 0) s = atomicAdd(work, 1u);
    s = __shfl_sync(0xFFFFFFFFu, s, 0);
    while (s < nslices) {
        const uint32_t ask = lane == 0 ? atomicAdd(work, 1u) : 0u;
        const uint32_t t = slices[2 * (size_t)s];
        const uint32_t beg = start[t] + slices[2 * (size_t)s + 1];
        const uint32_t cnt = min((uint32_t)kSliceParticles, start[t + 1] - beg);
        int o[3];
        tile_origin(g, t, o);
        auto issue = [&](int stage, uint32_t r) {
            const uint32_t pid = perm[beg + r];
#pragma unroll
            for (int f = 0; f < DIM; ++f) cp_async4(at(stage, f), p.x[f] + pid);
            if constexpr (BINORDER) {
                cp_async4(at(stage, DIM), p.m + pid);
                if (p.id) cp_async4(at(stage, DIM + 1), p.id + pid);
            }
            return pid;
        };
        uint32_t pid_next = 0u;
        if constexpr (BINORDER) {
            pid_next = lane < cnt ? issue(0, lane) : 0u;
            cp_async_commit();
        }
        for (int h = lane; h < Hl::NODES; h += 32) {
            int hx, hy, hz;
            Hl::node(h, hx, hy, hz);
            const int gx = o[0] + hx, gy = o[1] + hy, gz = o[2] + hz;
            const bool in = gx < g.n[0] && gy < g.n[1] && (DIM == 2 || gz < g.n[2]);
            const int64_t node = in ? node_index(g, gx, gy, gz) : 0;
#pragma unroll
            for (int c = 0; c < NCH; ++c) vw[c * Hl::SIZE + h] = in ? vel[c * g.nodes + node] : 0.f;
        }
        __syncwarp();
        const uint32_t rounds = (cnt + 31) / 32;
        if constexpr (!BINORDER) {
            // in place: positions in registers a round ahead, perm two rounds ahead
            uint32_t pid = lane < cnt ? perm[beg + lane] : 0u;
            pid_next = lane + 32 < cnt ? perm[beg + lane + 32] : 0u;
            float xc[DIM], xn[DIM];
#pragma unroll
            for (int l = 0; l < DIM; ++l) xc[l] = lane < cnt ? p.x[l][pid] : 0.f;
            for (uint32_t qr = 0; qr < rounds; ++qr) {
                const uint32_t r = qr * 32 + lane;
#pragma unroll
                for (int l = 0; l < DIM; ++l) xn[l] = r + 32 < cnt ? p.x[l][pid_next] : 0.f;
                const uint32_t pid_after = r + 64 < cnt ? perm[beg + r + 64] : 0u;
                if (r < cnt) {
                    auto rec = [&](int f) { return xc[f]; };
                    gather_one<DIM, T, false, EL, VC>(g, p, q, pid, pid, rec, o, sv, dt, c4, smax, rmax);
                }
#pragma unroll
                for (int l = 0; l < DIM; ++l) xc[l] = xn[l];
                pid = pid_next;
                pid_next = pid_after;
            }
        } else {
            // bin order: x, m and id copied into shared memory (cp.async) a round ahead
            int stage = 0;
            for (uint32_t qr = 0; qr < rounds; ++qr) {
                const uint32_t r = qr * 32 + lane;
                const uint32_t pid = pid_next;
                if (qr + 1 < rounds && r + 32 < cnt) pid_next = issue(stage ^ 1, r + 32);
                cp_async_commit();
                cp_async_wait<1>();
                if (r < cnt) {
                    const int st = stage;
                    auto rec = [&](int f) { return *at(st, f); };
                    gather_one<DIM, T, BINORDER, EL, VC>(g, p, q, pid, BINORDER ? beg + r : pid, rec, o, sv, dt, c4,
                                                         smax, rmax);
                }
                stage ^= 1;
            }
        }
        __syncwarp();
        s = __shfl_sync(0xFFFFFFFFu, ask, 0);
    }
    cp_async_wait<0>();
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(smax));
    if (lane == 0 && wmax) atomicMax(&status[MPM_ST_MAX_SPEED], wmax);
    warp_max_to(rmax, &status[MPM_ST_G2P_RANGE]);
}

// Particles past the sorted in-domain part (outside the domain): copied.
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
        k_g2p<DIM, T, EL, VC><<<dev.sms * (1024 / kG2PThreads), kG2PThreads, 0, st>>>(
            g, in, out, vel, w.perm, w.key, w.slices, w.start, w.status, dt, c4);
    else
        k_g2p_w<DIM, T, OUT == kBinOrder, EL, VC><<<dev.sms * 4, kP2GThreads, 0, st>>>(
            g, in, out, vel, w.perm, w.slices, w.start, w.status, dt, c4);
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
