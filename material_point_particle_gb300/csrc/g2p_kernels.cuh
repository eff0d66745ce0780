// g2p_kernels.cuh -- the G2P kernel (the gather of one particle, one warp per
// work item, in place, in bin order or sorted with the bank-class
// interleave), templated on where the node velocities come from (gather.cuh,
// load_halo): the velocity grid, or the accumulators with the grid
// update applied as the halo loads.  Included by grid_g2p.cu (the velocity
// grid) and g2p_update.cu (the accumulators), so that the two sets of
// instances compile in parallel.
//
// G2P (implementation guide, section 1: a gather, every particle writes only
// itself; section 3.1 Part 1 and 3.3.2 "gather d and D (= B*4)"): new
// velocity, APIC affine matrix C = B * 4/dx^2 in cell units, advection
// x += dt v; for elastic particles also F <- (I + dt C) F (section 3.3.2;
// stress.cuh).
#pragma once

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


// Warp-level stable counting sort of a slice of cnt (> 32) binned particles
// (perm[beg ..]) by the bank class of their base cells: ord[e + e / 32] = the
// bin-order index of the e-th entry of the class-sorted slice, stable in bin
// order.  cls: cnt bytes, cbase: 32 words, all the warp's own shared
// memory.
template <int DIM, int T>
__device__ __forceinline__ void warp_class_order(const uint32_t *__restrict__ key, const uint32_t *__restrict__ perm,
                                                 uint32_t beg, uint32_t cnt, uint8_t *cls, uint32_t *cbase,
                                                 uint16_t *ord, uint32_t lane) {
    cbase[lane] = 0;
    __syncwarp();
    // classes, and the count of each
    for (uint32_t r0 = 0; r0 < cnt; r0 += 32) {
        const uint32_t r = r0 + lane;
        const bool live = r < cnt;
        const uint32_t c = live ? cell_class<DIM, T>(key[perm[beg + r]]) : 32u + lane;  // dead lanes: alone
        if (live) cls[r] = (uint8_t)c;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, c);
        if (live && (peers & lanemask_lt()) == 0) cbase[c] += (uint32_t)__popc(peers);
        __syncwarp();
    }
    // each class's first place: exclusive scan over the 32 classes
    const uint32_t v = cbase[lane];
    uint32_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if ((int)lane >= d) inc += t2;
    }
    __syncwarp();
    cbase[lane] = inc - v;
    __syncwarp();
    // places, in bin order within each class
    for (uint32_t r0 = 0; r0 < cnt; r0 += 32) {
        const uint32_t r = r0 + lane;
        const bool live = r < cnt;
        const uint32_t c = live ? (uint32_t)cls[r] : 32u + lane;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, c);
        const uint32_t below = (uint32_t)__popc(peers & lanemask_lt());
        if (live) {
            const uint32_t e = cbase[c] + below;
            ord[e + (e >> 5)] = (uint16_t)r;
        }
        __syncwarp();
        if (live && below == 0) cbase[c] += (uint32_t)__popc(peers);
        __syncwarp();
    }
}

// Where the warp G2P writes the new state: in place, in bin order
// (out[j] = new state of in[perm[j]]), or sorted (bin order with the
// bank-class interleave inside each slice).
enum WarpOrder { kWarpInPlace = 0, kWarpBinOrder = 1, kWarpSorted = 2 };

// G2P with one warp per work item (the P2G kernel's shape), in place, in
// bin order or sorted.  Each warp stages its tile's velocity halo in shared
// memory and takes 32 particles a round; each lane gathers its particle
// (gather_one, the same arithmetic).  In place, the new state overwrites the
// particle's own entry (the mpm_g2p contract), and each lane loads its next
// particle's position into registers while the current one gathers.  In bin
// order, place j of the slice takes the particle of bin-order index j; sorted,
// place j takes the one the interleave puts there (warp_class_order, then
// interleave_entry; a slice of at most 32 keeps bin order).  Either way x, m
// and id are copied into a per-warp double buffer in shared memory a round
// ahead, and consecutive lanes write consecutive places.  No block barrier
// couples the warps.
// Threads per block of k_g2p_w: sorted, four warps (each warp's shared
// memory holds the interleave's order too).
template <int ORDER>
__host__ __device__ constexpr int g2p_w_threads() {
    return ORDER == 2 ? 128 : kP2GThreads;
}

template <int DIM, int T, int ORDER, bool EL, bool VC, int UPD>
__global__ void __launch_bounds__(g2p_w_threads<ORDER>()) k_g2p_w(GridP g, PartsF p, PartsF q, const void *__restrict__ src,
                                                       float dtg0, float dtg1, float dtg2,
                                                       uint32_t *__restrict__ readers,
                                                       const uint32_t *__restrict__ count,
                                                       const uint32_t *__restrict__ perm,
                                                       const uint32_t *__restrict__ key,
                                                       const uint32_t *__restrict__ slices,
                                                       const uint32_t *__restrict__ start,
                                                       uint32_t *__restrict__ status, float dt, float c4) {
    using Hl = HaloU<DIM, T>;
    constexpr bool MOVED = ORDER != kWarpInPlace;
    constexpr bool SORTED = ORDER == kWarpSorted;
    constexpr int NW = g2p_w_threads<ORDER>() / 32;
    constexpr int NCH = DIM + (VC ? 1 : 0);
    constexpr int NF = MOVED ? DIM + 2 : DIM;  // staged: x (and m, id)
    __shared__ float svel[NW][NCH * Hl::SIZE];
    __shared__ float sbuf[NW][MOVED ? 2 * NF * 32 : 1];
    // sorted: the interleave's order, the classes, the class counters
    __shared__ uint16_t sord[SORTED ? NW : 1][SORTED ? kSliceParticles + kSliceParticles / 32 : 1];
    __shared__ uint8_t scls[SORTED ? NW : 1][SORTED ? kSliceParticles : 1];
    __shared__ uint32_t scb[SORTED ? NW : 1][32];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    float *vw = svel[warp];
    const VelHalo<DIM, T> sv{vw, vw + Hl::SIZE, DIM == 3 ? vw + 2 * Hl::SIZE : vw, VC ? vw + DIM * Hl::SIZE : vw};
    float *wb = sbuf[warp];
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    uint32_t *work = &status[MPM_ST_WORK_G2P];
    [[maybe_unused]] const float dtg[3] = {dtg0, dtg1, dtg2};
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
        // bin-order index of the particle that goes to place pos of the slice
        [[maybe_unused]] const bool interleaved = SORTED && cnt > 32u;
        auto source = [&](uint32_t pos) -> uint32_t {
            if constexpr (SORTED) {
                if (interleaved) {
                    const uint32_t e = interleave_entry(pos, cnt);
                    return sord[warp][e + (e >> 5)];
                }
            }
            return pos;
        };
        auto issue = [&](int stage, uint32_t pos) {
            const uint32_t pid = perm[beg + source(pos)];
#pragma unroll
            for (int f = 0; f < DIM; ++f) cp_async4(at(stage, f), p.x[f] + pid);
            if constexpr (MOVED) {
                cp_async4(at(stage, DIM), p.m + pid);
                if (p.id) cp_async4(at(stage, DIM + 1), p.id + pid);
            }
            return pid;
        };
        if constexpr (SORTED)
            if (interleaved) warp_class_order<DIM, T>(key, perm, beg, cnt, scls[warp], scb[warp], sord[warp], lane);
        uint32_t pid_next = 0u;
        if constexpr (MOVED) {
            pid_next = lane < cnt ? issue(0, lane) : 0u;
            cp_async_commit();
        }
        load_halo<DIM, T, VC, UPD>(g, src, dtg, o, vw, (int)lane, 32);
        __syncwarp();
        if constexpr (UPD != 0) {
            using AccT = typename AccOf<UPD>::T;
            release_blocks<DIM, T, AccT, DIM + 1 + (VC ? 1 : 0)>(g, t, readers, count,
                                                                 const_cast<AccT *>(static_cast<const AccT *>(src)),
                                                                 lane);
        }
        const uint32_t rounds = (cnt + 31) / 32;
        if constexpr (!MOVED) {
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
            // x, m and id copied into shared memory (cp.async) a round ahead
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
                    gather_one<DIM, T, true, EL, VC>(g, p, q, pid, beg + r, rec, o, sv, dt, c4, smax, rmax);
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

}  // namespace mpm
