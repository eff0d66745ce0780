// g2p_kernels.cuh -- the G2P kernels (the gather of one particle, the sorted
// kernel with one block per work item, the warp kernel in place or in bin
// order), templated on where the node velocities come from (gather.cuh,
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
// gathered as v is and written to phi.  xo: the particle's position after the
// call (the new one when it moved).
template <int DIM, int T, bool MOVED, bool EL, bool VC, typename Rec>
__device__ __forceinline__ void gather_one(const GridP &g, const PartsF &p, const PartsF &q, uint32_t pid,
                                           uint32_t dst, const Rec &rec, const int o[3], const VelHalo<DIM, T> &sv,
                                           float dt, float c4, float &smax, uint32_t &rmax, float (&xo)[DIM]) {
    using Hl = HaloU<DIM, T>;
    float x[DIM], f[3] = {0.f, 0.f, 0.f};
    int b[3] = {0, 0, 0};
#pragma unroll
    for (int l = 0; l < DIM; ++l) xo[l] = x[l] = rec(l);
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
    for (int l = 0; l < DIM; ++l) q.x[l][dst] = xo[l] = __fmaf_rn(dt, vn[l], x[l]);
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
// UPD (load_halo): node velocities from the velocity grid (0) or from
// the accumulators with the grid update applied on load (1: int64, 2: int32),
// the accumulators then cleared as the G2P goes (release_blocks).
template <int DIM, int T, bool EL, bool VC, int UPD>
__global__ void __launch_bounds__(kG2PThreads) k_g2p(GridP g, PartsF p, PartsF q, const void *__restrict__ src,
                                                     float dtg0, float dtg1, float dtg2,
                                                     uint32_t *__restrict__ readers,
                                                     const uint32_t *__restrict__ count,
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
    // node velocities (and volume fractions), one plane per value
    __shared__ float sv_all[(DIM + (VC ? 1 : 0)) * Hl::SIZE];
    const VelHalo<DIM, T> sv{sv_all, sv_all + Hl::SIZE, DIM == 3 ? sv_all + 2 * Hl::SIZE : sv_all,
                             VC ? sv_all + DIM * Hl::SIZE : sv_all};
    __shared__ float sbuf[BUF];
    // [(qi, warp)][class], rows padded to 33 words: the scan reads a column
    __shared__ uint32_t hist[NQ * NWARP * 33];
    __shared__ uint32_t cstart[32];
    // sorted entry e -> bin-order entry, at e + e / 32: the interleaved reads
    // take entries R apart
    __shared__ uint32_t order[kSliceParticles + kSliceParticles / 32];
    const uint32_t lane = lane_id();
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    [[maybe_unused]] const float dtg[3] = {dtg0, dtg1, dtg2};
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
        load_halo<DIM, T, VC, UPD, 1>(g, src, dtg, o, sv_all, (int)threadIdx.x, (int)blockDim.x);
        if constexpr (UPD != 0) {
            using AccT = typename AccOf<UPD>::T;
            __syncthreads();  // every thread's halo loads are done
            if (threadIdx.x < 32)
                release_blocks<DIM, T, AccT, DIM + 1 + (VC ? 1 : 0)>(g, t, readers, count,
                                                                     const_cast<AccT *>(static_cast<const AccT *>(src)),
                                                                     lane);
        }
        if (cnt <= 32u) {
            // one round: the order inside it does not matter, bin order is kept
            cp_async_wait<0>();
            __syncthreads();
            if (threadIdx.x < cnt) {
                const uint32_t r = threadIdx.x;
                auto rec = [&](int f) { return sbuf[f * kSliceParticles + r]; };
                float xo[DIM];
                gather_one<DIM, T, true, EL, VC>(g, p, q, pids[0], beg + r, rec, o, sv, dt, c4, smax, rmax, xo);
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
                    float xo[DIM];
                    gather_one<DIM, T, true, EL, VC>(g, p, q, perm[beg + r], beg + pos, rec, o, sv, dt, c4, smax,
                                                     rmax, xo);
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
// warps.  NK (in place): each lane also writes the key of its particle's new
// position to next_key and adds it to the tile histogram count_next (the
// binning of the next step takes both, MPM_BIN_KEYS_FROM_G2P).
template <int DIM, int T, bool BINORDER, bool EL, bool VC, int UPD, bool NK = false>
__global__ void __launch_bounds__(kP2GThreads) k_g2p_w(GridP g, PartsF p, PartsF q, const void *__restrict__ src,
                                                       float dtg0, float dtg1, float dtg2,
                                                       uint32_t *__restrict__ readers,
                                                       const uint32_t *__restrict__ count,
                                                       const uint32_t *__restrict__ perm,
                                                       const uint32_t *__restrict__ slices,
                                                       const uint32_t *__restrict__ start,
                                                       uint32_t *__restrict__ status, float dt, float c4,
                                                       uint32_t *__restrict__ next_key = nullptr,
                                                       uint32_t *__restrict__ count_next = nullptr) {
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
        load_halo<DIM, T, VC, UPD>(g, src, dtg, o, vw, (int)lane, 32);
        __syncwarp();
        if constexpr (UPD != 0) {
            using AccT = typename AccOf<UPD>::T;
            release_blocks<DIM, T, AccT, DIM + 1 + (VC ? 1 : 0)>(g, t, readers, count,
                                                                 const_cast<AccT *>(static_cast<const AccT *>(src)),
                                                                 lane);
        }
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
                float xo[DIM];
                if (r < cnt) {
                    auto rec = [&](int f) { return xc[f]; };
                    gather_one<DIM, T, false, EL, VC>(g, p, q, pid, pid, rec, o, sv, dt, c4, smax, rmax, xo);
                }
                if constexpr (NK) {
                    // the key of the position just written, and its tile's count (one add per tile a round)
                    constexpr int LOG = T == 4 ? 2 : 3;
                    const bool live = r < cnt;
                    uint32_t bk = 0xFFFFFFFFu;
                    if (live) {
                        const uint32_t k = key_of_x<DIM, T>(g, xo);
                        next_key[pid] = k;
                        bk = k == kKeyInvalid ? (uint32_t)g.ntiles : k >> (DIM * LOG);
                    }
                    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bk);
                    if (live && (peers & lanemask_lt()) == 0) atomicAdd(&count_next[bk], (uint32_t)__popc(peers));
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
                    float xo[DIM];
                    gather_one<DIM, T, BINORDER, EL, VC>(g, p, q, pid, BINORDER ? beg + r : pid, rec, o, sv, dt, c4,
                                                         smax, rmax, xo);
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
