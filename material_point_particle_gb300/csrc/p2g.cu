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
// Work item: a slice of at most 1024 consecutive binned particles of one
// tile (T^dim base cells), taken from a global work counter.  A CTA zeroes
// the tile's (T+2)^dim x (dim+1) int32 accumulators in shared memory, each
// thread computes its particles' shares and adds each one with a shared
// atomic as soon as it is formed, and the CTA flushes every nonzero node with
// one global atomic add (neighbouring slices and tiles overlap on halo nodes,
// so the flush must add).  The int32 halo is flushed after every 512
// particles, so no halo sum can overflow.
#include "common.cuh"
#include "internal.h"
#include "range.cuh"
#include "scatter.cuh"
#include "stress.cuh"

namespace mpm {

template <int DIM, int T, bool EL, bool VC, typename Rec>
__device__ __forceinline__ void scatter_float(const GridP &g, const Rec &rec, const int o[3], float *sacc,
                                              const StressP &sp, uint32_t &degenerate) {
    using Hl = Halo<DIM, T>;
    using Fl = P2GFields<DIM, EL, VC>;
    float f[3] = {0.f, 0.f, 0.f};
    int b[3] = {0, 0, 0};
    float xs[DIM];
#pragma unroll
    for (int l = 0; l < DIM; ++l) xs[l] = rec(l);
    if (!in_tile_x<DIM>(g, xs, o, b, f)) return;
    float v[DIM], C[DIM * DIM], w[3][3], dd[3][3];
#pragma unroll
    for (int k = 0; k < DIM; ++k) v[k] = rec(DIM + k);
    load_affine<DIM, EL, VC>(rec, sp, C, degenerate);
    const float m = rec(2 * DIM + DIM * DIM);
    [[maybe_unused]] float q = 0.f;
    if constexpr (VC) q = __fmul_rn(rec(Fl::VOLF), g.vcell);
#pragma unroll
    for (int l = 0; l < DIM; ++l) {
        quad_weights(f[l], w[l]);
#pragma unroll
        for (int a = 0; a < 3; ++a) dd[l][a] = __fmul_rn(__fsub_rn((float)a, f[l]), g.dx);
    }
    const int hb = DIM == 3 ? (b[0] - o[0]) + (b[1] - o[1]) * Hl::SY + (b[2] - o[2]) * Hl::SZ
                            : (b[0] - o[0]) + (b[1] - o[1]) * Hl::SY;
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
                const int at = hb + Hl::off(a);
                atomicAdd(&sacc[at], W);
                if constexpr (VC) {
                    const float Wvxy = __fmul_rn(__fmul_rn(w[0][a0], q), w[1][a1]);
                    atomicAdd(&sacc[(DIM + 1) * Hl::SIZE + at], DIM == 3 ? __fmul_rn(Wvxy, w[2][a2]) : Wvxy);
                }
#pragma unroll
                for (int k = 0; k < DIM; ++k) {
                    const float vel = DIM == 3 ? __fmaf_rn(C[k * DIM + 2], dd[2][a2], h1[k]) : h1[k];
                    atomicAdd(&sacc[(1 + k) * Hl::SIZE + at], __fmul_rn(W, vel));
                }
            }
        }
    }
}

// One warp per work item (a slice of at most 1024 binned particles of one
// tile), so no CTA barrier couples the warps: each warp owns a compact halo
// of the tile's (T+2)^dim nodes x (dim+1) int32 accumulators.  Per item: 32
// particles a round; each lane loads its next particle's position into
// registers while the current one scatters, and the rest of the record
// (v, C, m, ...) at the start of its round, so the shared-memory pipe, which
// the scatter's atomics keep busy, carries nothing else.  With the elastic
// state (two blocks per SM) the whole record is copied into a per-warp double
// buffer in shared memory (cp.async) a round ahead instead.  Every 512
// particles and at the end the warp adds each
// nonzero halo entry to the grid with one global atomic and clears it
// (neighbouring tiles overlap on the halo, so the flush adds).  Particles
// stored in bank-class interleaved order (the sorted G2P) put the 32 lanes of
// a round in different banks.
//
// Two instances, one per share path; the bound check before the scatter
// (k_bound) picks one and the other returns at once.  WIDE = false: shares
// below 2^22 (one fma each).  WIDE = true: 64-bit shares (exact integer
// product), each split into two int32 halves in two halo planes per channel
// (twice the shared memory, so four warps per block); a particle whose
// shares could reach 2^43 adds them straight to the global grid instead.
// `verify` (the bound was taken from the records of the previous P2G and
// G2P): a particle above that range is not scattered, and the call's scatter
// is undone afterwards (k_rollback).
template <bool WIDE, bool EL>
struct P2GShape {
    static constexpr int WARPS = WIDE ? 4 : 8;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int MIN_BLOCKS = WIDE ? (EL ? 2 : 3) : (EL ? 2 : 3);
};

template <int DIM, int T, typename AccT, bool EL, bool VC, bool WIDE>
__global__ void __launch_bounds__(P2GShape<WIDE, EL>::THREADS, P2GShape<WIDE, EL>::MIN_BLOCKS)
    k_p2g_fixed(GridP g, PartsF p, const uint32_t *__restrict__ perm, const uint32_t *__restrict__ slices,
                const uint32_t *__restrict__ start, uint32_t *__restrict__ status, AccT *__restrict__ acc,
                StressP sp, int verify) {
    using Hl = HaloU<DIM, T>;
    using Fl = P2GFields<DIM, EL, VC>;
    using Sh = P2GShape<WIDE, EL>;
    constexpr int NCH = Stencil<DIM>::NC + (VC ? 1 : 0);  // accumulator channels
    constexpr int HW = (WIDE ? 2 : 1) * NCH * Hl::NODES;  // halo words per warp
    __shared__ __align__(16) int32_t shalo[Sh::WARPS][HW];
    // with the elastic state the whole record is staged in shared memory (at two blocks per SM
    // register loads' latency would not hide behind other warps); otherwise nothing is
    constexpr int NS = EL ? Fl::NF : 1;
    __shared__ float sbuf[Sh::WARPS][EL ? 2 * NS * 32 : 1];
    if (status[MPM_ST_FLAGS] & kFlagNoScatter) return;
    if (status[MPM_ST_SHARE_PATH] != (WIDE ? 1u : 0u)) return;
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    int32_t *wh = shalo[warp];
    float *wb = sbuf[warp];
    const uint32_t halo = (uint32_t)__cvta_generic_to_shared(wh);
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    const uint32_t Rrec = status[MPM_ST_RANGE];
    const float h = __fmul_rn(1.5f, g.dx);
    uint32_t *work = &status[MPM_ST_WORK_P2G];
    for (int i = lane; i < HW; i += 32) wh[i] = 0;
    __syncwarp();
    auto at = [&](int stage, int f) { return wb + (stage * NS + f) * 32 + lane; };
    auto issue = [&](int stage, uint32_t pid) {
#pragma unroll
        for (int f = 0; f < NS; ++f) cp_async4(at(stage, f), Fl::src(p, f) + pid);
    };
    uint32_t s = 0, degenerate = 0, mrec = 0, qrec = 0;
    if (lane == 0) s = atomicAdd(work, 1u);
    s = __shfl_sync(0xFFFFFFFFu, s, 0);
    while (s < nslices) {
        const uint32_t ask = lane == 0 ? atomicAdd(work, 1u) : 0u;  // the next item, used at the end
        const uint32_t t = slices[2 * (size_t)s];
        const uint32_t beg = start[t] + slices[2 * (size_t)s + 1];
        const uint32_t cnt = min((uint32_t)kSliceParticles, start[t + 1] - beg);
        int o[3];
        tile_origin(g, t, o);
        // every nonzero halo entry added to the grid once, and cleared
        auto flush = [&]() {
            __syncwarp();
            for (int hh = lane; hh < Hl::NODES; hh += 32) {
                int hx, hy, hz;
                Hl::node(hh, hx, hy, hz);
                const int gx = o[0] + hx, gy = o[1] + hy, gz = o[2] + hz;
                const bool on = gx < g.n[0] && gy < g.n[1] && (DIM == 2 || gz < g.n[2]);
                const int64_t node = node_index(g, gx, gy, gz);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    long long val = wh[c * Hl::NODES + hh];
                    if constexpr (WIDE) val += (long long)wh[(NCH + c) * Hl::NODES + hh] * (1ll << 22);
                    if (val == 0) continue;
                    wh[c * Hl::NODES + hh] = 0;
                    if constexpr (WIDE) wh[(NCH + c) * Hl::NODES + hh] = 0;
                    if (!on) continue;
                    if constexpr (sizeof(AccT) == 8)
                        atomicAdd(reinterpret_cast<unsigned long long *>(acc + c * g.nodes + node),
                                  (unsigned long long)val);
                    else
                        atomicAdd(reinterpret_cast<int *>(acc + c * g.nodes + node), (int)val);
                }
            }
            __syncwarp();
        };
        // one particle: false when it is not scattered (not in this tile's box, or above the
        // recorded range)
        auto one = [&](const auto &rec) -> bool {
            float xs[DIM], f[3] = {0.f, 0.f, 0.f};
            int b[3] = {0, 0, 0};
#pragma unroll
            for (int l = 0; l < DIM; ++l) xs[l] = rec(l);
            if (!in_box_x<DIM, T>(g, xs, o, b, f)) return false;
            const float m = rec(2 * DIM + DIM * DIM);
            [[maybe_unused]] float q = 0.f;
            if constexpr (VC) q = __fmul_rn(rec(Fl::VOLF), g.vcell);
            mrec = max_bits(mrec, fabsf(m));
            if constexpr (VC) qrec = max_bits(qrec, fabsf(q));
            const int hb = DIM == 3 ? (b[0] - o[0]) + (b[1] - o[1]) * Hl::SY + (b[2] - o[2]) * Hl::SZ
                                    : (b[0] - o[0]) + (b[1] - o[1]) * Hl::SY;
            float v[DIM], C[DIM * DIM];
#pragma unroll
            for (int k = 0; k < DIM; ++k) v[k] = rec(DIM + k);
            if constexpr (!WIDE) {
                if (verify) {
#pragma unroll
                    for (int j = 0; j < DIM * DIM; ++j) C[j] = rec(2 * DIM + j);
                    if (particle_range_bits<VC>(range_r_bits<DIM>(v, C, h), m, q) > Rrec) return false;
                }
                const SharedAdd<Hl> ad{halo + 4u * (uint32_t)hb};
                scatter_shares<DIM, EL, VC, false>(g, rec, f, ad, sp, degenerate);
            } else {
                load_affine<DIM, EL, VC>(rec, sp, C, degenerate);
                const uint32_t Rp = particle_range_bits<VC>(range_r_bits<DIM>(v, C, h), m, q);
                if (verify && Rp > Rrec) return false;
                if (__fmul_rn(__uint_as_float(Rp), g.S) <= 0x1p42f) {
                    const SharedAdd64<Hl, NCH> ad{halo + 4u * (uint32_t)hb};
                    scatter_shares_wide<DIM, EL, VC>(g, rec, f, ad, v, C);
                } else {  // shares that could reach 2^43: straight to the grid
                    const GlobalAdd64<DIM, AccT> ad{acc, g.nodes, g.n[0], (int64_t)g.n[0] * g.n[1],
                                                    node_index(g, b[0], b[1], DIM == 3 ? b[2] : 0)};
                    scatter_shares_wide<DIM, EL, VC>(g, rec, f, ad, v, C);
                }
            }
            return true;
        };
        uint32_t bad = 0;
        const uint32_t rounds = (cnt + 31) / 32;
        // the int32 halo accumulators are flushed every 16 rounds: at most 512
        // shares reach one entry between two flushes
        // perm is read one round ahead of its use, so no round waits on it
        uint32_t pid = lane < cnt ? perm[beg + lane] : 0u;
        uint32_t pid_next = lane + 32 < cnt ? perm[beg + lane + 32] : 0u;
        if constexpr (!EL) {
            // the positions in registers a round ahead, the rest of the record at the start of its round
            float xc[DIM], xn[DIM];
#pragma unroll
            for (int l = 0; l < DIM; ++l) xc[l] = lane < cnt ? p.x[l][pid] : 0.f;
            for (uint32_t qq = 0; qq < rounds; ++qq) {
                const uint32_t r = qq * 32 + lane;
#pragma unroll
                for (int l = 0; l < DIM; ++l) xn[l] = r + 32 < cnt ? p.x[l][pid_next] : 0.f;
                const uint32_t pid_after = r + 64 < cnt ? perm[beg + r + 64] : 0u;
                if (r < cnt) {
                    float rest[Fl::NF - DIM];
#pragma unroll
                    for (int f = DIM; f < Fl::NF; ++f) rest[f - DIM] = Fl::src(p, f)[pid];
                    auto rec = [&](int f) { return f < DIM ? xc[f] : rest[f - DIM]; };
                    if (!one(rec)) ++bad;
                }
#pragma unroll
                for (int l = 0; l < DIM; ++l) xc[l] = xn[l];
                pid = pid_next;
                pid_next = pid_after;
                if ((qq + 1) % 16 == 0 && qq + 1 < rounds) flush();
            }
        } else {
            // the whole record copied into shared memory (cp.async) a round ahead
            if (lane < cnt) issue(0, pid);
            cp_async_commit();
            int stage = 0;
            for (uint32_t qq = 0; qq < rounds; ++qq) {
                const uint32_t r = qq * 32 + lane;
                if (qq + 1 < rounds && r + 32 < cnt) issue(stage ^ 1, pid_next);
                const uint32_t pid_after = r + 64 < cnt ? perm[beg + r + 64] : 0u;
                cp_async_commit();
                cp_async_wait<1>();
                if (r < cnt) {
                    const int st = stage;
                    auto rec = [&](int f) { return *at(st, f); };
                    if (!one(rec)) ++bad;
                }
                stage ^= 1;
                pid_next = pid_after;
                if ((qq + 1) % 16 == 0 && qq + 1 < rounds) flush();
            }
        }
        flush();
        bad = __reduce_add_sync(0xFFFFFFFFu, bad);
        if (bad && lane == 0) {
            atomicAdd(&status[MPM_ST_N_OUT_OF_RANGE], bad);
            atomicOr(&status[MPM_ST_FLAGS], (1u << MPM_E_BOUND) | kFlagRollback);
        }
        s = __shfl_sync(0xFFFFFFFFu, ask, 0);
    }
    cp_async_wait<0>();
    warp_max_to(mrec, &status[MPM_ST_P2G_MASS]);
    if constexpr (VC) warp_max_to(qrec, &status[MPM_ST_P2G_VOLUME]);
    if constexpr (EL) {
        degenerate = __reduce_add_sync(0xFFFFFFFFu, degenerate);
        if (degenerate && lane == 0) atomicAdd(&status[MPM_ST_N_DEGENERATE], degenerate);
    }
}

// --------------------------------------------------------------------------
// The bound before the scatter ("particle to grid transfer in checked integer
// arithmetic", the program: the bounds line runs first, and if it fails
// nothing is scattered).

// R = max of R_p over the binned (in-domain) particles, read from the state
// P2G is about to scatter (elastic particles: the stress-folded matrix).
template <int DIM, bool EL, bool VC>
__global__ void __launch_bounds__(256) k_range(GridP g, PartsF p, const uint32_t *__restrict__ key,
                                               uint32_t *__restrict__ status, StressP sp) {
    using Fl = P2GFields<DIM, EL, VC>;
    const float h = __fmul_rn(1.5f, g.dx);
    uint32_t Rb = 0, unused = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += (int64_t)gridDim.x * blockDim.x) {
        if (key[i] == kKeyInvalid) continue;
        auto rec = [&](int f) { return Fl::src(p, f)[i]; };
        float v[DIM], C[DIM * DIM];
#pragma unroll
        for (int k = 0; k < DIM; ++k) v[k] = rec(DIM + k);
        load_affine<DIM, EL, VC>(rec, sp, C, unused);
        [[maybe_unused]] float q = 0.f;
        if constexpr (VC) q = __fmul_rn(rec(Fl::VOLF), g.vcell);
        Rb = max(Rb, particle_range_bits<VC>(range_r_bits<DIM>(v, C, h), rec(2 * DIM + DIM * DIM), q));
    }
    warp_max_to(Rb, &status[MPM_ST_RANGE]);
}

// One thread, before the scatter: resets the P2G call's counters, takes R
// from the pass above or from the records (then clears the records for this
// call's own), and applies the test the oracle states (fp64, this order):
// B = S*R*(1 + 2^-10) + 28, count * B within 2^62 (int64) or 2^31 - 1024
// (int32, count = most stencils covering a node).  Failing, P2G scatters
// nothing; passing, the share path is chosen.
__global__ void k_bound(GridP g, uint32_t *__restrict__ status, int from_records) {
    if (threadIdx.x != 0) return;
    status[MPM_ST_N_DEGENERATE] = 0;
    status[MPM_ST_WORK_P2G] = 0;
    status[MPM_ST_N_OUT_OF_RANGE] = 0;
    uint32_t flags = status[MPM_ST_FLAGS] & ~((1u << MPM_E_BOUND) | kFlagNoScatter | kFlagRollback);
    uint32_t Rb;
    if (from_records) {
        const float M = __uint_as_float(status[MPM_ST_P2G_MASS]);
        const float rG = __uint_as_float(status[MPM_ST_G2P_RANGE]);
        Rb = __float_as_uint(__fmul_rn(M, rG));
        if (isnan(M) || isnan(rG)) Rb = 0x7FFFFFFFu;
        if (g.vc) Rb = max(Rb, status[MPM_ST_P2G_VOLUME]);
        status[MPM_ST_RANGE] = Rb;
    } else {
        Rb = status[MPM_ST_RANGE];
    }
    status[MPM_ST_P2G_MASS] = 0;
    status[MPM_ST_P2G_VOLUME] = 0;
    status[MPM_ST_SHARE_PATH] = 0;
    const double R = (double)__uint_as_float(Rb);
    const double S = (double)g.S;
    const double B = __dadd_rn(__dmul_rn(__dmul_rn(S, R), 1.0 + 0x1p-10), 28.0);
    const uint32_t count = g.acc_mode == MPM_ACC_I32 ? status[MPM_ST_MAX_NEIGHBOURS] : status[MPM_ST_N_VALID];
    const double limit = g.acc_mode == MPM_ACC_I32 ? 2147482624.0 : 0x1p62;
    if (!(__dmul_rn((double)count, B) <= limit)) {
        flags |= (1u << MPM_E_BOUND) | kFlagNoScatter;
    } else {
        const double fast = __dmul_rn(__dmul_rn(__dmul_rn((double)g.wmax, S), R), 1.0 + 0x1p-10);
        status[MPM_ST_SHARE_PATH] = fast <= (double)kShareLimit ? 0u : 1u;
    }
    status[MPM_ST_FLAGS] = flags;
}

// Undoes a scatter whose particles broke the range it was checked with: the
// grid was zero on entry, so it is cleared again.  Returns at once otherwise.
template <typename AccT>
__global__ void __launch_bounds__(256) k_rollback(AccT *__restrict__ acc, int64_t words,
                                                  const uint32_t *__restrict__ status) {
    if (!(status[MPM_ST_FLAGS] & kFlagRollback)) return;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += (int64_t)gridDim.x * blockDim.x)
        acc[i] = 0;
}

void launch_rollback(const GridP &g, void *grid_acc, const uint32_t *status, const DeviceInfo &dev,
                     cudaStream_t st) {
    const int64_t words = (int64_t)(g.dim + 1 + g.vc) * g.nodes;
    if (g.acc_mode == MPM_ACC_I32)
        k_rollback<int32_t><<<dev.sms, 256, 0, st>>>((int32_t *)grid_acc, words, status);
    else
        k_rollback<long long><<<dev.sms, 256, 0, st>>>((long long *)grid_acc, words, status);
}

// Float-atomic P2G (comparison variant: fp32 adds, order dependent).
template <int DIM, int T, bool EL, bool VC>
__global__ void __launch_bounds__(kP2GThreads) k_p2g_float(GridP g, PartsF p, const uint32_t *__restrict__ perm,
                                                           const uint32_t *__restrict__ slices,
                                                           const uint32_t *__restrict__ start,
                                                           uint32_t *__restrict__ status,
                                                           float *__restrict__ acc, StressP sp) {
    using St = Stencil<DIM>;
    using Hl = Halo<DIM, T>;
    using Fl = P2GFields<DIM, EL, VC>;
    constexpr int NCH = St::NC + (VC ? 1 : 0);
    uint32_t degenerate = 0;
    __shared__ float sacc[NCH * Hl::SIZE];
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    __shared__ uint32_t item_sh;
    uint32_t next = 0;
    for (uint32_t s = grab_item(&status[MPM_ST_WORK_P2G], &item_sh); s < nslices; s = publish_item(next, &item_sh)) {
        next = ask_item(&status[MPM_ST_WORK_P2G]);
        const uint32_t t = slices[2 * (size_t)s], first = slices[2 * (size_t)s + 1];
        const uint32_t beg = start[t] + first;
        const uint32_t cnt = min((uint32_t)kSliceParticles, start[t + 1] - beg);
        int o[3];
        tile_origin(g, t, o);
        for (int h = threadIdx.x; h < Hl::NODES; h += blockDim.x) {
            int hx, hy, hz, idx;
            Hl::node(h, hx, hy, hz, idx);
#pragma unroll
            for (int c = 0; c < NCH; ++c) sacc[c * Hl::SIZE + idx] = 0.f;
        }
        __syncthreads();
        for (uint32_t r = threadIdx.x; r < cnt; r += blockDim.x) {
            const uint32_t pid = perm[beg + r];
            auto rec = [&](int f) { return Fl::src(p, f)[pid]; };
            scatter_float<DIM, T, EL, VC>(g, rec, o, sacc, sp, degenerate);
        }
        __syncthreads();
        for (int h = threadIdx.x; h < Hl::NODES; h += blockDim.x) {
            int hx, hy, hz, idx;
            Hl::node(h, hx, hy, hz, idx);
            const int gx = o[0] + hx, gy = o[1] + hy, gz = o[2] + hz;
            if (gx >= g.n[0] || gy >= g.n[1] || (DIM == 3 && gz >= g.n[2])) continue;
            const int64_t node = node_index(g, gx, gy, gz);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const float val = sacc[c * Hl::SIZE + idx];
                if (val != 0.f) atomicAdd(acc + c * g.nodes + node, val);
            }
        }
        __syncthreads();
    }
    if constexpr (EL) {
        degenerate = __reduce_add_sync(0xFFFFFFFFu, degenerate);
        if (degenerate && lane_id() == 0) atomicAdd(&status[MPM_ST_N_DEGENERATE], degenerate);
    }
}

template <int DIM, int T, typename AccT, bool EL, bool VC>
void launch_p2g_fixed(const GridP &g, const PartsF &p, const WsView &w, AccT *acc, const StressP &sp, int verify,
                      const DeviceInfo &dev, cudaStream_t st) {
    // both share paths; the one k_bound did not pick returns at once
    k_p2g_fixed<DIM, T, AccT, EL, VC, false><<<dev.sms * 4, P2GShape<false, EL>::THREADS, 0, st>>>(
        g, p, w.perm, w.slices, w.start, w.status, acc, sp, verify);
    k_p2g_fixed<DIM, T, AccT, EL, VC, true><<<dev.sms * 8, P2GShape<true, EL>::THREADS, 0, st>>>(
        g, p, w.perm, w.slices, w.start, w.status, acc, sp, verify);
}

template <int DIM, int T, bool EL, bool VC>
void launch_p2g_t(const GridP &g, const PartsF &p, const WsView &w, void *grid_acc, const StressP &sp,
                  bool records, const DeviceInfo &dev, cudaStream_t st) {
    if (g.acc_mode == MPM_ACC_F32) {
        k_p2g_float<DIM, T, EL, VC><<<dev.sms * 4, kP2GThreads, 0, st>>>(g, p, w.perm, w.slices, w.start,
                                                                         w.status, (float *)grid_acc, sp);
        return;
    }
    // the bound, before any particle is scattered: R from a pass over the state, or from the records
    if (!records) {
        cudaMemsetAsync(&w.status[MPM_ST_RANGE], 0, sizeof(uint32_t), st);
        if (p.n > 0) {
            const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((p.n + 255) / 256, dev.sms * 8));
            k_range<DIM, EL, VC><<<blocks, 256, 0, st>>>(g, p, w.key, w.status, sp);
        }
    }
    k_bound<<<1, 32, 0, st>>>(g, w.status, records ? 1 : 0);
    if (g.acc_mode == MPM_ACC_I64)
        launch_p2g_fixed<DIM, T, long long, EL, VC>(g, p, w, (long long *)grid_acc, sp, records, dev, st);
    else
        launch_p2g_fixed<DIM, T, int32_t, EL, VC>(g, p, w, (int32_t *)grid_acc, sp, records, dev, st);
    if (records) launch_rollback(g, grid_acc, w.status, dev, st);
}

template <int DIM, int T>
void launch_p2g_dt(const GridP &g, const PartsF &p, const WsView &w, void *grid_acc, const StressP &sp,
                   bool records, const DeviceInfo &dev, cudaStream_t st) {
    const bool el = p.F[0] != nullptr;
    if (el && g.vc)
        launch_p2g_t<DIM, T, true, true>(g, p, w, grid_acc, sp, false, dev, st);
    else if (el)
        launch_p2g_t<DIM, T, true, false>(g, p, w, grid_acc, sp, false, dev, st);
    else if (g.vc)
        launch_p2g_t<DIM, T, false, true>(g, p, w, grid_acc, sp, records, dev, st);
    else
        launch_p2g_t<DIM, T, false, false>(g, p, w, grid_acc, sp, records, dev, st);
}

mpm_status launch_p2g(const GridP &g, const PartsF &p, const WsView &w, void *grid_acc, float dt, bool records,
                      const DeviceInfo &dev, cudaStream_t st) {
    const StressP sp{p.mu, p.lam, dt, (4.0f * g.inv_dx) * g.inv_dx};
    if (g.acc_mode == MPM_ACC_F32) {  // the fixed-point modes reset these in k_bound
        static_assert(MPM_ST_WORK_P2G == MPM_ST_N_DEGENERATE + 1, "adjacent status words");
        cudaMemsetAsync(&w.status[MPM_ST_N_DEGENERATE], 0, 2 * sizeof(uint32_t), st);
    }
    if (g.dim == 3 && g.T == 4)
        launch_p2g_dt<3, 4>(g, p, w, grid_acc, sp, records, dev, st);
    else if (g.dim == 2 && g.T == 8)
        launch_p2g_dt<2, 8>(g, p, w, grid_acc, sp, records, dev, st);
    else
        return MPM_E_ARG;
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
