// gather.cuh -- the G2P stencil sums from a tile's velocity halo in shared
// memory (used by the G2P kernels and by the fused gather-scatter step).
//
// The new velocity v' = sum_a w(a) v(a) and the APIC matrix B_kl =
// sum_a w(a) v_k(a) e_l(a) (implementation guide, section 3.1, Part 1, and
// 3.3.2, "gather d and D (= B*4)"), taken axis by axis, innermost axis first,
// each three-term sum as fma(w2,t2, fma(w1,t1, w0*t0)): the order the oracle
// states.  The x and y components go through packed fp32x2 arithmetic, which
// rounds each lane exactly as the scalar operation.
#pragma once

#include "common.cuh"

namespace mpm {

__device__ __forceinline__ float sum3(const float w[3], const float t[3]) {
    return __fmaf_rn(w[2], t[2], __fmaf_rn(w[1], t[1], __fmul_rn(w[0], t[0])));
}

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// sum3 on two independent lanes (each lane exactly the scalar sum3)
__device__ __forceinline__ float2 sum3x2(const float2 w[3], const float2 t[3]) {
    return __ffma2_rn(w[2], t[2], __ffma2_rn(w[1], t[1], __fmul2_rn(w[0], t[0])));
}

// Velocity halo of one tile in shared memory, in the compact layout HaloU of
// the P2G accumulators, one array per component.
template <int DIM, int T>
struct VelHalo {
    float *x, *y, *z;
    float *phi;  // node volume fractions (volume channel)
};

// v' and B of the particle whose stencil starts at halo offset hb, from its
// weights w and w * e (e = node offset in cells).
template <int DIM, int T>
__device__ __forceinline__ void gather_vB(const VelHalo<DIM, T> &sv, int hb, const float (&w)[3][3],
                                          const float (&we)[3][3], float (&vn)[DIM], float (&Bm)[DIM][DIM]) {
    using Hl = HaloU<DIM, T>;
    float2 W[3][3], WE[3][3];
#pragma unroll
    for (int l = 0; l < DIM; ++l)
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            W[l][a] = f2(w[l][a]);
            WE[l][a] = f2(we[l][a]);
        }
    const float *vx = sv.x + hb, *vy = sv.y + hb;
    if constexpr (DIM == 3) {
        // x and y packed
        float2 Y[3], Ye[3], Yq[3];
#pragma unroll
        for (int a0 = 0; a0 < 3; ++a0) {
            float2 Z[3], Zq[3];
#pragma unroll
            for (int a1 = 0; a1 < 3; ++a1) {
                float2 t[3];
#pragma unroll
                for (int a2 = 0; a2 < 3; ++a2) {
                    const int i = a0 + a1 * Hl::SY + a2 * Hl::SZ;
                    t[a2] = make_float2(vx[i], vy[i]);
                }
                Z[a1] = sum3x2(W[2], t);
                Zq[a1] = sum3x2(WE[2], t);
            }
            Y[a0] = sum3x2(W[1], Z);
            Ye[a0] = sum3x2(WE[1], Z);
            Yq[a0] = sum3x2(W[1], Zq);
        }
        const float2 v2 = sum3x2(W[0], Y), b0 = sum3x2(WE[0], Y), b1 = sum3x2(W[0], Ye), b2 = sum3x2(W[0], Yq);
        vn[0] = v2.x;
        vn[1] = v2.y;
        Bm[0][0] = b0.x;
        Bm[1][0] = b0.y;
        Bm[0][1] = b1.x;
        Bm[1][1] = b1.y;
        Bm[0][2] = b2.x;
        Bm[1][2] = b2.y;
        // z alone
        const float *vz = sv.z + hb;
        float Ys[3], Yes[3], Yqs[3];
#pragma unroll
        for (int a0 = 0; a0 < 3; ++a0) {
            float Z[3], Zq[3];
#pragma unroll
            for (int a1 = 0; a1 < 3; ++a1) {
                float t[3];
#pragma unroll
                for (int a2 = 0; a2 < 3; ++a2) t[a2] = vz[a0 + a1 * Hl::SY + a2 * Hl::SZ];
                Z[a1] = sum3(w[2], t);
                Zq[a1] = sum3(we[2], t);
            }
            Ys[a0] = sum3(w[1], Z);
            Yes[a0] = sum3(we[1], Z);
            Yqs[a0] = sum3(w[1], Zq);
        }
        vn[2] = sum3(w[0], Ys);
        Bm[2][0] = sum3(we[0], Ys);
        Bm[2][1] = sum3(w[0], Yes);
        Bm[2][2] = sum3(w[0], Yqs);
    } else {
        float2 Y[3], Ye[3];
#pragma unroll
        for (int a0 = 0; a0 < 3; ++a0) {
            float2 t[3];
#pragma unroll
            for (int a1 = 0; a1 < 3; ++a1) t[a1] = make_float2(vx[a0 + a1 * Hl::SY], vy[a0 + a1 * Hl::SY]);
            Y[a0] = sum3x2(W[1], t);
            Ye[a0] = sum3x2(WE[1], t);
        }
        const float2 v2 = sum3x2(W[0], Y), b0 = sum3x2(WE[0], Y), b1 = sum3x2(W[0], Ye);
        vn[0] = v2.x;
        vn[1] = v2.y;
        Bm[0][0] = b0.x;
        Bm[1][0] = b0.y;
        Bm[0][1] = b1.x;
        Bm[1][1] = b1.y;
    }
}

// sum_a w(a) phi(a) in the order of v (the volume channel's gather).
template <int DIM, int T>
__device__ __forceinline__ float gather_phi(const VelHalo<DIM, T> &sv, int hb, const float (&w)[3][3]) {
    using Hl = HaloU<DIM, T>;
    const float *vp = sv.phi + hb;
    float Yp[3];
#pragma unroll
    for (int a0 = 0; a0 < 3; ++a0) {
        if constexpr (DIM == 3) {
            float Zp[3];
#pragma unroll
            for (int a1 = 0; a1 < 3; ++a1) {
                float t[3];
#pragma unroll
                for (int a2 = 0; a2 < 3; ++a2) t[a2] = vp[a0 + a1 * Hl::SY + a2 * Hl::SZ];
                Zp[a1] = sum3(w[2], t);
            }
            Yp[a0] = sum3(w[1], Zp);
        } else {
            float t[3];
#pragma unroll
            for (int a1 = 0; a1 < 3; ++a1) t[a1] = vp[a0 + a1 * Hl::SY];
            Yp[a0] = sum3(w[1], t);
        }
    }
    return sum3(w[0], Yp);
}

// Interleaved slices.  The sorted output keeps each slice in its place but
// orders it by the bank class of the particles' base cells (cell_class: the
// cell's offset in the compact halo modulo 32, x + 6y + 36z in a 4^3 tile,
// x + 10y in an 8^2 tile), stable in bin order, then deals the class-sorted entries out
// column by column over rounds of 32: with R = ceil(cnt / 32) rounds and
// L = cnt - 32 (R - 1) lanes in the last one, lane l holds sorted entries
// [cum(l), cum(l + 1)), cum(l) = l R - max(0, l - L), and entry
// cum(l) + rho sits at rho * 32 + l.  So the 32 entries of a round come from
// classes spread over the whole range.  Cells of different classes put a
// given stencil node in different shared-memory banks, and particles move a
// small fraction of a cell per step, so P2G and G2P, which take particles 32
// at a time in storage order, meet few bank conflicts.

// Sorted entry held by place pos of an interleaved slice of cnt entries.
__device__ __forceinline__ uint32_t interleave_entry(uint32_t pos, uint32_t cnt) {
    const uint32_t R = (cnt + 31) / 32, L = cnt - 32 * (R - 1);
    const uint32_t l = pos & 31u, rho = pos >> 5;
    return l * R - (l > L ? l - L : 0u) + rho;
}

// Stable counting sort of a slice of cnt binned particles by bank class
// (cell_class of each particle's key): order[e + e / 32] = the bin-order
// index of the e-th entry of the class-sorted slice.  Counts per (round,
// warp, class), scanned class-major.  pids[qi] = perm entry of bin-order
// index threadIdx.x + qi * NT.  All NT threads of the block call it; it
// synchronises the block.  hist: NQ * NWARP * 33 words (rows padded to 33:
// the scan reads a column); cstart: 32 words.
template <int DIM, int T, int NT>
__device__ __forceinline__ void class_order(const uint32_t *__restrict__ key, const uint32_t (&pids)[kSliceParticles / NT],
                                            uint32_t cnt, uint32_t *hist, uint32_t *cstart, uint32_t *order) {
    constexpr int NQ = kSliceParticles / NT;
    constexpr int NWARP = NT / 32;
    static_assert(NQ * NWARP == 32, "one warp-scan lane per (round, warp)");
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    uint32_t cls[NQ], below[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        const uint32_t r = threadIdx.x + qi * NT;
        cls[qi] = r < cnt ? cell_class<DIM, T>(key[pids[qi]]) : 32u;
    }
    for (int i = threadIdx.x; i < NQ * NWARP * 33; i += blockDim.x) hist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, cls[qi]);
        below[qi] = (uint32_t)__popc(peers & lanemask_lt());
        if (cls[qi] < 32u && below[qi] == 0) hist[(qi * NWARP + warp) * 33 + cls[qi]] = (uint32_t)__popc(peers);
    }
    __syncthreads();
    for (uint32_t c = warp; c < 32; c += NWARP) {
        const uint32_t v = hist[lane * 33 + c];
        uint32_t inc = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if ((int)lane >= d) inc += t2;
        }
        hist[lane * 33 + c] = inc - v;
        if (lane == 31) cstart[c] = inc;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t v = cstart[lane];
        uint32_t inc = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if ((int)lane >= d) inc += t2;
        }
        cstart[lane] = inc - v;
    }
    __syncthreads();
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        const uint32_t r = threadIdx.x + qi * NT;
        if (cls[qi] < 32u) {
            const uint32_t e = cstart[cls[qi]] + hist[(qi * NWARP + warp) * 33 + cls[qi]] + below[qi];
            order[e + (e >> 5)] = r;
        }
    }
}

// --------------------------------------------------------------------------
// Where the G2P kernels take node velocities from.  UPD = 0: the velocity
// grid of mpm_grid_update.  UPD = 1, 2, 3: the accumulators of mpm_p2g
// (int64, int32, fp32) with the grid update applied to each node as the halo
// loads (implementation guide, section 2.1, the worked shape: the load is
// the grid pass), the arithmetic of mpm_grid_update: v = (float)P / (float)M
// + dt*g (zero where M == 0), then the boundary sign test; with the volume
// channel phi = (float)V * 2^-scale.
template <int UPD>
struct AccOf {
    using T = float;
};
template <>
struct AccOf<1> {
    using T = long long;
};
template <>
struct AccOf<2> {
    using T = int32_t;
};

// The node values of a tile's halo into shared memory: node h of the compact
// layout goes to v[c * SIZE + h] for each value c (dim velocities, then phi).
// Thread `me` of `stride` threads takes nodes me, me + stride, ...; each
// takes B nodes at a time with every load issued before any value is used,
// so that the loads of a batch are in flight together.
template <int DIM, int T, bool VC, int UPD, int B = 4>
__device__ __forceinline__ void load_halo(const GridP &g, const void *src, const float (&dtg)[3], const int (&o)[3],
                                          float *v, int me, int stride) {
    using Hl = HaloU<DIM, T>;
    constexpr int NV = DIM + (VC ? 1 : 0);
    constexpr int NL = UPD == 0 ? NV : DIM + 1 + (VC ? 1 : 0);  // values loaded per node
    using LT = typename AccOf<UPD>::T;
    const LT *base = static_cast<const LT *>(src);
    for (int h0 = me; h0 < Hl::NODES; h0 += B * stride) {
        LT a[B][NL];
        int gi[B][3];
        bool in[B];
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int h = h0 + i * stride;
            int hx, hy, hz;
            Hl::node(h < Hl::NODES ? h : 0, hx, hy, hz);
            gi[i][0] = o[0] + hx;
            gi[i][1] = o[1] + hy;
            gi[i][2] = o[2] + hz;
            in[i] = h < Hl::NODES && gi[i][0] < g.n[0] && gi[i][1] < g.n[1] && (DIM == 2 || gi[i][2] < g.n[2]);
            const int64_t node = in[i] ? node_index(g, gi[i][0], gi[i][1], DIM == 3 ? gi[i][2] : 0) : 0;
#pragma unroll
            for (int c = 0; c < NL; ++c) a[i][c] = in[i] ? base[c * g.nodes + node] : (LT)0;
        }
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int h = h0 + i * stride;
            if (h >= Hl::NODES) break;
            float out[NV];
            if constexpr (UPD == 0) {
#pragma unroll
                for (int c = 0; c < NV; ++c) out[c] = a[i][c];
            } else {
#pragma unroll
                for (int c = 0; c < NV; ++c) out[c] = 0.f;
                const float M = acc_to_float(a[i][0]);
                if (M != 0.f) {
#pragma unroll
                    for (int l = 0; l < DIM; ++l) {
                        float vl = __fadd_rn(__fdiv_rn(acc_to_float(a[i][1 + l]), M), dtg[l]);
                        if ((gi[i][l] < g.boundary && vl < 0.f) || (gi[i][l] > g.n[l] - 1 - g.boundary && vl > 0.f))
                            vl = 0.f;
                        out[l] = vl;
                    }
                }
                if constexpr (VC) out[DIM] = in[i] ? __fmul_rn(acc_to_float(a[i][DIM + 1]), g.inv_S) : 0.f;
            }
#pragma unroll
            for (int c = 0; c < NV; ++c) v[c * Hl::SIZE + h] = out[c];
        }
    }
}

// The consumed accumulators are cleared as the G2P goes (the guide's "the
// grid clear can ride along"): node block b (tile^dim nodes) is read only by
// the work items of the tiles b - delta, delta in {0,1}^dim, each loading its
// tile's halo once into shared memory.  After it has, a work item of tile t
// counts itself a reader of each of its blocks t + delta; the reader that
// completes a block's count (the slices of those tiles, ceil(count / 1024)
// each) clears the block's accumulators, every channel, and resets the
// count.  So each touched node is zero after the G2P, as mpm_grid_update
// leaves it, and no block is cleared before its last reader has loaded it.
// Called by one whole warp, after the halo loads of its work item are done.
template <int DIM, int T, typename AccT, int NCH>
__device__ __forceinline__ void release_blocks(const GridP &g, uint32_t t, uint32_t *readers, const uint32_t *count,
                                               AccT *acc, uint32_t lane) {
    constexpr int LOG = T == 4 ? 2 : 3;
    const int tc[3] = {(int)(t % (uint32_t)g.nt[0]), (int)((t / (uint32_t)g.nt[0]) % (uint32_t)g.nt[1]),
                       DIM == 3 ? (int)(t / ((uint32_t)g.nt[0] * (uint32_t)g.nt[1])) : 0};
    int bc[3] = {0, 0, 0};
    bool done = false;
    if (lane < (1u << DIM)) {
        bool valid = true;
#pragma unroll
        for (int l = 0; l < DIM; ++l) {
            bc[l] = tc[l] + (int)((lane >> l) & 1u);
            valid = valid && bc[l] < g.nb[l];
        }
        if (valid) {
            uint32_t expect = 0;
#pragma unroll
            for (int d = 0; d < (1 << DIM); ++d) {
                int u[3] = {0, 0, 0};
                bool ok = true;
#pragma unroll
                for (int l = 0; l < DIM; ++l) {
                    u[l] = bc[l] - ((d >> l) & 1);
                    ok = ok && u[l] >= 0 && u[l] < g.nt[l];
                }
                if (ok) {
                    const uint32_t c = count[((int64_t)u[2] * g.nt[1] + u[1]) * g.nt[0] + u[0]];
                    expect += (c + kSliceParticles - 1) / kSliceParticles;
                }
            }
            const int64_t blk = ((int64_t)bc[2] * g.nb[1] + bc[1]) * g.nb[0] + bc[0];
            if (atomicAdd(&readers[blk], 1u) + 1u == expect) {
                readers[blk] = 0u;
                done = true;
            }
        }
    }
    uint32_t todo = __ballot_sync(0xFFFFFFFFu, done);
    while (todo) {
        const int j = __ffs(todo) - 1;
        todo &= todo - 1u;
        const int b0 = __shfl_sync(0xFFFFFFFFu, bc[0], j), b1 = __shfl_sync(0xFFFFFFFFu, bc[1], j);
        const int b2 = __shfl_sync(0xFFFFFFFFu, bc[2], j);
        for (int i = (int)lane; i < (DIM == 3 ? T * T * T : T * T); i += 32) {
            const int x = b0 * T + (i & (T - 1)), y = b1 * T + ((i >> LOG) & (T - 1));
            const int z = DIM == 3 ? b2 * T + (i >> (2 * LOG)) : 0;
            if (x >= g.n[0] || y >= g.n[1] || (DIM == 3 && z >= g.n[2])) continue;
            const int64_t node = node_index(g, x, y, z);
#pragma unroll
            for (int c = 0; c < NCH; ++c) acc[c * g.nodes + node] = (AccT)0;
        }
    }
}

}  // namespace mpm
