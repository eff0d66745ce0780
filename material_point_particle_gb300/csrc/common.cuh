// common.cuh -- device-side parameters and helpers shared by the CUDA kernels
// of the MPM transfer library (binning, P2G, grid update, G2P).  Internal to
// the library: nothing here is part of the C ABI.
#pragma once

#include <cstdint>
#include <type_traits>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/mpm.h"

namespace mpm {

constexpr uint32_t kKeyInvalid = 0xFFFFFFFFu;
// Particles per P2G/G2P work item (a slice of one tile's sorted particles),
// and the threads of the CTAs that process them.
constexpr int kSliceParticles = 1024;
constexpr int kP2GThreads = 256;
constexpr int kG2PThreads = 256;
// 1.5 * 2^23: adding it to |t| < 2^22 leaves rint(t) in the low mantissa bits.
constexpr float kMagic = 12582912.0f;
constexpr int32_t kMagicBits = 0x4B400000;
// A share must stay below 2^22 in magnitude; the range test keeps this margin.
constexpr float kShareLimit = 4190208.0f;  // 2^22 - 4096
// Status flag set by a check that runs before P2G: P2G then scatters nothing.
constexpr uint32_t kFlagNoScatter = 1u << 16;
// Status flag set by a scatter that met a particle above the range its bound
// was checked with: the scatter is undone (k_rollback).
constexpr uint32_t kFlagRollback = 1u << 17;

// Everything a kernel needs to know about the grid, derived once on the host.
struct GridP {
    int dim;
    int n[3];
    float dx, inv_dx;
    int acc_mode;
    float S;             // 2^scale_log2 as fp32
    int T;               // tile edge in cells
    int T_log2;
    int nt[3];           // tiles per axis (1 on unused axes)
    int cpt_log2;        // log2(cells per tile) = dim * T_log2
    int64_t ntiles;      // product of nt
    int64_t nodes;       // product of n (n[2] = 1 in 2D)
    int H;               // halo edge T + 2
    int halo_nodes;      // H^dim
    int nb[3];           // node blocks (T^dim nodes) per axis
    int64_t nblocks;
    int boundary;        // boundary_nodes
    float wmax;          // 0.75^dim
    int vc;              // 1: grid-recovered volume channel
    float vcell;         // inv_dx^dim, (inv_dx * inv_dx) [* inv_dx]
    float inv_S;         // 2^-scale_log2 (1 in float mode)
};

// Particle SoA as raw typed pointers.
struct PartsF {
    float *x[3];
    float *v[3];
    float *C[9];
    const float *m;
    uint32_t *id;
    float *F[9];  // elastic state (F[0] null for none): deformation gradient
    float *vol;   // rest volume (elastic state, volume channel)
    float mu, lam;
    float *phi;   // volume channel: grid-recovered volume fraction (G2P output)
    int64_t n;
};

__device__ __forceinline__ uint32_t lane_id() {
    uint32_t l;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
    return l;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// An accumulator value as fp32, rounded to nearest (the grid update's (float)P, (float)M).
template <typename AccT>
__device__ __forceinline__ float acc_to_float(AccT v) {
    if constexpr (sizeof(AccT) == 8)
        return __ll2float_rn((long long)v);
    else if constexpr (std::is_same<AccT, float>::value)
        return v;
    else
        return __int2float_rn((int)v);
}

// Status word helpers: flags are bit (1 << mpm_status).
__device__ __forceinline__ void set_flag(uint32_t *status, int code) {
    atomicOr(&status[MPM_ST_FLAGS], 1u << code);
}

// Stencil base and fraction along one axis; false outside the domain
// (0.5 <= xi < n - 1.5): b = floor(xi - 0.5), f = xi - b.  Every operation is
// one IEEE fp32 rounding.  The floor goes through the fp32 adder: for
// 0 <= y < 2^23 the sum y + 2^23 rounded down is 2^23 + floor(y) exactly, an
// fp32 number whose bit pattern is that of 2^23 plus floor(y), so b is an
// integer subtraction and (float)b a subtraction of 2^23 (no conversions).
// The domain test is then 0 <= b <= n - 3: grids have at most 2^20 nodes per
// axis, so y = xi - 0.5 is exact wherever it can pass, and a y below 0, at or
// above 2^23, infinite or NaN leaves a b outside that range.
__device__ __forceinline__ bool base_frac(float x, float inv_dx, int n, int &b, float &f) {
    const float xi = __fmul_rn(x, inv_dx);
    const float t = __fadd_rd(__fsub_rn(xi, 0.5f), 8388608.0f);
    b = __float_as_int(t) - 0x4B000000;
    if ((uint32_t)b > (uint32_t)(n - 3)) return false;
    f = __fsub_rn(xi, __fsub_rn(t, 8388608.0f));
    return true;
}

// Tile-major cell key with the tile shape known at compile time.
template <int DIM, int T>
__device__ __forceinline__ uint32_t cell_key_t(const GridP &g, const int b[3]) {
    constexpr int LOG = T == 4 ? 2 : 3;
    uint32_t tile = 0, local = 0;
#pragma unroll
    for (int l = DIM - 1; l >= 0; --l) {
        tile = tile * (uint32_t)g.nt[l] + ((uint32_t)b[l] >> LOG);
        local = (local << LOG) | ((uint32_t)b[l] & (T - 1));
    }
    return (tile << (DIM * LOG)) | local;
}

// The key of position x (kKeyInvalid outside the domain), as the binning computes it.
template <int DIM, int T>
__device__ __forceinline__ uint32_t key_of_x(const GridP &g, const float (&x)[DIM]) {
    int b[3] = {0, 0, 0};
    float f;
    bool ok = true;
#pragma unroll
    for (int l = 0; l < DIM; ++l) ok = base_frac(x[l], g.inv_dx, g.n[l], b[l], f) && ok;
    return ok ? cell_key_t<DIM, T>(g, b) : kKeyInvalid;
}

// Quadratic B-spline weights at distances f, f-1, f-2 from the stencil's
// first node (f in [0.5, 1.5)).
__device__ __forceinline__ void quad_weights(float f, float w[3]) {
    float t0 = __fsub_rn(1.5f, f);
    float t1 = __fsub_rn(f, 1.0f);
    float t2 = __fsub_rn(f, 0.5f);
    w[0] = __fmul_rn(0.5f, __fmul_rn(t0, t0));
    w[1] = __fsub_rn(0.75f, __fmul_rn(t1, t1));
    w[2] = __fmul_rn(0.5f, __fmul_rn(t2, t2));
}

// Tile-major key of base cell b (tile id * T^dim + cell within tile).
__device__ __forceinline__ uint32_t cell_key(const GridP &g, const int b[3]) {
    uint32_t tile = 0, local = 0;
    const uint32_t mask = (uint32_t)g.T - 1;
#pragma unroll
    for (int l = 2; l >= 0; --l) {
        if (l >= g.dim) continue;
        tile = tile * (uint32_t)g.nt[l] + ((uint32_t)b[l] >> g.T_log2);
        local = (local << g.T_log2) | ((uint32_t)b[l] & mask);
    }
    return (tile << g.cpt_log2) | local;
}

__device__ __forceinline__ void tile_origin(const GridP &g, uint32_t tile, int o[3]) {
    o[0] = (int)(tile % (uint32_t)g.nt[0]) * g.T;
    uint32_t r = tile / (uint32_t)g.nt[0];
    o[1] = (int)(r % (uint32_t)g.nt[1]) * g.T;
    o[2] = g.dim == 3 ? (int)(r / (uint32_t)g.nt[1]) * g.T : 0;
}

// Base cell and fraction of particle pid, and whether that base cell lies in
// the tile at origin o (it does for every particle binned into the tile from
// the same positions; the test keeps shared-memory indices in range if the
// positions changed after binning).
template <int DIM>
__device__ __forceinline__ bool in_tile(const GridP &g, const PartsF &p, uint32_t pid, const int o[3], int b[3],
                                        float f[3]) {
    bool ok = true;
#pragma unroll
    for (int l = 0; l < DIM; ++l) {
        ok = ok && base_frac(p.x[l][pid], g.inv_dx, g.n[l], b[l], f[l]);
        ok = ok && b[l] >= o[l] && b[l] < o[l] + g.T;
    }
    return ok;
}

// The same test on positions already loaded.
template <int DIM>
__device__ __forceinline__ bool in_tile_x(const GridP &g, const float *x, const int o[3], int b[3], float f[3]) {
    bool ok = true;
#pragma unroll
    for (int l = 0; l < DIM; ++l) {
        ok = ok && base_frac(x[l], g.inv_dx, g.n[l], b[l], f[l]);
        ok = ok && b[l] >= o[l] && b[l] < o[l] + g.T;
    }
    return ok;
}

// Dynamic work distribution from a global counter.  A CTA takes its first
// item with grab_item; inside the loop, thread 0 asks for the next item at
// the top (ask_item: the atomic's latency overlaps the item's work) and
// publish_item hands it to the whole CTA at the bottom.
__device__ __forceinline__ uint32_t grab_item(uint32_t *counter, uint32_t *sh) {
    __syncthreads();
    if (threadIdx.x == 0) *sh = atomicAdd(counter, 1u);
    __syncthreads();
    return *sh;
}
__device__ __forceinline__ uint32_t ask_item(uint32_t *counter) {
    return threadIdx.x == 0 ? atomicAdd(counter, 1u) : 0u;
}
__device__ __forceinline__ uint32_t publish_item(uint32_t next, uint32_t *sh) {
    __syncthreads();
    if (threadIdx.x == 0) *sh = next;
    __syncthreads();
    return *sh;
}

// Compile-time loop: f(std::integral_constant<int, i>) for i = 0 .. N-1.
template <typename F, int... I>
__device__ __forceinline__ void static_for_impl(F &f, std::integer_sequence<int, I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F &&f) {
    static_for_impl(f, std::make_integer_sequence<int, N>{});
}

// Shared-memory add without a result, at a constant byte offset from a
// shared address.
template <int OFF>
__device__ __forceinline__ void red_shared_add(uint32_t base, int32_t v) {
    asm volatile("red.shared.add.s32 [%0+%1], %2;" ::"r"(base), "n"(OFF), "r"(v));
}

// Asynchronous 4-byte global -> shared copies (cp.async), grouped per thread.
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gsrc) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// The particle record of P2G: x[dim], v[dim], C[dim*dim], m, then with the
// elastic state F[dim*dim], and vol when the elastic state or the volume
// channel needs it.
template <int DIM, bool EL = false, bool VC = false>
struct P2GFields {
    static constexpr int BASE = DIM + DIM + DIM * DIM + 1;  // index of F[0]
    static constexpr int VOLF = BASE + (EL ? DIM * DIM : 0);  // index of vol
    static constexpr int NF = VOLF + (EL || VC ? 1 : 0);
    __device__ static const float *src(const PartsF &p, int f) {
        return f < DIM                    ? p.x[f]
               : f < 2 * DIM              ? p.v[f - DIM]
               : f < 2 * DIM + DIM * DIM  ? p.C[f - 2 * DIM]
               : f < BASE                 ? p.m
               : f < VOLF                 ? p.F[f - BASE]
                                          : p.vol;
    }
};

__device__ __forceinline__ int64_t node_index(const GridP &g, int i, int j, int k) {
    return ((int64_t)k * g.n[1] + j) * g.n[0] + i;
}

template <int DIM>
struct Stencil {
    static constexpr int NA = DIM == 3 ? 27 : 9;
    static constexpr int NC = DIM + 1;
    static constexpr int CENTRE = DIM == 3 ? 13 : 4;  // a = (1,1,1) / (1,1)
};

// Shared-memory halo of one tile: (T+2)^dim nodes, x fastest, rows and planes
// padded so that the 32 cells of one rank-major group (a 4x4x2 or 8x4 block)
// fall in 32 different banks: row pitch 36 = 4 (mod 32), plane pitch
// 240 = 16 (mod 32) in 3D; row pitch 40 = 8 (mod 32) in 2D.
template <int DIM, int T>
struct Halo {
    static constexpr int H = T + 2;
    static constexpr int SY = DIM == 3 ? 36 : 40;
    static constexpr int SZ = DIM == 3 ? 240 : 0;
    static constexpr int SIZE = DIM == 3 ? (H - 1) * SZ + (H - 1) * SY + H : (H - 1) * SY + H;
    static constexpr int NODES = DIM == 3 ? H * H * H : H * H;
    // padded offset of stencil node a = a0*9 + a1*3 + a2 (3D) or a0*3 + a1 (2D)
    __device__ static constexpr int off(int a) {
        return DIM == 3 ? (a / 9) + (a / 3 % 3) * SY + (a % 3) * SZ : (a / 3) + (a % 3) * SY;
    }
    // padded index and grid coordinates of halo node h (x fastest)
    __device__ static void node(int h, int &hx, int &hy, int &hz, int &idx) {
        hx = h % H;
        hy = (h / H) % H;
        hz = DIM == 3 ? h / (H * H) : 0;
        idx = hx + hy * SY + hz * SZ;
    }
};

// Compact shared-memory halo of one tile: (T+2)^dim nodes, x fastest, no
// padding (row pitch H, plane pitch H^2), channel c at c * NODES.  Node
// (hx, hy, hz) sits in bank (hx + H hy + H^2 hz) mod 32, so particles whose
// base cells have different bank classes (cell_class) add to, or read, a given
// stencil node in different banks.
template <int DIM, int T>
struct HaloU {
    static constexpr int H = T + 2;
    static constexpr int SY = H;
    static constexpr int SZ = DIM == 3 ? H * H : 0;
    static constexpr int NODES = DIM == 3 ? H * H * H : H * H;
    static constexpr int SIZE = NODES;
    // offset of stencil node a = a0*9 + a1*3 + a2 (3D) or a0*3 + a1 (2D)
    __device__ static constexpr int off(int a) {
        return DIM == 3 ? (a / 9) + (a / 3 % 3) * SY + (a % 3) * SZ : (a / 3) + (a % 3) * SY;
    }
    __device__ static void node(int h, int &hx, int &hy, int &hz) {
        hx = h % H;
        hy = (h / H) % H;
        hz = DIM == 3 ? h / (H * H) : 0;
    }
};

// Bank class of a base cell from the in-tile bits of its key
// (local = lx + T ly + T^2 lz): its compact-halo offset modulo 32.
template <int DIM, int T>
__device__ __forceinline__ uint32_t cell_class(uint32_t key) {
    constexpr int H = T + 2;
    constexpr int LOG = T == 4 ? 2 : 3;
    const uint32_t lx = key & (T - 1), ly = (key >> LOG) & (T - 1);
    const uint32_t lz = DIM == 3 ? (key >> (2 * LOG)) & (T - 1) : 0u;
    return (lx + H * ly + H * H * lz) & 31u;
}

}  // namespace mpm
