// bin.cu -- cell keys and the stable counting sort of particles into tiles.
//
// "Particle Worlds, part 3", Step 3 and Step 4: a counting sort in three
// phases, histogram -> exclusive prefix sum -> scatter, the scan as per-block
// scans, a scan of the block totals and an add-back.  The page's scatter
// claims slots with an atomic cursor and so leaves the order inside a bucket
// unspecified; the implementation guide (section 2.1, caveat (b), and rule 3)
// asks for every such race to be neutralised by a sort on a stable key.
// Here the buckets are tiles of T^dim base cells (section 2.1: bin into
// tiles, sort an index buffer, particles never move), the atomic scatter
// fills each tile's range, and one CTA per tile then sorts the range by
// (cell, particle index) in shared memory, which makes the permutation the
// stable sort of the keys -- a deterministic function of the keys.
//
// Kernels (all on the caller's stream, no host synchronisation):
//   k_keys          key per particle, warp-aggregated tile histogram,
//                   out-of-domain count (int32 mode: per-cell counts)
//   k_scan_reduce / k_scan_top / k_scan_final
//                   exclusive scans of (count, P2G slices, active flag) over
//                   the buckets; active-tile list, P2G work list, cursors
//   k_scatter       warp-aggregated atomic scatter of indices into buckets
//   k_tile_order    per-tile order: claims sorted back into index order, a
//                   stable counting sort by cell, the rank-major write-out
//   k_nbr_bound     int32 mode: most stencils covering one node (the
//                   accumulator bound, checked before any scatter)
#include "common.cuh"
#include "internal.h"

namespace mpm {

// --------------------------------------------------------------------------
__global__ void k_keys(GridP g, PartsF p, uint32_t *__restrict__ key, uint32_t *__restrict__ count,
                       uint32_t *__restrict__ cellcount, uint32_t *__restrict__ status) {
    const int64_t n = p.n;
    const uint32_t lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const uint32_t bucket_invalid = (uint32_t)g.ntiles;
    for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32; base < n;
         base += warps * 32) {
        const int64_t i = base + lane;
        uint32_t k = kKeyInvalid, bucket = 0xFFFFFFFFu;
        if (i < n) {
            int b[3] = {0, 0, 0};
            float f;
            bool ok = true;
            for (int l = 0; l < g.dim; ++l) ok = ok && base_frac(p.x[l][i], g.inv_dx, g.n[l], b[l], f);
            if (ok) {
                k = cell_key(g, b);
                bucket = k >> g.cpt_log2;
                if (cellcount) atomicAdd(&cellcount[k], 1u);
            } else {
                bucket = bucket_invalid;
            }
            key[i] = k;
        }
        // warp-aggregated histogram: one atomic per distinct bucket in the warp
        const uint32_t live = __ballot_sync(0xFFFFFFFFu, i < n);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bucket) & live;
        if (i < n && (peers & lanemask_lt()) == 0) {
            atomicAdd(&count[bucket], (uint32_t)__popc(peers));
            if (bucket == bucket_invalid) atomicAdd(&status[MPM_ST_N_OUTSIDE], (uint32_t)__popc(peers));
        }
    }
}

// --------------------------------------------------------------------------
// Scans over the nb = ntiles + 1 buckets (the last bucket holds the particles
// outside the domain).  Each thread of a 256-thread block owns 4 buckets.
constexpr int kScanThreads = 256;
constexpr int kScanItems = 4;
constexpr int kScanBlock = kScanThreads * kScanItems;

struct Tri {
    uint32_t a, b, c;
};

__device__ __forceinline__ Tri tri_add(Tri x, Tri y) { return {x.a + y.a, x.b + y.b, x.c + y.c}; }

__device__ __forceinline__ Tri bucket_values(const GridP &g, const uint32_t *count, int64_t nb, int64_t b) {
    if (b >= nb) return {0, 0, 0};
    uint32_t c = count[b];
    if (b == nb - 1) return {c, 0, 0};  // outside-the-domain bucket: no P2G work
    return {c, (c + kSliceParticles - 1) / kSliceParticles, c > 0 ? 1u : 0u};
}

// Block-wide exclusive scan of one Tri per thread; returns the block total.
__device__ Tri block_exclusive_scan(Tri v, Tri &excl) {
    __shared__ Tri warp_tot[kScanThreads / 32];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    Tri inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t a = __shfl_up_sync(0xFFFFFFFFu, inc.a, d);
        uint32_t b = __shfl_up_sync(0xFFFFFFFFu, inc.b, d);
        uint32_t c = __shfl_up_sync(0xFFFFFFFFu, inc.c, d);
        if ((int)lane >= d) inc = tri_add(inc, {a, b, c});
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    Tri before = {0, 0, 0}, total = {0, 0, 0};
    for (int w = 0; w < kScanThreads / 32; ++w) {
        if (w < (int)warp) before = tri_add(before, warp_tot[w]);
        total = tri_add(total, warp_tot[w]);
    }
    excl = {before.a + inc.a - v.a, before.b + inc.b - v.b, before.c + inc.c - v.c};
    __syncthreads();
    return total;
}

__global__ void k_scan_reduce(GridP g, const uint32_t *__restrict__ count, int64_t nb, Tri *__restrict__ partial) {
    const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    Tri s = {0, 0, 0};
    for (int j = 0; j < kScanItems; ++j) s = tri_add(s, bucket_values(g, count, nb, b0 + j));
    Tri excl;
    Tri tot = block_exclusive_scan(s, excl);
    if (threadIdx.x == 0) partial[blockIdx.x] = tot;
}

// One block: exclusive scan of the block totals (in place) and the grand totals.
__global__ void k_scan_top(Tri *__restrict__ partial, int64_t nblocks, const uint32_t *__restrict__ count,
                           int64_t nb, uint32_t *__restrict__ status) {
    Tri carry = {0, 0, 0};
    for (int64_t base = 0; base < nblocks; base += kScanThreads) {
        int64_t i = base + threadIdx.x;
        Tri v = i < nblocks ? partial[i] : Tri{0, 0, 0};
        Tri excl;
        Tri tot = block_exclusive_scan(v, excl);
        if (i < nblocks) partial[i] = tri_add(carry, excl);
        carry = tri_add(carry, tot);
    }
    if (threadIdx.x == 0) {
        status[MPM_ST_N_VALID] = carry.a - count[nb - 1];
        status[MPM_ST_N_SLICES] = carry.b;
        status[MPM_ST_N_ACTIVE] = carry.c;
    }
}

__global__ void k_scan_final(GridP g, const uint32_t *__restrict__ count, int64_t nb, const Tri *__restrict__ partial,
                             uint32_t *__restrict__ start, uint32_t *__restrict__ cursor,
                             uint32_t *__restrict__ active, uint32_t *__restrict__ slices,
                             uint32_t *__restrict__ status) {
    const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    Tri v[kScanItems];
    Tri s = {0, 0, 0};
    for (int j = 0; j < kScanItems; ++j) {
        v[j] = bucket_values(g, count, nb, b0 + j);
        s = tri_add(s, v[j]);
    }
    Tri excl;
    block_exclusive_scan(s, excl);
    Tri run = tri_add(partial[blockIdx.x], excl);
    for (int j = 0; j < kScanItems; ++j) {
        const int64_t b = b0 + j;
        if (b >= nb) break;
        start[b] = run.a;
        cursor[b] = run.a;
        if (v[j].c) active[run.c] = (uint32_t)b;
        for (uint32_t s2 = 0; s2 < v[j].b; ++s2) {
            slices[2 * (int64_t)(run.b + s2)] = (uint32_t)b;
            slices[2 * (int64_t)(run.b + s2) + 1] = s2 * kSliceParticles;
        }
        run = tri_add(run, v[j]);
        if (b == nb - 1) start[nb] = run.a;
    }
}

// --------------------------------------------------------------------------
__global__ void k_scatter(GridP g, const uint32_t *__restrict__ key, int64_t n, uint32_t *__restrict__ cursor,
                          uint32_t *__restrict__ tmp) {
    const uint32_t lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const uint32_t bucket_invalid = (uint32_t)g.ntiles;
    for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32; base < n;
         base += warps * 32) {
        const int64_t i = base + lane;
        uint32_t bucket = 0xFFFFFFFFu;
        if (i < n) {
            uint32_t k = key[i];
            bucket = k == kKeyInvalid ? bucket_invalid : (k >> g.cpt_log2);
        }
        const uint32_t live = __ballot_sync(0xFFFFFFFFu, i < n);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bucket) & live;
        const uint32_t leader = __ffs(peers) - 1;
        uint32_t slot = 0;
        if (i < n && lane == leader) slot = atomicAdd(&cursor[bucket], (uint32_t)__popc(peers));
        slot = __shfl_sync(0xFFFFFFFFu, slot, leader);
        if (i < n) tmp[slot + __popc(peers & lanemask_lt())] = (uint32_t)i;
    }
}

// --------------------------------------------------------------------------
// The order inside each tile.  The atomic scatter filled each bucket with
// "claims": one per warp and bucket, holding that warp's lanes of the bucket
// in lane (= index) order, and all sharing idx >> 5 (a warp covers 32
// consecutive indices per round).  So sorting the claims by idx >> 5 puts the
// bucket in index order.  In steady state a tile has few claims; from a cold
// order every entry is its own claim and this is a plain sort.  A stable
// counting sort by cell follows (cell-major, each cell in index order), then
// the rank-major write-out: each group of 32 cells lists rank 0 of its cells,
// then rank 1, and so on.  Buckets above kOrderCap entries use global scratch
// instead of shared memory (same code, generic pointers).
constexpr int kOrderThreads = 256;
constexpr int kOrderCap = 4096;
constexpr int kOrderWarps = kOrderThreads / 32;

__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t &total, uint32_t *sh) {
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if ((int)lane >= d) inc += t;
    }
    if (lane == 31) sh[warp] = inc;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kOrderWarps; ++w) {
        const uint32_t t = sh[w];
        before += (w < (int)warp) ? t : 0u;
        tot += t;
    }
    __syncthreads();
    total = tot;
    return before + inc - v;
}

// Ascending bitonic sort of n_pow2 keys, block-wide (shared or global memory).
__device__ void block_bitonic(unsigned long long *s, uint32_t n_pow2) {
    for (uint32_t k = 2; k <= n_pow2; k <<= 1) {
        for (uint32_t j = k >> 1; j > 0; j >>= 1) {
            for (uint32_t t = threadIdx.x; t < (n_pow2 >> 1); t += blockDim.x) {
                const uint32_t i = (t / j) * 2 * j + (t % j);
                const uint32_t pr = i + j;
                const bool up = (i & k) == 0;
                const unsigned long long a = s[i], b = s[pr];
                if ((a > b) == up) {
                    s[i] = b;
                    s[pr] = a;
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kOrderThreads)
k_tile_order(GridP g, const uint32_t *__restrict__ key, uint32_t *tmp, const uint32_t *__restrict__ start,
             const uint32_t *__restrict__ count, const uint32_t *__restrict__ active, int64_t nb, uint32_t *perm,
             uint32_t *gH, unsigned long long *gCW, uint32_t *__restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned long long *sCW = reinterpret_cast<unsigned long long *>(smem_raw);
    uint32_t *sA = reinterpret_cast<uint32_t *>(sCW + kOrderCap);
    uint32_t *sS = sA + kOrderCap;
    uint32_t *sH = sS + kOrderCap;
    __shared__ uint32_t cnt64[64], cs64[65], run64[64];
    __shared__ uint32_t wcnt[kOrderWarps][64], woff[kOrderWarps][64];
    __shared__ uint32_t scan_sh[kOrderWarps];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    const uint32_t n_active = status[MPM_ST_N_ACTIVE];
    const uint32_t cmask = (1u << g.cpt_log2) - 1;
    for (uint32_t item = blockIdx.x; item <= n_active; item += gridDim.x) {
        const bool outside = item == n_active;
        const uint32_t b = outside ? (uint32_t)(nb - 1) : active[item];
        const uint32_t beg = start[b], cnt = count[b];
        if (cnt == 0) continue;
        if (cnt == 1) {
            if (threadIdx.x == 0) perm[beg] = tmp[beg];
            continue;
        }
        const bool small = cnt <= (uint32_t)kOrderCap;
        if (!small && threadIdx.x == 0) atomicAdd(&status[MPM_ST_N_BIG_TILES], 1u);
        uint32_t *A = small ? sA : tmp + beg;
        uint32_t *S = small ? sS : perm + beg;
        uint32_t *H = small ? sH : gH + (size_t)beg + item;
        unsigned long long *CW = small ? sCW : gCW + 2 * (size_t)beg;
        if (small)
            for (uint32_t i = threadIdx.x; i < cnt; i += blockDim.x) A[i] = tmp[beg + i];
        __syncthreads();
        // claims: heads where idx >> 5 changes
        uint32_t nclaims = 0;
        for (uint32_t base = 0; base < cnt; base += blockDim.x) {
            const uint32_t i = base + threadIdx.x;
            uint32_t head = 0, w = 0;
            if (i < cnt) {
                w = A[i] >> 5;
                head = (i == 0 || w != (A[i - 1] >> 5)) ? 1u : 0u;
            }
            uint32_t tot;
            const uint32_t ex = block_excl_scan(head, tot, scan_sh);
            if (head) {
                const uint32_t k = nclaims + ex;
                H[k] = i;
                CW[k] = ((unsigned long long)w << 32) | k;
            }
            nclaims += tot;
        }
        uint32_t np2 = 1;
        while (np2 < nclaims) np2 <<= 1;
        for (uint32_t k = nclaims + threadIdx.x; k < np2; k += blockDim.x) CW[k] = ~0ull;
        if (threadIdx.x == 0) H[nclaims] = cnt;
        __syncthreads();
        if (nclaims > 1) block_bitonic(CW, np2);
        // claims in index order: copy each claim to its destination
        uint32_t done = 0;
        for (uint32_t base = 0; base < nclaims; base += blockDim.x) {
            const uint32_t j = base + threadIdx.x;
            uint32_t len = 0, k = 0;
            if (j < nclaims) {
                k = (uint32_t)(CW[j] & 0xFFFFFFFFu);
                len = H[k + 1] - H[k];
            }
            uint32_t tot;
            const uint32_t ex = block_excl_scan(len, tot, scan_sh);
            if (j < nclaims) {
                const uint32_t d = done + ex, src = H[k];
                for (uint32_t e = 0; e < len; ++e) S[d + e] = A[src + e];
            }
            done += tot;
        }
        __syncthreads();
        if (outside) {
            if (small)
                for (uint32_t i = threadIdx.x; i < cnt; i += blockDim.x) perm[beg + i] = S[i];
            __syncthreads();
            continue;
        }
        // stable counting sort by cell: S (index order) -> A (cell-major)
        if (threadIdx.x < 64) cnt64[threadIdx.x] = 0;
        __syncthreads();
        for (uint32_t base = 0; base < cnt; base += blockDim.x) {
            const uint32_t i = base + threadIdx.x;
            const uint32_t c = i < cnt ? (key[S[i]] & cmask) : 64u;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, c);
            if (i < cnt && (peers & lanemask_lt()) == 0) atomicAdd(&cnt64[c], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const uint32_t a0 = cnt64[2 * lane], a1 = cnt64[2 * lane + 1];
            uint32_t inc = a0 + a1;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, d);
                if ((int)lane >= d) inc += t;
            }
            const uint32_t ex = inc - a0 - a1;
            cs64[2 * lane] = ex;
            cs64[2 * lane + 1] = ex + a0;
            run64[2 * lane] = ex;
            run64[2 * lane + 1] = ex + a0;
            if (lane == 31) cs64[64] = inc;
        }
        __syncthreads();
        for (uint32_t base = 0; base < cnt; base += blockDim.x) {
            const uint32_t i = base + threadIdx.x;
            const uint32_t c = i < cnt ? (key[S[i]] & cmask) : 64u;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, c);
            const uint32_t rank = __popc(peers & lanemask_lt());
            wcnt[warp][lane] = 0;
            wcnt[warp][lane + 32] = 0;
            __syncwarp();
            if (i < cnt && rank == 0) wcnt[warp][c] = __popc(peers);
            __syncthreads();
            if (threadIdx.x < 64) {
                uint32_t r = run64[threadIdx.x];
                for (int w2 = 0; w2 < kOrderWarps; ++w2) {
                    woff[w2][threadIdx.x] = r;
                    r += wcnt[w2][threadIdx.x];
                }
                run64[threadIdx.x] = r;
            }
            __syncthreads();
            if (i < cnt) A[woff[warp][c] + rank] = S[i];
            __syncthreads();
        }
        // rank-major write-out, one warp per group of 32 cells
        if (warp < 2) {
            const uint32_t c = warp * 32 + lane;
            const uint32_t nc = cnt64[c], first = cs64[c];
            uint32_t seg = warp == 0 ? 0u : cs64[32];
            for (uint32_t r = 0;; ++r) {
                const uint32_t m = __ballot_sync(0xFFFFFFFFu, nc > r);
                if (m == 0) break;
                if (nc > r) perm[beg + seg + __popc(m & lanemask_lt())] = A[first + r];
                seg += __popc(m);
            }
        }
        __syncthreads();
    }
}

// --------------------------------------------------------------------------
// int32 accumulators: for every node, the number of particles whose stencil
// covers it is the sum of the counts of the 3^dim base cells below it.
__global__ void k_nbr_bound(GridP g, const uint32_t *__restrict__ cellcount, uint32_t *__restrict__ status) {
    uint32_t best = 0;
    for (int64_t node = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; node < g.nodes;
         node += (int64_t)gridDim.x * blockDim.x) {
        int idx[3];
        idx[0] = (int)(node % g.n[0]);
        idx[1] = (int)((node / g.n[0]) % g.n[1]);
        idx[2] = (int)(node / ((int64_t)g.n[0] * g.n[1]));
        uint32_t sum = 0;
        for (int a2 = 0; a2 < (g.dim == 3 ? 3 : 1); ++a2)
            for (int a1 = 0; a1 < 3; ++a1)
                for (int a0 = 0; a0 < 3; ++a0) {
                    int b[3] = {idx[0] - a0, idx[1] - a1, g.dim == 3 ? idx[2] - a2 : 0};
                    bool ok = true;
                    for (int l = 0; l < g.dim; ++l) ok = ok && b[l] >= 0 && b[l] <= g.n[l] - 3;
                    if (ok) sum += cellcount[cell_key(g, b)];
                }
        best = max(best, sum);
    }
    for (int d = 16; d > 0; d >>= 1) best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, d));
    if (lane_id() == 0 && best > 0) {
        atomicMax(&status[MPM_ST_MAX_NEIGHBOURS], best);
        if (best > kI32MaxContributions) atomicOr(&status[MPM_ST_FLAGS], (1u << MPM_E_BOUND) | kFlagNoScatter);
    }
}

// --------------------------------------------------------------------------
mpm_status launch_bin(const GridP &g, const PartsF &p, const WsView &w, const DeviceInfo &dev,
                      cudaStream_t st) {
    const int64_t n = p.n;
    const int64_t nb = g.ntiles + 1;
    cudaMemsetAsync(w.status, 0, MPM_STATUS_WORDS * sizeof(uint32_t), st);
    cudaMemsetAsync(w.count, 0, nb * sizeof(uint32_t), st);
    if (w.cellcount) cudaMemsetAsync(w.cellcount, 0, (size_t)(g.ntiles << g.cpt_log2) * sizeof(uint32_t), st);
    const int threads = 256;
    const int grid_p = (int)std::max<int64_t>(1, std::min<int64_t>((n + threads - 1) / threads, dev.sms * 8));
    if (n > 0) k_keys<<<grid_p, threads, 0, st>>>(g, p, w.key, w.count, w.cellcount, w.status);
    const int64_t nblk = (nb + kScanBlock - 1) / kScanBlock;
    k_scan_reduce<<<(unsigned)nblk, kScanThreads, 0, st>>>(g, w.count, nb, (Tri *)w.partial);
    k_scan_top<<<1, kScanThreads, 0, st>>>((Tri *)w.partial, nblk, w.count, nb, w.status);
    k_scan_final<<<(unsigned)nblk, kScanThreads, 0, st>>>(g, w.count, nb, (const Tri *)w.partial, w.start,
                                                          w.cursor, w.active, w.slices, w.status);
    if (n > 0) {
        k_scatter<<<grid_p, threads, 0, st>>>(g, w.key, n, w.cursor, w.tmp);
        const int smem = kOrderCap * (8 + 4 + 4 + 4) + 16;
        cudaFuncSetAttribute(k_tile_order, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        k_tile_order<<<dev.sms * 2, kOrderThreads, smem, st>>>(g, w.key, w.tmp, w.start, w.count, w.active, nb, w.perm,
                                                             w.gH, (unsigned long long *)w.gCW, w.status);
    }
    if (w.cellcount) k_nbr_bound<<<dev.sms * 4, 256, 0, st>>>(g, w.cellcount, w.status);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
